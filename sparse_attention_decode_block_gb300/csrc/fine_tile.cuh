// The exact index scores of a tile of up to kFtTok tokens whose FP8 e4m3
// keys (128 dims, 128 bytes a row) are staged in shared memory, for one CTA
// of kFtThreads threads (LeanSparse, Section 5: the exact pass rescores the
// retained candidates with their original FP8 indexer keys).  Two scores:
//   head sum          f_t = scale_t * q_sum . e4m3(k8_t)
//   weighted ReLU     f_t = scale_t * sum_g w_g ReLU(q_g . e4m3(k8_t))
//                     (Eq. 6's head aggregation on the exact keys;
//                     scale_t >= 0, so scale_t ReLU(x) = ReLU(scale_t x)).
// The weighted-ReLU dots of all 64 heads are a dense [64 x 128] x
// [128 x tokens] product, run as f16 m16n8k16 MMAs with fp32 accumulation:
// e4m3 values are exact in f16, and bf16 queries are exact in f16 for
// 2^-17 <= |q| < 2^16 (a larger one is flagged by the caller).
#pragma once

#include "lsa_device.cuh"

namespace lsa {
namespace {

constexpr int kFtThreads = 512;
constexpr int kFtWarps = kFtThreads / 32;
constexpr int kFtTok = 1024;   // tokens of one tile at most

// Byte offset of 16-byte chunk u of token t's 128-byte key row: the chunk
// index is XORed with t mod 8, so that 8 consecutive tokens' same chunk
// fall in different banks.
__device__ __forceinline__ uint32_t cf_key_off(int t, int u) { return (uint32_t)(t * 128 + ((u ^ (t & 7)) << 4)); }

// Two floats -> f16x2 (low half = lo).
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
    return h2;
}

// This warp's weighted-ReLU operands: the A fragments of its 16 heads
// (M-tile warp % 4) over 128 dims in f16, with the k index permuted within
// each 16-dim slice (logical k 2cc, 2cc+1, 2cc+8, 2cc+9 = dims 4cc .. 4cc+3,
// the permutation of the B fragments in wrelu_tile_partials), and the two
// head weights each lane applies.  q64: the group's 64 query rows of 128
// dims; w64: their weights.  Returns true when a query element is outside
// f16's exact range (every thread of the CTA must then agree to score
// nothing: see wrelu_zero).
struct WreluQ {
    uint32_t qa[8][4];
    float w_lo, w_hi;
};

__device__ __forceinline__ bool wrelu_load_q(const uint16_t *q64, const float *w64, WreluQ &Q)
{
    const int lane = threadIdx.x & 31, mt = (threadIdx.x >> 5) & 3;
    const int rr = lane >> 2, cc = lane & 3;
    const uint16_t *q0 = q64 + (16 * mt + rr) * 128;
    const uint16_t *q8 = q0 + 8 * 128;
    bool big = false;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint2 x0 = *reinterpret_cast<const uint2 *>(q0 + 16 * ks + 4 * cc);
        const uint2 x8 = *reinterpret_cast<const uint2 *>(q8 + 16 * ks + 4 * cc);
        const float2 f00 = bf2_to_f2(x0.x), f01 = bf2_to_f2(x0.y);
        const float2 f80 = bf2_to_f2(x8.x), f81 = bf2_to_f2(x8.y);
        big |= fabsf(f00.x) >= 65536.f || fabsf(f00.y) >= 65536.f || fabsf(f01.x) >= 65536.f ||
               fabsf(f01.y) >= 65536.f || fabsf(f80.x) >= 65536.f || fabsf(f80.y) >= 65536.f ||
               fabsf(f81.x) >= 65536.f || fabsf(f81.y) >= 65536.f;
        Q.qa[ks][0] = pack_f16x2(f00.x, f00.y);
        Q.qa[ks][1] = pack_f16x2(f80.x, f80.y);
        Q.qa[ks][2] = pack_f16x2(f01.x, f01.y);
        Q.qa[ks][3] = pack_f16x2(f81.x, f81.y);
    }
    Q.w_lo = w64[16 * mt + rr];
    Q.w_hi = w64[16 * mt + rr + 8];
    return big;
}

__device__ __forceinline__ void wrelu_zero(WreluQ &Q)
{
    Q.w_lo = Q.w_hi = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) Q.qa[ks][0] = Q.qa[ks][1] = Q.qa[ks][2] = Q.qa[ks][3] = 0u;
}

// The weighted ReLUs of the staged keys (kb: shared address of the key
// rows, cf_key_off layout) summed over each warp's 16 heads: part[mt][t]
// for the four M-tiles mt.  Warp w takes M-tile w % 4 over every fourth
// group of 16 tokens starting at w / 4.  The caller adds the four parts in
// order and applies scale_t.
__device__ __forceinline__ void wrelu_tile_partials(uint32_t kb, int ntok, const WreluQ &Q, float *part)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int mt = warp & 3, th = warp >> 2;
    const int rr = lane >> 2, cc = lane & 3;
    const int ng = (ntok + 15) / 16;
    for (int gi = th; gi < ng; gi += kFtWarps / 4) {
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        const int t0 = gi * 16 + rr, t1 = t0 + 8;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t k0, k1;
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(k0) : "r"(kb + cf_key_off(t0, ks) + 4 * cc));
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(k1) : "r"(kb + cf_key_off(t1, ks) + 4 * cc));
            const uint32_t b00 = e4m3x2_to_f16x2((uint16_t)(k0 & 0xffffu));
            const uint32_t b01 = e4m3x2_to_f16x2((uint16_t)(k0 >> 16));
            const uint32_t b10 = e4m3x2_to_f16x2((uint16_t)(k1 & 0xffffu));
            const uint32_t b11 = e4m3x2_to_f16x2((uint16_t)(k1 >> 16));
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+f"(s0[0]), "+f"(s0[1]), "+f"(s0[2]), "+f"(s0[3])
                : "r"(Q.qa[ks][0]), "r"(Q.qa[ks][1]), "r"(Q.qa[ks][2]), "r"(Q.qa[ks][3]), "r"(b00), "r"(b01));
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+f"(s1[0]), "+f"(s1[1]), "+f"(s1[2]), "+f"(s1[3])
                : "r"(Q.qa[ks][0]), "r"(Q.qa[ks][1]), "r"(Q.qa[ks][2]), "r"(Q.qa[ks][3]), "r"(b10), "r"(b11));
        }
        // lane holds heads rr (s[0], s[1]) and rr + 8 (s[2], s[3]) of tokens
        // 2cc, 2cc + 1 of each 8-token n-tile: weight, ReLU, then the sum
        // over the 8 lanes sharing cc
        float u0 = Q.w_lo * fmaxf(s0[0], 0.f) + Q.w_hi * fmaxf(s0[2], 0.f);
        float u1 = Q.w_lo * fmaxf(s0[1], 0.f) + Q.w_hi * fmaxf(s0[3], 0.f);
        float u2 = Q.w_lo * fmaxf(s1[0], 0.f) + Q.w_hi * fmaxf(s1[2], 0.f);
        float u3 = Q.w_lo * fmaxf(s1[1], 0.f) + Q.w_hi * fmaxf(s1[3], 0.f);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            u0 += __shfl_xor_sync(0xffffffffu, u0, off);
            u1 += __shfl_xor_sync(0xffffffffu, u1, off);
            u2 += __shfl_xor_sync(0xffffffffu, u2, off);
            u3 += __shfl_xor_sync(0xffffffffu, u3, off);
        }
        if (rr == 0) {
            part[mt * kFtTok + gi * 16 + 2 * cc] = u0;
            part[mt * kFtTok + gi * 16 + 2 * cc + 1] = u1;
            part[mt * kFtTok + gi * 16 + 8 + 2 * cc] = u2;
            part[mt * kFtTok + gi * 16 + 8 + 2 * cc + 1] = u3;
        }
    }
}

__device__ __forceinline__ float wrelu_combine(const float *part, int t)
{
    return (part[t] + part[kFtTok + t]) + (part[2 * kFtTok + t] + part[3 * kFtTok + t]);
}

// The head-sum dot q_sum . e4m3(k8_t) of staged token t, 8 lanes per token
// (16 dims each, qs: this lane's 16 dims of the query sum); every lane of
// the 8 gets the sum.
__device__ __forceinline__ float headsum_dot(const uint8_t *keys, int t, const float (&qs)[16])
{
    const int sub = threadIdx.x & 7;
    const uint4 kv = *reinterpret_cast<const uint4 *>(keys + cf_key_off(t, sub));
    const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 lo = e4m3x2_to_f2((uint16_t)(w[e] & 0xffffu));
        const float2 hi = e4m3x2_to_f2((uint16_t)(w[e] >> 16));
        acc = fmaf(qs[4 * e + 0], lo.x, acc);
        acc = fmaf(qs[4 * e + 1], lo.y, acc);
        acc = fmaf(qs[4 * e + 2], hi.x, acc);
        acc = fmaf(qs[4 * e + 3], hi.y, acc);
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    return acc;
}

}  // namespace
}  // namespace lsa

// One 16-token item of K and V through a warp's ring of cp.async stages, and
// the attention of a GQA group (2..8 query heads, MMA rows 0..G-1) over it:
// S = Q K^T and O += P V as m16n8k16 MMAs with an online softmax in the
// log2 domain (Vortex blog post, block top-k equation: the softmax over the
// attended tokens).  Shared by the even-split attention kernel and the
// one-CTA-per-row decode step kernel.
#pragma once

#include "lsa_device.cuh"

namespace lsa {
namespace {

// Bytes of one item's K tile (16 rows of DK bf16 in XOR-swizzled 16-row x
// 128-byte sub-tiles); the V tile follows it.
template <int DK>
__host__ __device__ constexpr int item_kbytes()
{
    return (DK / 64) * kChunk * 128;
}

// Copies rows [0, n) of an item into ring stage st (shared address): K rows
// from kb, V rows from vb, row strides kts / vts in elements.
template <int DK>
__device__ __forceinline__ void stage_item_kv(uint32_t st, const uint8_t *kb, const uint8_t *vb, int64_t kts,
                                              int64_t vts, int n, uint64_t pol)
{
    constexpr int CPR = DK / 8;
    constexpr int CPL = kChunk * CPR / 32;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < CPL; ++u) {
        const int q = lane + 32 * u;
        const int t = q / CPR, ch = q % CPR;
        if (t < n) {
            cp_async16_policy(st + swizzle_offset(t, ch), kb + (int64_t)t * kts * 2 + ch * 16, pol);
            cp_async16_policy(st + item_kbytes<DK>() + swizzle_offset(t, ch), vb + (int64_t)t * vts * 2 + ch * 16,
                              pol);
        }
    }
}

// The running softmax state of the group over the tokens seen so far: the
// log2-domain maximum m and sum l per head, and the unnormalised output o
// (this lane's m16n8 accumulator fragments over DK / 8 column tiles).
template <int DK>
struct GroupState {
    float m, l;
    float o[DK / 8][4];
};

template <int DK>
__device__ __forceinline__ void group_state_reset(GroupState<DK> &s)
{
    s.m = -INFINITY;
    s.l = 0.f;
#pragma unroll
    for (int nt = 0; nt < DK / 8; ++nt) s.o[nt][0] = s.o[nt][1] = s.o[nt][2] = s.o[nt][3] = 0.f;
}

// Attends the n > 0 tokens of the item staged at kbase (shared address of
// its K tile; stage: the same stage's generic pointer) with the group's
// query fragments qa0 / qa2, and folds them into s.  Rows n .. 15 of the V
// tile are zeroed first (they meet zero weights, and 0 * NaN must not
// happen).
template <int DK>
__device__ __forceinline__ void attend_staged_item(uint32_t kbase, uint8_t *stage, int n, const uint32_t (&qa0)[DK / 16],
                                                   const uint32_t (&qa2)[DK / 16], float scale_log2, GroupState<DK> &s)
{
    constexpr int CPR = DK / 8;
    const int lane = threadIdx.x & 31;
    const int cc = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;
    const int tk = (mi >> 1) * 8 + r8, ck = mi & 1;
    const int tv = (mi & 1) * 8 + r8, cv = mi >> 1;
    const uint32_t vbase = kbase + item_kbytes<DK>();
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < DK / 16; ++ks) {
        uint32_t b[4];
        ldsm_x4(b, kbase + swizzle_offset(tk, 2 * ks + ck));
        mma_bf16_rows8(s0, qa0[ks], qa2[ks], b[0], b[1]);
        mma_bf16_rows8(s1, qa0[ks], qa2[ks], b[2], b[3]);
    }
    const int t0 = 2 * cc;
    const float z0 = t0 < n ? s0[0] * scale_log2 : -INFINITY;
    const float z1 = t0 + 1 < n ? s0[1] * scale_log2 : -INFINITY;
    const float z2 = t0 + 8 < n ? s1[0] * scale_log2 : -INFINITY;
    const float z3 = t0 + 9 < n ? s1[1] * scale_log2 : -INFINITY;
    float mx = fmaxf(fmaxf(z0, z1), fmaxf(z2, z3));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(s.m, mx);
    float alpha = 1.f;
    uint32_t pa0 = 0u, pa2 = 0u;
    if (mn != -INFINITY) {
        alpha = fast_ex2(s.m - mn);
        pa0 = pack_bf16x2(fast_ex2(z0 - mn), fast_ex2(z1 - mn));
        pa2 = pack_bf16x2(fast_ex2(z2 - mn), fast_ex2(z3 - mn));
        s.m = mn;
    }
    // the denominator sums the same bf16-rounded weights the MMA uses
    const float2 p01 = bf2_to_f2(pa0), p23 = bf2_to_f2(pa2);
    float ps = (p01.x + p01.y) + (p23.x + p23.y);
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    s.l = s.l * alpha + ps;
#pragma unroll
    for (int nt = 0; nt < DK / 8; ++nt) {
        s.o[nt][0] *= alpha;
        s.o[nt][1] *= alpha;
    }
    if (n < kChunk) {
        for (int q = lane; q < (kChunk - n) * CPR; q += 32) {
            const int t = n + q / CPR, ch = q % CPR;
            *reinterpret_cast<uint4 *>(stage + item_kbytes<DK>() + swizzle_offset(t, ch)) = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
    }
#pragma unroll
    for (int dt = 0; dt < DK / 16; ++dt) {
        uint32_t b[4];
        ldsm_x4_t(b, vbase + swizzle_offset(tv, 2 * dt + cv));
        mma_bf16_rows8(s.o[2 * dt], pa0, pa2, b[0], b[1]);
        mma_bf16_rows8(s.o[2 * dt + 1], pa0, pa2, b[2], b[3]);
    }
}

}  // namespace
}  // namespace lsa

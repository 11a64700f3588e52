// Block summaries: the bf16 mean key of every full block, one warp per
// (page, KV head) block; or Quest's element-wise maximum and minimum keys
// of the block (Vortex blog post, end of "Why Long Generations Are
// Expensive", and the Quest listing in "Writing an algorithm: vFlow").  The mean is summed in fp64 and rounded to bf16
// once, so it does not depend on the order of the reduction (Vortex blog
// post, "Block top-k attention": each block is summarized by its mean key,
// computed once when the block fills; forward_cache of the vFlow listing).
#include "lsa_device.cuh"

namespace lsa {
namespace {

constexpr int kWarpsPerCta = 8;

template <bool kNonCoherent>
__device__ __forceinline__ uint4 load16(const uint8_t *p)
{
    if constexpr (kNonCoherent) {
        return ldg_nc_v4(p);
    } else {
        return *reinterpret_cast<const uint4 *>(p);
    }
}

// One warp sums the b keys of block (page p, head h) and writes the bf16
// mean.  Lanes own 16-byte chunks of the key row; when a row has fewer than
// 32 chunks, lanes also split the tokens into phases and the phases are
// added with shuffles at the end (fp64 addition of these bf16 / scaled e4m3
// values is exact, so the order does not change the result).
template <bool kNonCoherent>
__device__ void summarize_block(const CacheView &c, int64_t p, int h, uint16_t *summ)
{
    const int lane = threadIdx.x & 31;
    const int b = c.b;
    const int epc = c.e4m3 ? 16 : 8;      // elements per 16-byte chunk
    const int nch = c.dk / epc;           // chunks per key row
    const int esz = c.e4m3 ? 1 : 2;
    const uint8_t *base = c.k + (p * c.kps + (int64_t)h * c.khs) * esz;
    const float *sbase = c.e4m3 ? c.kscale + p * c.sps + (int64_t)h * c.shs : nullptr;
    uint16_t *dst = summ + (p * c.hkv + h) * (int64_t)c.dk;
    const double db = (double)b;

    int phases = 1;
    if (nch < 32 && (32 % nch) == 0) phases = 32 / nch;
    for (int c0 = 0; c0 < nch; c0 += 32 / phases) {
        const int ch = c0 + (phases > 1 ? (lane % nch) : lane);
        const int ph = phases > 1 ? lane / nch : 0;
        const bool active = ch < nch;
        double sum[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) sum[i] = 0.0;
        if (active) {
            for (int t = ph; t < b; t += phases) {
                uint4 v = load16<kNonCoherent>(base + (int64_t)t * c.kts * esz + ch * 16);
                if (c.e4m3) {
                    const double sc = (double)sbase[t];
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float2 lo = e4m3x2_to_f2((uint16_t)(w[i] & 0xffffu));
                        float2 hi = e4m3x2_to_f2((uint16_t)(w[i] >> 16));
                        sum[4 * i + 0] += sc * (double)lo.x;
                        sum[4 * i + 1] += sc * (double)lo.y;
                        sum[4 * i + 2] += sc * (double)hi.x;
                        sum[4 * i + 3] += sc * (double)hi.y;
                    }
                } else {
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float2 f = bf2_to_f2(w[i]);
                        sum[2 * i + 0] += (double)f.x;
                        sum[2 * i + 1] += (double)f.y;
                    }
                }
            }
        }
        // add the token phases
        for (int off = nch; phases > 1 && off < 32; off <<= 1) {
#pragma unroll
            for (int i = 0; i < 16; ++i) sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], off);
        }
        if (active && ph == 0) {
            uint32_t packed[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // fp64 division is correctly rounded, as is the mean the
                // definition asks for; a product with 1/b is not when b is
                // not a power of two
                uint32_t lo = f64_to_bf16_rne(sum[2 * i] / db);
                uint32_t hi = f64_to_bf16_rne(sum[2 * i + 1] / db);
                packed[i] = lo | (hi << 16);
            }
            uint4 *d = reinterpret_cast<uint4 *>(dst + (int64_t)ch * epc);
            d[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            if (c.e4m3) d[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
    }
}

// Quest summaries of one block (page p, head h): the element-wise maximum
// and minimum of its b keys, written as [max (dk), min (dk)] bf16 (exact:
// they are key values).  Lanes own 8-dim chunks; rows wider than a warp take
// several chunks per lane.
template <bool kNonCoherent>
__device__ void minmax_block(const CacheView &c, int64_t p, int h, uint16_t *summ)
{
    const int lane = threadIdx.x & 31;
    const int nch = c.dk / 8;
    const uint8_t *base = c.k + (p * c.kps + (int64_t)h * c.khs) * 2;
    uint16_t *dst = summ + (p * c.hkv + h) * (int64_t)2 * c.dk;
    for (int ch = lane; ch < nch; ch += 32) {
        float mx[8], mn[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            mx[i] = -INFINITY;
            mn[i] = INFINITY;
        }
        for (int t = 0; t < c.b; ++t) {
            const uint4 v = load16<kNonCoherent>(base + (int64_t)t * c.kts * 2 + ch * 16);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = bf2_to_f2(w[i]);
                mx[2 * i] = fmaxf(mx[2 * i], f.x);
                mx[2 * i + 1] = fmaxf(mx[2 * i + 1], f.y);
                mn[2 * i] = fminf(mn[2 * i], f.x);
                mn[2 * i + 1] = fminf(mn[2 * i + 1], f.y);
            }
        }
        uint32_t px[4], pn[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // bf16 values held as floats: the upper halves are the bits
            px[i] = (__float_as_uint(mx[2 * i]) >> 16) | (__float_as_uint(mx[2 * i + 1]) & 0xffff0000u);
            pn[i] = (__float_as_uint(mn[2 * i]) >> 16) | (__float_as_uint(mn[2 * i + 1]) & 0xffff0000u);
        }
        *reinterpret_cast<uint4 *>(dst + ch * 8) = make_uint4(px[0], px[1], px[2], px[3]);
        *reinterpret_cast<uint4 *>(dst + c.dk + ch * 8) = make_uint4(pn[0], pn[1], pn[2], pn[3]);
    }
}

template <bool QUEST>
__global__ void __launch_bounds__(kWarpsPerCta * 32) k_build_summaries(SummaryArgs a)
{
    const int64_t item = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    const int64_t per_req = (int64_t)a.max_blocks * a.c.hkv;
    const int64_t r = item / per_req;
    if (r >= a.batch) return;
    const int64_t rem = item - r * per_req;
    const int j = (int)(rem / a.c.hkv);
    const int h = (int)(rem % a.c.hkv);
    int L = a.lens[r];
    if (L < 0 || (int64_t)L > (int64_t)a.max_blocks * a.c.b) {
        if ((threadIdx.x & 31) == 0 && j == 0 && h == 0) flag_error(a.status, LSA_ERR_BOUNDS);
        return;
    }
    if ((int64_t)(j + 1) * a.c.b > L) return;   // partial or unused block
    const int p = a.pt[r * a.max_blocks + j];
    if (p < 0 || p >= a.c.num_pages) {
        if ((threadIdx.x & 31) == 0) flag_error(a.status, LSA_ERR_BOUNDS);
        return;
    }
    if constexpr (QUEST) minmax_block<true>(a.c, p, h, a.summ);
    else summarize_block<true>(a.c, p, h, a.summ);
}

// One CTA per request, one warp per KV head: write the new token's key and
// value into its slot, and when that fills the block, summarize it.
template <bool QUEST>
__global__ void k_append(SummaryArgs a)
{
    const int r = blockIdx.x;
    const int h = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const CacheView &c = a.c;
    const int L = a.lens[r];
    __syncthreads();   // every warp has read the old length
    const int j = L / c.b, t = L % c.b;
    bool ok = L >= 0 && j < a.max_blocks;
    int p = ok ? a.pt[(int64_t)r * a.max_blocks + j] : -1;
    ok = ok && p >= 0 && p < c.num_pages;
    if (!ok) {
        if (lane == 0 && h == 0) flag_error(a.status, LSA_ERR_BOUNDS);
    } else {
        // key row
        const uint4 *ksrc = reinterpret_cast<const uint4 *>(a.k_new + ((int64_t)r * c.hkv + h) * c.dk);
        uint4 *kdst = reinterpret_cast<uint4 *>(
            const_cast<uint8_t *>(c.k) + ((int64_t)p * c.kps + (int64_t)h * c.khs + (int64_t)t * c.kts) * 2);
        for (int i = lane; i < c.dk / 8; i += 32) kdst[i] = ksrc[i];
        if (!c.v_alias) {
            const uint4 *vsrc = reinterpret_cast<const uint4 *>(a.v_new + ((int64_t)r * c.hkv + h) * c.dv);
            uint4 *vdst = reinterpret_cast<uint4 *>(
                const_cast<uint8_t *>(c.v) + ((int64_t)p * c.vps + (int64_t)h * c.vhs + (int64_t)t * c.vts) * 2);
            for (int i = lane; i < c.dv / 8; i += 32) vdst[i] = vsrc[i];
        }
        __syncwarp();
        if (t == c.b - 1) {
            __threadfence_block();
            if constexpr (QUEST) minmax_block<false>(c, p, h, a.summ);
            else summarize_block<false>(c, p, h, a.summ);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && ok) a.lens[r] = L + 1;
}

}  // namespace

cudaError_t launch_build_summaries(const SummaryArgs &a, cudaStream_t s, bool quest)
{
    const int64_t items = (int64_t)a.batch * a.max_blocks * a.c.hkv;
    if (items == 0) return cudaSuccess;
    const int64_t grid = (items + kWarpsPerCta - 1) / kWarpsPerCta;
    if (quest) k_build_summaries<true><<<(unsigned)grid, kWarpsPerCta * 32, 0, s>>>(a);
    else k_build_summaries<false><<<(unsigned)grid, kWarpsPerCta * 32, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_append(const SummaryArgs &a, cudaStream_t s, bool quest, bool *unsupported)
{
    *unsupported = a.c.e4m3 != 0 || a.c.hkv > 32 || (quest && a.c.dk % 8 != 0);
    if (*unsupported || a.batch == 0) return cudaSuccess;
    if (quest) k_append<true><<<a.batch, 32 * a.c.hkv, 0, s>>>(a);
    else k_append<false><<<a.batch, 32 * a.c.hkv, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace lsa

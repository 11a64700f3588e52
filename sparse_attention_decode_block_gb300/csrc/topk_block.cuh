// Exact top-k of one score row by one block of 256 threads (Vortex blog
// post, block top-k equation: the k largest scores, ties to the lower
// index, output in ascending column order).
//
// Thread t holds the keys of the contiguous columns [t*KPT, (t+1)*KPT) in
// registers (order-preserving 32-bit keys, 0 = not a candidate).  A lower
// bound on the k-th largest key comes cheaply from the threads' maxima: if
// lo0 is the k-th largest thread maximum, at least k threads hold a key
// >= lo0, so at least k keys are >= lo0, and on typical rows only a little
// more than k are.  Those keys are compacted in column order into shared
// memory (one block scan); every thread then ranks one or two of them
// against all (larger key first, then lower column), the k of rank < k are
// the selection and a second scan gives their ascending output positions.
// Rows where the bound leaves more than kTfCand keys (heavy ties) take a
// block-wide bisection over all keys instead.  Either way the result is the
// same exact, bit-reproducible selection.
#pragma once

#include "lsa_device.cuh"

namespace lsa {
namespace {

constexpr int kTfThreads = 256;
constexpr int kTfWarps = kTfThreads / 32;
constexpr int kTfCand = 512;   // candidates the final warp takes (16 per lane)

// Block-wide sum / max of one value per thread; every thread gets the
// result.  `red` holds kTfWarps words; two barriers.
__device__ __forceinline__ uint32_t tf_block_sum(uint32_t v, uint32_t *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_add_sync(0xffffffffu, v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < kTfWarps; ++w) t += red[w];
    __syncthreads();
    return t;
}

__device__ __forceinline__ uint32_t tf_block_max(uint32_t v, uint32_t *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = __reduce_max_sync(0xffffffffu, v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < kTfWarps; ++w) t = max(t, red[w]);
    __syncthreads();
    return t;
}

// Block-wide exclusive scan of one value per thread; *total gets the sum.
__device__ __forceinline__ uint32_t tf_block_scan(uint32_t v, uint32_t *red, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kTfWarps; ++w) {
        const uint32_t x = red[w];
        before += w < warp ? x : 0u;
        all += x;
    }
    __syncthreads();
    *total = all;
    return before + incl - v;
}

struct TopkScratch {
    uint32_t red[kTfWarps];
    uint32_t tmax[kTfThreads];
    uint32_t ck[kTfCand];
    int32_t cc[kTfCand];
    uint32_t lo;
};

// Selects the top min(k, candidates) columns of the row srow[0, n) (fp32
// scores; -inf = not a candidate; NaN = not a candidate, flagged) and calls
// out(position, column) for each; returns how many.  Every thread of the
// block (kTfThreads) must call it; KPT * kTfThreads >= n.  row_aligned: srow
// is 16-byte aligned (16-byte loads).
template <int KPT, class Out>
__device__ int block_topk(const float *srow, int n, bool row_aligned, int k, uint32_t *status, TopkScratch &sm,
                          Out out)
{
    static_assert(KPT % 4 == 0, "keys per thread come in fours");
    const int tid = threadIdx.x;
    const int c0 = tid * KPT;

    // keys (all loads first; 16-byte loads when the row is 16-byte aligned)
    float v[KPT];
    const bool vec = row_aligned && c0 + KPT <= n;
    if (vec) {
#pragma unroll
        for (int e = 0; e < KPT; e += 4) {
            const float4 f = *reinterpret_cast<const float4 *>(srow + c0 + e);
            v[e] = f.x;
            v[e + 1] = f.y;
            v[e + 2] = f.z;
            v[e + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < KPT; ++e) v[e] = c0 + e < n ? srow[c0 + e] : -INFINITY;
    }
    uint32_t keys[KPT];
    bool nan = false;
    uint32_t nvt = 0, m1 = 0;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
        nan |= isnan(v[e]);
        keys[e] = (isnan(v[e]) || v[e] == -INFINITY) ? 0u : float_to_key(v[e]);
        nvt += keys[e] != 0u;
        m1 = max(m1, keys[e]);
    }
    if (nan) flag_error(status, LSA_ERR_NAN);
    const int nv = (int)tf_block_sum(nvt, sm.red);
    const uint32_t kmax = tf_block_max(m1, sm.red);
    const int keff = min(k, nv);

    uint32_t thresh = 0;   // selection: keys > thresh, then the first take_eq keys == thresh
    int take_eq = 0;
    bool done = keff == 0;
    if (keff > 0 && keff < nv) {
        // lower bound: the keff-th largest thread maximum (1 when fewer than
        // keff threads hold a candidate), found by ranking every thread's
        // maximum against all the others (ties ranked by thread index)
        const int ntv = (int)tf_block_sum(m1 != 0u ? 1u : 0u, sm.red);
        sm.tmax[tid] = m1;
        if (tid == 0) sm.lo = 1u;
        __syncthreads();
        if (keff <= ntv && m1 != 0u) {
            int rank = 0;
            for (int u = 0; u < kTfThreads; ++u) {
                const uint32_t x = sm.tmax[u];
                rank += (x > m1) | ((x == m1) & (u < tid));
            }
            if (rank == keff - 1) sm.lo = m1;
        }
        __syncthreads();
        const uint32_t lo0 = sm.lo;
        uint32_t cnt = 0;
#pragma unroll
        for (int e = 0; e < KPT; ++e) cnt += keys[e] >= lo0;
        uint32_t C = 0;
        uint32_t pos = tf_block_scan(cnt, sm.red, &C);
        if (C <= (uint32_t)kTfCand) {
            // the candidates, in column order, to shared memory
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                if (keys[e] >= lo0) {
                    sm.ck[pos] = keys[e];
                    sm.cc[pos] = c0 + e;
                    ++pos;
                }
            }
            __syncthreads();
            // exact rank of candidates tid and tid + 256 (larger key first,
            // then lower column); the keff of rank < keff are the selection
            const int i0 = tid, i1 = tid + kTfThreads;
            const uint32_t k0 = i0 < (int)C ? sm.ck[i0] : 0u, k1 = i1 < (int)C ? sm.ck[i1] : 0u;
            int r0 = 0, r1 = 0;
            for (int j = 0; j < (int)C; ++j) {
                const uint32_t x = sm.ck[j];
                r0 += (x > k0) | ((x == k0) & (j < i0));
                r1 += (x > k1) | ((x == k1) & (j < i1));
            }
            const uint32_t f0 = (i0 < (int)C && r0 < keff) ? 1u : 0u, f1 = (i1 < (int)C && r1 < keff) ? 1u : 0u;
            uint32_t tot = 0;
            const uint32_t ex = tf_block_scan(f0 | (f1 << 16), sm.red, &tot);
            if (f0) out((int)(ex & 0xffffu), sm.cc[i0]);
            if (f1) out((int)((tot & 0xffffu) + (ex >> 16)), sm.cc[i1]);
            done = true;
        } else {
            // heavy ties: bisection over all keys of the row
            uint64_t lo = lo0, hi = (uint64_t)kmax + 1;
            while (hi - lo > 1) {
                const uint32_t mid = (uint32_t)(lo + ((hi - lo) >> 1));
                uint32_t c = 0;
#pragma unroll
                for (int e = 0; e < KPT; ++e) c += keys[e] >= mid;
                const int cs = (int)tf_block_sum(c, sm.red);
                if (cs >= keff) lo = mid;
                else hi = mid;
                if (cs == keff) break;
            }
            thresh = (uint32_t)lo;
            uint32_t g = 0;
#pragma unroll
            for (int e = 0; e < KPT; ++e) g += keys[e] > thresh;
            take_eq = keff - (int)tf_block_sum(g, sm.red);
        }
    }
    if (!done) {
        // every key > thresh and the first take_eq keys == thresh, in column
        // order (keff == nv: thresh = 0 takes every candidate)
        uint32_t pc = 0;
#pragma unroll
        for (int e = 0; e < KPT; ++e)
            pc += (keys[e] > thresh ? 1u : 0u) + (keys[e] != 0u && keys[e] == thresh ? 0x10000u : 0u);
        uint32_t total = 0;
        const uint32_t ex = tf_block_scan(pc, sm.red, &total);
        int gb = (int)(ex & 0xffffu), qb = (int)(ex >> 16);
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
            const bool gt = keys[e] > thresh, eq = keys[e] != 0u && keys[e] == thresh;
            if (gt || (eq && qb < take_eq)) out(gb + min(qb, take_eq), c0 + e);
            gb += gt;
            qb += eq;
        }
    }
    return keff;
}

}  // namespace
}  // namespace lsa

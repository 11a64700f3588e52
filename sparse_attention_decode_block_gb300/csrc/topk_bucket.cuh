// Exact top-k of one row by one block of NT threads, for rows of up to
// NT * KPT columns and any k (Vortex blog post, block top-k equation: the k
// largest scores, ties to the lower index, output in ascending column order).
//
// The selection buckets the scores by a monotone remap of their values
// (Vortex, "Making it fast": the radix top-k's buckets are spread by a
// monotone remap of the values).  Here the remap is linear between the
// row's smallest and largest candidate score, over kBkBins buckets: one
// pass of shared-memory counts, far less contended than the leading digits
// of the float bit patterns, which crowd into a few dozen bins.  The
// bucket that holds the k-th largest score is then resolved exactly: its
// few keys are ranked by (larger key, lower column).  Because the remap is
// monotone, every key in a higher bucket is at least every key in a lower
// one, so the selection is the exact top-k.  When the boundary bucket holds
// more than kBkCap keys (heavy ties or extreme skew) a bisection over the
// keys finds the threshold instead.  The stochastic early exit (approximate,
// opt-in) is the APPROX variant below.
#pragma once

#include "lsa_device.cuh"

namespace lsa {
namespace {

constexpr int kBkBins = 2048;
constexpr int kBkCap = 512;

template <int NT>
struct BucketScratch {
    uint32_t hist[kBkBins];
    uint32_t ck[kBkCap];          // keys of the boundary bucket, in column order
    uint8_t pick[kBkCap];         // selected among them
    uint32_t red[NT / 32][3];
    uint32_t bucket, gt, cnt;     // boundary bucket, keys in higher buckets, keys in it
};

// Block-wide exclusive scan of one value per thread; *total gets the sum.
// One barrier; the caller separates two uses of `red` by another barrier.
template <int NT>
__device__ __forceinline__ uint32_t bk_scan(uint32_t v, uint32_t (*red)[3], uint32_t *total)
{
    constexpr int W = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) red[warp][0] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) {
        const uint32_t x = red[w][0];
        before += w < warp ? x : 0u;
        all += x;
    }
    *total = all;
    return before + incl - v;
}

// Block-wide (sum, min, max) of one triple per thread; every thread gets the
// result.  Two barriers.
template <int NT>
__device__ __forceinline__ uint3 bk_sum_min_max(uint32_t s, uint32_t mn, uint32_t mx, uint32_t (*red)[3])
{
    constexpr int W = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    s = __reduce_add_sync(0xffffffffu, s);
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0) {
        red[warp][0] = s;
        red[warp][1] = mn;
        red[warp][2] = mx;
    }
    __syncthreads();
    uint3 r = make_uint3(0u, 0xffffffffu, 0u);
#pragma unroll
    for (int w = 0; w < W; ++w) {
        r.x += red[w][0];
        r.y = min(r.y, red[w][1]);
        r.z = max(r.z, red[w][2]);
    }
    __syncthreads();
    return r;
}

template <int NT>
__device__ __forceinline__ uint32_t bk_sum(uint32_t v, uint32_t (*red)[3])
{
    return bk_sum_min_max<NT>(v, 0u, 0u, red).x;
}

// SplitMix64 (Steele, Lea and Flood, OOPSLA 2014), counter style: output n
// (n >= 1) of the generator seeded with `seed` is the variant-13 finaliser
// of seed + n * 0x9e3779b97f4a7c15.
__host__ __device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t n)
{
    uint64_t z = seed + n * 0x9e3779b97f4a7c15ULL;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

// Selects the top min(k, candidates) of the keys (order-preserving, 0 = not a
// candidate) held KPT per thread, thread t holding columns [t*KPT, (t+1)*KPT),
// and calls out(position, column) for each selected column, positions in
// ascending column order; returns how many.  Every thread of the block must
// call it.
//
// APPROX: the stochastic early exit (Vortex, "Making it fast"): the keys in
// buckets above the boundary bucket are the confident winners, and the rest
// are sampled from the boundary bucket instead of ranked: numbered in column
// order 0 .. cnt-1, those within (k - winners) steps after sample mod cnt,
// circularly, are taken (sample: a SplitMix64 output drawn by the caller).
template <int NT, int KPT, bool APPROX = false, class Out>
__device__ int block_bucket_topk(const uint32_t (&keys)[KPT], int k, BucketScratch<NT> &sm, Out out,
                                 uint64_t sample = 0)
{
    static_assert(KPT <= 64, "selection mask of 64 bits");
    const int tid = threadIdx.x;
    const int c0 = tid * KPT;
    uint32_t nv = 0, kmn = 0xffffffffu, kmx = 0u;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
        if (keys[e] != 0u) {
            ++nv;
            kmn = min(kmn, keys[e]);
            kmx = max(kmx, keys[e]);
        }
    }
    const uint3 agg = bk_sum_min_max<NT>(nv, kmn, kmx, sm.red);
    const int nvalid = (int)agg.x;
    const int keff = min(max(k, 0), nvalid);
    if (keff == 0) return 0;

    uint64_t sel = 0;   // this thread's selected columns
    if (keff == nvalid) {
#pragma unroll
        for (int e = 0; e < KPT; ++e) sel |= (uint64_t)(keys[e] != 0u) << e;
    } else {
        // ---- buckets by the linear remap of the values between the row's
        // smallest and largest candidate (monotone: a larger key never lands
        // in a lower bucket)
        const float vmin = key_to_float(agg.y), vmax = key_to_float(agg.z);
        const float span = vmax - vmin;
        const float scale = (span > 0.f && span < INFINITY) ? (float)kBkBins / span : 0.f;
        auto bucket_of = [&](uint32_t key) -> int {
            if (scale == 0.f) return 0;
            const float x = (key_to_float(key) - vmin) * scale;
            return x >= (float)(kBkBins - 1) ? kBkBins - 1 : (int)x;
        };
        // each key's bucket, computed once (-1 for non-candidates)
        int bk[KPT];
#pragma unroll
        for (int e = 0; e < KPT; ++e) bk[e] = keys[e] != 0u ? bucket_of(keys[e]) : -1;
        for (int i = tid; i < kBkBins; i += NT) sm.hist[i] = 0u;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < KPT; ++e)
            if (bk[e] >= 0) atomicAdd(&sm.hist[bk[e]], 1u);
        __syncthreads();
        // thread t owns the BPT buckets below kBkBins - t * BPT; an exclusive
        // scan in thread order counts the keys in higher buckets
        constexpr int BPT = kBkBins / NT;
        static_assert(BPT >= 1 && kBkBins % NT == 0, "buckets per thread");
        const int top = kBkBins - 1 - tid * BPT;
        uint32_t cown = 0;
#pragma unroll
        for (int e = 0; e < BPT; ++e) cown += sm.hist[top - e];
        uint32_t tot = 0;
        uint32_t g = bk_scan<NT>(cown, sm.red, &tot);
#pragma unroll
        for (int e = 0; e < BPT; ++e) {
            const uint32_t cb = sm.hist[top - e];
            if (g < (uint32_t)keff && (uint32_t)keff <= g + cb) {
                sm.bucket = (uint32_t)(top - e);
                sm.gt = g;
                sm.cnt = cb;
            }
            g += cb;
        }
        __syncthreads();
        const int B = (int)sm.bucket;
        const int take = keff - (int)sm.gt;   // 1 .. cnt
        const int cnt = (int)sm.cnt;
        // every key in a higher bucket is selected; the boundary bucket's
        // keys are decided below
        uint64_t inb = 0;
        uint32_t nb = 0;
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
            sel |= (uint64_t)(bk[e] > B) << e;
            inb |= (uint64_t)(bk[e] == B) << e;
            nb += bk[e] == B;
        }
        if (APPROX) {
            uint32_t dummy = 0;
            const uint32_t base = bk_scan<NT>(nb, sm.red, &dummy);
            const uint32_t off = (uint32_t)(sample % (uint64_t)cnt);
            uint32_t pos = base;
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                if ((inb >> e) & 1ull) {
                    if ((pos + (uint32_t)cnt - off) % (uint32_t)cnt < (uint32_t)take) sel |= (uint64_t)1 << e;
                    ++pos;
                }
            }
        } else if (cnt <= kBkCap) {
            // the boundary bucket's keys, in column order, then each ranked
            // against all of them (larger key first, then lower column)
            uint32_t dummy = 0;
            const uint32_t base = bk_scan<NT>(nb, sm.red, &dummy);
            {
                uint32_t pos = base;
#pragma unroll
                for (int e = 0; e < KPT; ++e)
                    if ((inb >> e) & 1ull) sm.ck[pos++] = keys[e];
            }
            __syncthreads();
            for (int i = tid; i < cnt; i += NT) {
                const uint32_t me = sm.ck[i];
                int rank = 0;
                for (int j = 0; j < cnt; ++j) {
                    const uint32_t y = sm.ck[j];
                    rank += (y > me) || (y == me && j < i);
                }
                sm.pick[i] = rank < take ? 1 : 0;
            }
            __syncthreads();
            uint32_t pos = base;
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                if ((inb >> e) & 1ull) {
                    if (sm.pick[pos]) sel |= (uint64_t)1 << e;
                    ++pos;
                }
            }
        } else {
            // heavy ties: the threshold T, the keff-th largest key, by
            // bisection; every key > T and the first (keff - #{> T}) keys
            // equal to T in column order
            uint64_t lo = agg.y, hi = (uint64_t)agg.z + 1;
            while (hi - lo > 1) {
                const uint32_t mid = (uint32_t)(lo + ((hi - lo) >> 1));
                uint32_t c = 0;
#pragma unroll
                for (int e = 0; e < KPT; ++e) c += keys[e] >= mid;
                const int cs = (int)bk_sum<NT>(c, sm.red);
                if (cs >= keff) lo = mid;
                else hi = mid;
                if (cs == keff) break;
            }
            const uint32_t T = (uint32_t)lo;
            uint32_t ngt = 0, neq = 0;
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                ngt += keys[e] > T;
                neq += keys[e] != 0u && keys[e] == T;
            }
            const int take_eq = keff - (int)bk_sum<NT>(ngt, sm.red);
            uint32_t dummy = 0;
            uint32_t eqr = bk_scan<NT>(neq, sm.red, &dummy);
            sel = 0;   // the bucket pass's choices are replaced by the threshold's
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                if (keys[e] > T) sel |= (uint64_t)1 << e;
                else if (keys[e] != 0u && keys[e] == T) {
                    if ((int)eqr < take_eq) sel |= (uint64_t)1 << e;
                    ++eqr;
                }
            }
        }
    }
    // ---- output positions in column order
    __syncthreads();   // separates the scans above from the one below
    uint32_t total = 0;
    uint32_t pos = bk_scan<NT>((uint32_t)__popcll(sel), sm.red, &total);
#pragma unroll
    for (int e = 0; e < KPT; ++e)
        if ((sel >> e) & 1ull) out((int)pos++, c0 + e);
    __syncthreads();   // the scratch may be reused by the caller
    return keff;
}

}  // namespace
}  // namespace lsa

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
// memory (one block scan) and each is ranked against all of them (larger
// key first, then lower column): by a linear count over broadcast reads
// when there are few, else through warp-sorted runs and binary searches.
// The k of rank < k are the selection and a second scan gives their
// ascending output positions.  Rows where the bound leaves more than
// kTfCand keys (heavy ties) take a block-wide bisection over all keys
// instead.  Every way gives the same exact, bit-reproducible selection.
#pragma once

#include "lsa_device.cuh"

namespace lsa {
namespace {

constexpr int kTfThreads = 256;
constexpr int kTfWarps = kTfThreads / 32;
constexpr int kTfCand = 512;     // candidates ranked through sorted runs at most
constexpr int kTfLinear = 128;   // candidates ranked by a linear count at most
constexpr int kTfTreeK = 64;     // k up to which the bound comes from the top-64 tree

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

// Block-wide exclusive scan of one value per thread below 2^BITS: each bit
// plane is counted with a warp ballot, and the warps' totals go through
// `red`, read after one barrier.  No trailing barrier: a caller uses a given
// `red` again only after at least one more barrier.
template <int BITS>
__device__ __forceinline__ uint32_t tf_block_scan_small(uint32_t v, uint32_t *red, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t ex = 0, wt = 0;
#pragma unroll
    for (int b = 0; b < BITS; ++b) {
        const uint32_t m = __ballot_sync(0xffffffffu, (v >> b) & 1u);
        ex += (uint32_t)__popc(m & lt) << b;
        wt += (uint32_t)__popc(m) << b;
    }
    if (lane == 0) red[warp] = wt;
    __syncthreads();
    uint32_t before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kTfWarps; ++w) {
        const uint32_t x = red[w];
        before += w < warp ? x : 0u;
        all += x;
    }
    *total = all;
    return before + ex;
}

struct TopkScratch {
    unsigned long long runs[kTfCand];   // sorted runs of 32 candidate sort keys
    uint32_t red[kTfWarps];
    uint32_t red2[kTfWarps];            // the second scan of the small-k path
    uint32_t tmax[kTfThreads];          // sorted runs of 32 thread maxima
    alignas(16) uint32_t ck[kTfCand + 4];   // + 4: zero padding for 16-byte reads
    int32_t cc[kTfCand];
    uint32_t lo;
};
static_assert(sizeof(((TopkScratch *)nullptr)->runs) >= 512 * 4, "the top-64 tree reuses the runs");

// One value per lane, sorted across the warp in descending order (bitonic
// network: lane 0 ends with the largest).
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
            v = keep_max ? max(v, o) : min(v, o);
        }
    }
    return v;
}

__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
            v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
        }
    }
    return v;
}

// Sorts the 64-entry bitonic sequence (lane i holds entries i and 32 + i)
// in descending order: hi = entry i, lo = entry 32 + i afterwards.
__device__ __forceinline__ void warp_bitonic_merge64_desc(uint32_t &hi, uint32_t &lo)
{
    const int lane = threadIdx.x & 31;
    const uint32_t a = max(hi, lo), b = min(hi, lo);
    hi = a;
    lo = b;
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        const uint32_t oh = __shfl_xor_sync(0xffffffffu, hi, j);
        const uint32_t ol = __shfl_xor_sync(0xffffffffu, lo, j);
        const bool keep_max = (lane & j) == 0;
        hi = keep_max ? max(hi, oh) : min(hi, oh);
        lo = keep_max ? max(lo, ol) : min(lo, ol);
    }
}

// The k-th largest (1 <= k <= 64) of the block's 256 values v, one per
// thread; every thread gets it.  Each warp sorts its 32 values; sorted runs
// are then merged pairwise keeping the 64 largest (the largest 64 of two
// descending runs A, B are the bitonic sequence max(A[i], B[63 - i])).
// tree: 384 words of scratch.
__device__ __forceinline__ uint32_t block_kth_largest64(uint32_t v, int k, uint32_t *tree, uint32_t *out)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t *l0 = tree;          // 8 runs of 32, then (aliased) 2 runs of 64
    uint32_t *l1 = tree + 256;    // 4 runs of 64 -> first half of the buffer reused
    l0[warp * 32 + lane] = warp_sort_desc(v);
    __syncthreads();
    if (warp < 4) {   // runs 2w and 2w + 1 -> sorted 64
        uint32_t hi = l0[(2 * warp) * 32 + lane];
        uint32_t lo = l0[(2 * warp + 1) * 32 + 31 - lane];
        warp_bitonic_merge64_desc(hi, lo);
        l1[warp * 64 + lane] = hi;   // l1 spans tree[256, 512): 4 x 64 = 256 words
        l1[warp * 64 + 32 + lane] = lo;
    }
    __syncthreads();
    if (warp < 2) {   // sorted 64s 2w and 2w + 1 -> their top 64, sorted
        const uint32_t *A = l1 + (2 * warp) * 64, *B = l1 + (2 * warp + 1) * 64;
        uint32_t hi = max(A[lane], B[63 - lane]);
        uint32_t lo = max(A[32 + lane], B[31 - lane]);
        warp_bitonic_merge64_desc(hi, lo);
        l0[warp * 64 + lane] = hi;
        l0[warp * 64 + 32 + lane] = lo;
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t *A = l0, *B = l0 + 64;
        uint32_t hi = max(A[lane], B[63 - lane]);
        uint32_t lo = max(A[32 + lane], B[31 - lane]);
        warp_bitonic_merge64_desc(hi, lo);
        if (lane == ((k - 1) & 31)) *out = k <= 32 ? hi : lo;
    }
    __syncthreads();
    return *out;
}

// Entries > x (GE: >= x) in R descending runs of 32 stored one after the
// other.  Branch-free binary searches advanced in lockstep, so the R loads
// of a step are independent.
template <bool GE, int R, class T>
__device__ __forceinline__ int runs_count(const T *runs, T x)
{
    int p[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const T y = runs[32 * r + 31];
        p[r] = (GE ? y >= x : y > x) ? 32 : 0;
    }
#pragma unroll
    for (int step = 16; step > 0; step >>= 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const T y = runs[32 * r + min(p[r] + step - 1, 31)];
            p[r] += (p[r] < 32 && (GE ? y >= x : y > x)) ? step : 0;
        }
    }
    int t = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) t += p[r];
    return t;
}

// Entries > x and entries >= x in R descending runs of 32 stored one after
// the other: both binary searches of every run advanced in lockstep.
template <int R>
__device__ __forceinline__ void runs_count_gt_ge(const uint32_t *runs, uint32_t x, int &gt, int &ge)
{
    int pg[R], pe[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t y = runs[32 * r + 31];
        pg[r] = y > x ? 32 : 0;
        pe[r] = y >= x ? 32 : 0;
    }
#pragma unroll
    for (int step = 16; step > 0; step >>= 1) {
        uint32_t yg[R], ye[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            yg[r] = runs[32 * r + min(pg[r] + step - 1, 31)];
            ye[r] = runs[32 * r + min(pe[r] + step - 1, 31)];
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            pg[r] += (pg[r] < 32 && yg[r] > x) ? step : 0;
            pe[r] += (pe[r] < 32 && ye[r] >= x) ? step : 0;
        }
    }
    gt = 0;
    ge = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        gt += pg[r];
        ge += pe[r];
    }
}

// Selects the top min(k, candidates) columns of the row srow[0, n) (fp32
// scores; -inf = not a candidate; NaN = not a candidate, flagged) and calls
// out(position, column) for each; returns how many.  Every thread of the
// block (kTfThreads) must call it; KPT * kTfThreads >= n.  row_aligned: srow
// is 16-byte aligned (16-byte loads).
// This thread's scores of the row srow[0, n) for block_topk_scores: columns
// [t*KPT, (t+1)*KPT), -inf past n (16-byte loads when the row is 16-byte
// aligned).
template <int KPT>
__device__ __forceinline__ void block_topk_load(const float *srow, int n, bool row_aligned, float (&v)[KPT])
{
    static_assert(KPT % 4 == 0, "keys per thread come in fours");
    const int c0 = threadIdx.x * KPT;
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
}

template <int KPT, class Out>
__device__ int block_topk_scores(const float (&v)[KPT], int k, uint32_t *status, TopkScratch &sm, Out out);

template <int KPT, class Out>
__device__ int block_topk(const float *srow, int n, bool row_aligned, int k, uint32_t *status, TopkScratch &sm,
                          Out out)
{
    float v[KPT];
    block_topk_load<KPT>(srow, n, row_aligned, v);
    return block_topk_scores<KPT>(v, k, status, sm, out);
}

// block_topk on scores already loaded by block_topk_load.
template <int KPT, class Out>
__device__ int block_topk_scores(const float (&v)[KPT], int k, uint32_t *status, TopkScratch &sm, Out out)
{
    const int tid = threadIdx.x;
    const int c0 = tid * KPT;
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
    if (k > 0 && k <= kTfTreeK) {
        // lo0: the k-th largest thread maximum (1 when fewer than k threads
        // hold a candidate: then every candidate is taken).  The C keys >=
        // lo0 hold the selection; when C is small each is ranked by P
        // threads (larger key first, then lower column), each counting over
        // a P-th of the candidates with broadcast 16-byte reads.
        const uint32_t lo0 = max(block_kth_largest64(m1, k, reinterpret_cast<uint32_t *>(sm.runs), &sm.lo), 1u);
        uint32_t cnt = 0;
#pragma unroll
        for (int e = 0; e < KPT; ++e) cnt += keys[e] >= lo0;
        uint32_t C = 0;
        constexpr int kCntBits = KPT <= 8 ? 4 : KPT <= 32 ? 6 : 16;
        uint32_t pos = tf_block_scan_small<kCntBits>(cnt, sm.red, &C);
        if (C <= (uint32_t)kTfLinear) {
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                if (keys[e] >= lo0) {
                    sm.ck[pos] = keys[e];
                    sm.cc[pos] = c0 + e;
                    ++pos;
                }
            }
            if (tid < 4) sm.ck[C + tid] = 0u;   // never above a candidate, never equal to one
            __syncthreads();
            const int lp = C <= (uint32_t)(kTfThreads / 4) ? 2 : 1;   // log2 P
            const int i = tid >> lp, q = tid & ((1 << lp) - 1);
            uint32_t rank = 0;
            if (i < (int)C) {
                // (key, complement of the candidate index): one 64-bit
                // compare orders by larger key, then lower column
                using u64 = unsigned long long;
                const u64 me = ((u64)sm.ck[i] << 32) | (0xffffffffu - (uint32_t)i);
                const uint4 *ck4 = reinterpret_cast<const uint4 *>(sm.ck);
                const int n4 = ((int)C + 3) >> 2;
                const int per = (n4 + (1 << lp) - 1) >> lp;
                const int j4e = min(n4, (q + 1) * per);
#pragma unroll 4
                for (int j4 = q * per; j4 < j4e; ++j4) {
                    const uint4 y = ck4[j4];
                    const uint32_t nj = 0xffffffffu - 4u * (uint32_t)j4;
                    rank += (((u64)y.x << 32) | nj) > me;
                    rank += (((u64)y.y << 32) | (nj - 1u)) > me;
                    rank += (((u64)y.z << 32) | (nj - 2u)) > me;
                    rank += (((u64)y.w << 32) | (nj - 3u)) > me;
                }
            }
            rank += __shfl_xor_sync(0xffffffffu, rank, 1);
            if (lp == 2) rank += __shfl_xor_sync(0xffffffffu, rank, 2);
            const uint32_t f = (i < (int)C && q == 0 && rank < (uint32_t)k) ? 1u : 0u;
            uint32_t tot = 0;
            const uint32_t ex = tf_block_scan_small<1>(f, sm.red2, &tot);
            if (f) out((int)ex, sm.cc[i]);
            return min(k, (int)C);
        }
        __syncthreads();   // every read of the scan's red done before the general path reuses it
    }
    // candidate keys (low half) and threads holding one (high half)
    const uint32_t both = tf_block_sum(nvt | (m1 != 0u ? 0x10000u : 0u), sm.red);
    const int nv = (int)(both & 0xffffu), ntv = (int)(both >> 16);
    const int keff = min(k, nv);

    uint32_t thresh = 0;   // selection: keys > thresh, then the first take_eq keys == thresh
    int take_eq = 0;
    bool done = keff == 0;
    if (keff > 0 && keff < nv) {
        // lower bound: the keff-th largest thread maximum (1 when fewer than
        // keff threads hold a candidate).  Each warp sorts its 32 maxima; a
        // thread's maximum is the keff-th largest when fewer than keff
        // maxima are above it and at least keff are at or above it, counted
        // by binary search in the eight sorted runs.
        sm.tmax[tid] = warp_sort_desc(m1);
        if (tid == 0) sm.lo = 1u;
        __syncthreads();
        if (keff <= ntv && m1 != 0u) {
            int gt, ge;
            runs_count_gt_ge<kTfWarps>(sm.tmax, m1, gt, ge);
            if (gt < keff && keff <= ge) sm.lo = m1;   // every thread that writes writes the same value
        }
        __syncthreads();
        const uint32_t lo0 = sm.lo;
        uint32_t cnt = 0;
#pragma unroll
        for (int e = 0; e < KPT; ++e) cnt += keys[e] >= lo0;
        uint32_t C = 0;
        uint32_t pos = tf_block_scan(cnt, sm.red, &C);
        if (C <= (uint32_t)kTfLinear) {
            // the candidates, in column order, to shared memory; candidate
            // tid's rank (larger key first, then lower column) is counted
            // against all of them with broadcast 16-byte reads
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                if (keys[e] >= lo0) {
                    sm.ck[pos] = keys[e];
                    sm.cc[pos] = c0 + e;
                    ++pos;
                }
            }
            if (tid < 4) sm.ck[C + tid] = 0u;   // never above a candidate, never equal to one
            __syncthreads();
            uint32_t f = 0;
            if (tid < (int)C) {
                const uint32_t mine = sm.ck[tid];
                const uint4 *ck4 = reinterpret_cast<const uint4 *>(sm.ck);
                uint32_t rank = 0;
                const int n4 = ((int)C + 3) >> 2;
#pragma unroll 4
                for (int j4 = 0; j4 < n4; ++j4) {
                    const uint4 y = ck4[j4];
                    const int j = 4 * j4;
                    rank += (y.x > mine) | ((y.x == mine) & (j < tid));
                    rank += (y.y > mine) | ((y.y == mine) & (j + 1 < tid));
                    rank += (y.z > mine) | ((y.z == mine) & (j + 2 < tid));
                    rank += (y.w > mine) | ((y.w == mine) & (j + 3 < tid));
                }
                f = rank < (uint32_t)keff ? 1u : 0u;
            }
            uint32_t tot = 0;
            const uint32_t ex = tf_block_scan(f, sm.red, &tot);
            if (f) out((int)ex, sm.cc[tid]);
            done = true;
        } else if (C <= (uint32_t)kTfCand) {
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
            // exact rank of candidates tid and tid + 256: sort key = (key,
            // complement of the candidate index), unique and ordered like
            // (larger key first, then lower column); each warp sorts its
            // lanes' sort keys and a rank is a sum of binary searches in the
            // sorted runs.  The keff of rank < keff are the selection.
            const int i0 = tid, i1 = tid + kTfThreads;
            const bool two = C > (uint32_t)kTfThreads;   // block-uniform
            auto skey = [&](int i) -> unsigned long long {
                return i < (int)C ? ((unsigned long long)sm.ck[i] << 32) | (0xffffffffu - (uint32_t)i) : 0ull;
            };
            const unsigned long long s0 = skey(i0), s1 = two ? skey(i1) : 0ull;
            sm.runs[tid] = warp_sort_desc(s0);
            if (two) sm.runs[kTfThreads + tid] = warp_sort_desc(s1);
            __syncthreads();
            int r0, r1 = 0;
            if (two) {
                r0 = runs_count<false, kTfCand / 32>(sm.runs, s0);
                r1 = runs_count<false, kTfCand / 32>(sm.runs, s1);
            } else {
                r0 = runs_count<false, kTfThreads / 32>(sm.runs, s0);
            }
            const uint32_t f0 = (i0 < (int)C && r0 < keff) ? 1u : 0u;
            const uint32_t f1 = (two && i1 < (int)C && r1 < keff) ? 1u : 0u;
            uint32_t tot = 0;
            const uint32_t ex = tf_block_scan(f0 | (f1 << 16), sm.red, &tot);
            if (f0) out((int)(ex & 0xffffu), sm.cc[i0]);
            if (f1) out((int)((tot & 0xffffu) + (ex >> 16)), sm.cc[i1]);
            done = true;
        } else {
            // heavy ties: bisection over all keys of the row
            const uint32_t kmax = tf_block_max(m1, sm.red);
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

// Top-k of one long row by a thread-block cluster of CS CTAs of NT threads,
// KPT columns per thread (Vortex blog post, block top-k equation: the k
// largest scores, ties to the lower index, output in ascending column
// order).  The selection is the bucketed one of topk_bucket.cuh (a linear,
// monotone remap of the values over kBkBins buckets, then an exact ranking
// of the boundary bucket; a bisection when that bucket is crowded), with
// the row spread over the cluster: every CTA counts its own slice of the
// columns, and the CTAs exchange what the selection needs through
// distributed shared memory between cluster barriers, reading as little of
// each other's memory as they can:
//   - per-CTA scalars (counts, smallest and largest key) are read by one
//     warp, one lane per CTA;
//   - the bucket counts are summed by remote atomic adds into the CTA that
//     owns each slice of the buckets, and every CTA then reads all the sums
//     (one 16-byte load a thread) and finds the boundary itself;
//   - the boundary bucket's keys stay where they are counted; each CTA
//     gathers the cluster's list (at most kBkCap keys), ranks all of it, and
//     so knows every CTA's output count without another exchange.
// Four cluster barriers in the common case: extremes, counts, boundary
// lists, and the last one before any CTA may leave.
// No CTA waits on a flag; the barriers are the hardware's, and the
// cluster's CTAs are co-scheduled by construction.  The APPROX variant
// samples the boundary bucket instead (the stochastic early exit of
// topk_bucket.cuh).
#pragma once

#include "topk_bucket.cuh"

namespace lsa {
namespace {

template <int NT, int CS>
struct ClusterTopkScratch {
    static constexpr int SL = kBkBins / CS;   // buckets per slice
    uint32_t hist[kBkBins];                   // this CTA's bucket counts
    uint32_t part[NT / SL][SL];               // partial slice sums
    uint32_t ssum[SL];                        // slice `rank` of the cluster's counts
    uint32_t ck[kBkCap];                      // this CTA's boundary-bucket keys, in column order
    uint32_t ckall[kBkCap];                   // the cluster's, gathered
    uint8_t pick[kBkCap];
    uint32_t red[NT / 32][3];
    __align__(16) uint32_t xch[8][4];         // this CTA's values of each exchange
    uint32_t off[CS + 1];                     // per-CTA offsets of the current exchange
    uint32_t bc[4];                           // the cluster's candidate count, extremes, this CTA's offset
    uint32_t bucket, gt, cnt, pad;            // boundary bucket, keys above it, keys in it
};

// Sum over the cluster of word w of exchange slot s (written before the
// last cluster barrier), and the part from CTAs of lower rank than this
// one, read by warp 0 (one lane per CTA) and returned to every thread.
// Two CTA barriers; `red` is used.
template <int NT, int CS>
__device__ __forceinline__ uint32_t cl_gather_sum(ClusterTopkScratch<NT, CS> &sm, int s, int w, uint32_t *below)
{
    static_assert(CS <= 32, "one lane per CTA");
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < 32) {
        const uint32_t me = cluster_rank();
        const uint32_t v =
            lane < CS ? ld_cluster_u32(cluster_map(smem_addr(&sm.xch[s][w]), (uint32_t)lane)) : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t all = __shfl_sync(0xffffffffu, incl, 31);
        const uint32_t lo = __shfl_sync(0xffffffffu, incl - v, (int)me);
        if (lane == 0) {
            sm.red[0][0] = all;
            sm.red[0][1] = lo;
        }
    }
    __syncthreads();
    const uint32_t all = sm.red[0][0];
    if (below) *below = sm.red[0][1];
    __syncthreads();
    return all;
}

// Selects the top min(k, candidates) of the cluster's keys (order-preserving,
// 0 = not a candidate).  Thread t of the CTA of cluster rank c holds KPT keys
// whose columns increase with (c, t, e); col0 is this thread's first column.
// Calls out(position, col0 + e) for each selected key, positions in
// ascending column order over the whole cluster; returns how many were
// selected (the same in every CTA).  Every thread of every CTA of the
// cluster must call it; it ends with a cluster barrier.  APPROX and sample:
// the stochastic early exit of block_bucket_topk (topk_bucket.cuh), the
// boundary bucket numbered in column order over the whole cluster.
template <int NT, int KPT, int CS, bool APPROX = false, class Out>
__device__ int cluster_bucket_topk(const uint32_t (&keys)[KPT], int k, int col0, ClusterTopkScratch<NT, CS> &sm,
                                   Out out, uint64_t sample = 0)
{
    static_assert(KPT <= 64, "selection mask of 64 bits");
    constexpr int SL = ClusterTopkScratch<NT, CS>::SL;
    constexpr int BPT = kBkBins / NT;
    static_assert(SL % 4 == 0 && BPT % 4 == 0 && SL % BPT == 0, "slice layout");
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t me = cluster_rank();

    // ---- candidates, smallest and largest key over the cluster (the slice
    // sums this CTA owns are cleared before the barrier that precedes every
    // remote add to them)
    for (int i = tid; i < SL; i += NT) sm.ssum[i] = 0u;
    uint32_t nv = 0, kmn = 0xffffffffu, kmx = 0u;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
        if (keys[e] != 0u) {
            ++nv;
            kmn = min(kmn, keys[e]);
            kmx = max(kmx, keys[e]);
        }
    }
    const uint3 loc = bk_sum_min_max<NT>(nv, kmn, kmx, sm.red);
    if (tid == 0) {
        sm.xch[0][0] = loc.x;
        sm.xch[0][1] = loc.y;
        sm.xch[0][2] = loc.z;
    }
    cluster_sync();   // (1)
    if (tid < 32) {
        uint4 x = make_uint4(0u, 0xffffffffu, 0u, 0u);
        if (lane < CS) x = ld_cluster_v4(cluster_map(smem_addr(&sm.xch[0][0]), (uint32_t)lane));
        const uint32_t n = __reduce_add_sync(0xffffffffu, x.x);
        const uint32_t mn = __reduce_min_sync(0xffffffffu, x.y);
        const uint32_t mx = __reduce_max_sync(0xffffffffu, x.z);
        uint32_t incl = x.x;   // valid keys of the CTAs before each lane's
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t below = __shfl_sync(0xffffffffu, incl - x.x, (int)me);
        if (lane == 0) {
            sm.bc[0] = n;
            sm.bc[1] = mn;
            sm.bc[2] = mx;
            sm.bc[3] = below;
        }
    }
    __syncthreads();
    const uint32_t nvalid = sm.bc[0], gmn = sm.bc[1], gmx = sm.bc[2], nv_below = sm.bc[3];
    const int keff = min(max(k, 0), (int)nvalid);
    if (keff == 0) {
        cluster_sync();
        return 0;
    }

    uint64_t sel = 0;
    uint32_t base = 0;   // selected keys of the CTAs before this one
    bool need_exchange = false;
    if (keff == (int)nvalid) {
#pragma unroll
        for (int e = 0; e < KPT; ++e) sel |= (uint64_t)(keys[e] != 0u) << e;
        base = nv_below;
    } else {
        const float vmin = key_to_float(gmn), vmax = key_to_float(gmx);
        const float span = vmax - vmin;
        const float scale = (span > 0.f && span < INFINITY) ? (float)kBkBins / span : 0.f;
        int bk[KPT];
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
            int bb = -1;
            if (keys[e] != 0u) {
                bb = 0;
                if (scale != 0.f) {
                    const float x = (key_to_float(keys[e]) - vmin) * scale;
                    bb = x >= (float)(kBkBins - 1) ? kBkBins - 1 : (int)x;
                }
            }
            bk[e] = bb;
        }
        for (int i = tid; i < kBkBins; i += NT) sm.hist[i] = 0u;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < KPT; ++e)
            if (bk[e] >= 0) atomicAdd(&sm.hist[bk[e]], 1u);
        __syncthreads();
        // this CTA's counts into the owners' slice sums
        for (int i = tid; i < kBkBins; i += NT) {
            const uint32_t h = sm.hist[i];
            if (h) red_cluster_add_u32(cluster_map(smem_addr(&sm.ssum[i % SL]), (uint32_t)(i / SL)), h);
        }
        cluster_sync();   // (2) every slice sum is complete
        // thread t reads the cluster's counts of its BPT buckets below
        // kBkBins - t * BPT (16 bytes at a time) and an exclusive scan in
        // thread order counts the keys in higher buckets
        const int top = kBkBins - 1 - tid * BPT;
        uint32_t cb[BPT];
#pragma unroll
        for (int q = 0; q < BPT / 4; ++q) {
            const int lo = top - 4 * q - 3;   // 4 buckets lo .. lo + 3, one owner
            const uint4 v = ld_cluster_v4(cluster_map(smem_addr(&sm.ssum[lo % SL]), (uint32_t)(lo / SL)));
            cb[4 * q] = v.w;
            cb[4 * q + 1] = v.z;
            cb[4 * q + 2] = v.y;
            cb[4 * q + 3] = v.x;
        }
        uint32_t cown = 0;
#pragma unroll
        for (int e = 0; e < BPT; ++e) cown += cb[e];
        uint32_t tot = 0;
        uint32_t g = bk_scan<NT>(cown, sm.red, &tot);
#pragma unroll
        for (int e = 0; e < BPT; ++e) {
            if (g < (uint32_t)keff && (uint32_t)keff <= g + cb[e]) {
                sm.bucket = (uint32_t)(top - e);
                sm.gt = g;
                sm.cnt = cb[e];
            }
            g += cb[e];
        }
        __syncthreads();
        const int B = (int)sm.bucket;
        const int take = keff - (int)sm.gt;   // 1 .. cnt
        const int cnt = (int)sm.cnt;
        uint64_t inb = 0;
        uint32_t nb = 0, nw = 0;
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
            sel |= (uint64_t)(bk[e] > B) << e;
            inb |= (uint64_t)(bk[e] == B) << e;
            nb += bk[e] == B;
            nw += bk[e] > B;
        }
        if (APPROX || cnt <= kBkCap) {
            // the boundary bucket's keys in column order over the cluster:
            // this CTA's after those of lower ranks; with them every CTA's
            // winners, so that each CTA knows every CTA's output count
            uint32_t nbc = 0, nwc = 0;
            const uint32_t lbase = bk_scan<NT>(nb, sm.red, &nbc);
            __syncthreads();   // the scan's reads of red are done before it is reused
            nwc = bk_sum<NT>(nw, sm.red);
            if (!APPROX) {
                uint32_t pos = lbase;
#pragma unroll
                for (int e = 0; e < KPT; ++e)
                    if ((inb >> e) & 1ull) sm.ck[pos++] = keys[e];
            }
            if (tid == 0) {
                sm.xch[1][0] = nbc;
                sm.xch[1][1] = nwc;
            }
            cluster_sync();   // (3)
            if (tid < 32) {
                uint32_t vb = 0, vw = 0;
                if (lane < CS) {
                    vb = ld_cluster_u32(cluster_map(smem_addr(&sm.xch[1][0]), (uint32_t)lane));
                    vw = ld_cluster_u32(cluster_map(smem_addr(&sm.xch[1][1]), (uint32_t)lane));
                }
                uint32_t incl = vb;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
                if (lane < CS) sm.off[lane] = incl - vb;
                if (lane == 0) sm.off[CS] = total;
                // winners of the CTAs before this one
                uint32_t iw = vw;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, iw, o);
                    if (lane >= o) iw += y;
                }
                const uint32_t wb = __shfl_sync(0xffffffffu, iw - vw, (int)me);
                if (lane == 0) sm.bc[3] = wb;
            }
            __syncthreads();
            const uint32_t cbase = sm.off[me];
            if (!APPROX) {
                // gather the cluster's boundary keys and rank all of them
                for (int gi = tid; gi < cnt; gi += NT) {
                    int owner = 0;
#pragma unroll
                    for (int c = 1; c < CS; ++c) owner += (uint32_t)gi >= sm.off[c];
                    sm.ckall[gi] = ld_cluster_u32(
                        cluster_map(smem_addr(&sm.ck[gi - (int)sm.off[owner]]), (uint32_t)owner));
                }
                __syncthreads();
                for (int gi = tid; gi < cnt; gi += NT) {
                    const uint32_t mine = sm.ckall[gi];
                    int rank = 0;
                    for (int j = 0; j < cnt; ++j) {
                        const uint32_t y = sm.ckall[j];
                        rank += (y > mine) || (y == mine && j < gi);
                    }
                    sm.pick[gi] = rank < take ? 1 : 0;
                }
                __syncthreads();
            }
            // boundary keys taken by the CTAs before this one
            const uint32_t off = APPROX ? (uint32_t)(sample % (uint64_t)cnt) : 0u;
            auto taken = [&](uint32_t gi) -> bool {
                return APPROX ? (gi + (uint32_t)cnt - off) % (uint32_t)cnt < (uint32_t)take : sm.pick[gi] != 0;
            };
            uint32_t tb = 0;
            for (uint32_t gi = (uint32_t)tid; gi < cbase; gi += NT) tb += taken(gi) ? 1u : 0u;
            tb = bk_sum<NT>(tb, sm.red);
            base = sm.bc[3] + tb;
            uint32_t pos = cbase + lbase;
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                if ((inb >> e) & 1ull) {
                    if (taken(pos)) sel |= (uint64_t)1 << e;
                    ++pos;
                }
            }
        } else {
            // heavy ties: the threshold T, the keff-th largest key, by a
            // bisection whose counts are summed over the cluster (two
            // exchange slots alternate: a slot is rewritten only after the
            // barrier that follows every CTA's reads of it)
            uint64_t lo = gmn, hi = (uint64_t)gmx + 1;
            int it = 0;
            while (hi - lo > 1) {
                const uint32_t mid = (uint32_t)(lo + ((hi - lo) >> 1));
                uint32_t c = 0;
#pragma unroll
                for (int e = 0; e < KPT; ++e) c += keys[e] >= mid;
                const uint32_t cc = bk_sum<NT>(c, sm.red);
                const int slot = 3 + (it & 1);
                if (tid == 0) sm.xch[slot][0] = cc;
                cluster_sync();
                const int cs = (int)cl_gather_sum<NT, CS>(sm, slot, 0, nullptr);
                if (cs >= keff) lo = mid;
                else hi = mid;
                ++it;
                if (cs == keff) break;
            }
            const uint32_t T = (uint32_t)lo;
            uint32_t ngt = 0, neq = 0;
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                ngt += keys[e] > T;
                neq += keys[e] != 0u && keys[e] == T;
            }
            const uint32_t ngt_cta = bk_sum<NT>(ngt, sm.red);
            uint32_t neq_cta = 0;
            const uint32_t leq = bk_scan<NT>(neq, sm.red, &neq_cta);
            if (tid == 0) {
                sm.xch[5][0] = ngt_cta;
                sm.xch[5][1] = neq_cta;
            }
            cluster_sync();
            __syncthreads();   // bk_scan's reads of red are done before it is reused
            const int take_eq = keff - (int)cl_gather_sum<NT, CS>(sm, 5, 0, nullptr);
            uint32_t eq_below = 0;
            cl_gather_sum<NT, CS>(sm, 5, 1, &eq_below);
            uint32_t eqr = eq_below + leq;
            sel = 0;
#pragma unroll
            for (int e = 0; e < KPT; ++e) {
                if (keys[e] > T) sel |= (uint64_t)1 << e;
                else if (keys[e] != 0u && keys[e] == T) {
                    if ((int)eqr < take_eq) sel |= (uint64_t)1 << e;
                    ++eqr;
                }
            }
            need_exchange = true;
        }
    }
    // ---- output positions in column order over the cluster
    __syncthreads();
    uint32_t tot = 0;
    uint32_t lpos = bk_scan<NT>((uint32_t)__popcll(sel), sm.red, &tot);
    if (need_exchange) {
        // (the bisection path) every CTA's output count
        if (tid == 0) sm.xch[6][0] = tot;
        cluster_sync();
        __syncthreads();
        cl_gather_sum<NT, CS>(sm, 6, 0, &base);
    }
    uint32_t pos = base + lpos;
#pragma unroll
    for (int e = 0; e < KPT; ++e)
        if ((sel >> e) & 1ull) out((int)pos++, col0 + e);
    cluster_sync();   // (4) no CTA leaves, or reuses the scratch, while another reads it
    return keff;
}

}  // namespace
}  // namespace lsa

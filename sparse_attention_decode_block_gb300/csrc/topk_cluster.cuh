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
//   - the bucket counts are reduce-scattered: CTA c sums bucket slice c
//     over the cluster, and every CTA then reads the slice totals and the
//     one slice that holds the boundary;
//   - the boundary bucket's keys stay where they are counted; each CTA
//     gathers the cluster's list (at most kBkCap keys) to rank its own.
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
    uint32_t bc[4];                           // boundary bucket, keys above it, keys in it
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
    static_assert(SL % 32 == 0 && NT % SL == 0 && CS % (NT / SL) == 0, "slice layout");
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t me = cluster_rank();

    // ---- candidates, smallest and largest key over the cluster
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
    cluster_sync();
    if (tid < 32) {
        uint4 x = make_uint4(0u, 0xffffffffu, 0u, 0u);
        if (lane < CS) x = ld_cluster_v4(cluster_map(smem_addr(&sm.xch[0][0]), (uint32_t)lane));
        const uint32_t n = __reduce_add_sync(0xffffffffu, x.x);
        const uint32_t mn = __reduce_min_sync(0xffffffffu, x.y);
        const uint32_t mx = __reduce_max_sync(0xffffffffu, x.z);
        if (lane == 0) {
            sm.bc[0] = n;
            sm.bc[1] = mn;
            sm.bc[2] = mx;
        }
    }
    __syncthreads();
    const uint32_t nvalid = sm.bc[0], gmn = sm.bc[1], gmx = sm.bc[2];
    const int keff = min(max(k, 0), (int)nvalid);
    if (keff == 0) {
        cluster_sync();
        return 0;
    }

    uint64_t sel = 0;
    if (keff == (int)nvalid) {
#pragma unroll
        for (int e = 0; e < KPT; ++e) sel |= (uint64_t)(keys[e] != 0u) << e;
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
        __syncthreads();   // every thread has read bc before it is rewritten below
        for (int i = tid; i < kBkBins; i += NT) sm.hist[i] = 0u;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < KPT; ++e)
            if (bk[e] >= 0) atomicAdd(&sm.hist[bk[e]], 1u);
        cluster_sync();   // every CTA's counts are complete
        // reduce-scatter: this CTA sums slice `me` (buckets me*SL ..) over
        // the cluster; thread (group g, bucket j) adds CS / NG ranks
        {
            constexpr int NG = NT / SL, RPG = CS / NG;
            const int j = tid % SL, g = tid / SL;
            const uint32_t a = smem_addr(&sm.hist[me * SL + j]);
            uint32_t v[RPG];
#pragma unroll
            for (int i = 0; i < RPG; ++i) v[i] = ld_cluster_u32(cluster_map(a, (uint32_t)(g * RPG + i)));
            uint32_t s = 0;
#pragma unroll
            for (int i = 0; i < RPG; ++i) s += v[i];
            sm.part[g][j] = s;
            __syncthreads();
            uint32_t t = 0;
            if (tid < SL) {
#pragma unroll
                for (int i = 0; i < NG; ++i) t += sm.part[i][tid];
                sm.ssum[tid] = t;
            }
            const uint32_t tot = bk_sum<NT>(t, sm.red);
            if (tid == 0) sm.xch[1][0] = tot;
        }
        cluster_sync();   // every slice sum is complete
        // every CTA finds the boundary: the slice that holds the keff-th
        // largest key (slice totals, one lane per CTA), then the bucket
        // within that slice (its SL sums, SL / 32 per lane)
        if (tid < 32) {
            const uint32_t tot =
                lane < CS ? ld_cluster_u32(cluster_map(smem_addr(&sm.xch[1][0]), (uint32_t)lane)) : 0u;
            // keys in this lane's slice and the ones above it
            uint32_t suf = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += y;
            }
            const uint32_t above_s = suf - tot;
            const unsigned hit =
                __ballot_sync(0xffffffffu, lane < CS && above_s < (uint32_t)keff && (uint32_t)keff <= suf);
            // exactly one slice holds it; were none found, no bucket is
            // either, and the crowded-boundary count below sends the
            // selection to the bisection, which needs no boundary
            const int cs_ = hit ? __ffs(hit) - 1 : 0;
            if (lane == 0) sm.bc[2] = 0x7fffffffu;
            __syncwarp();
            const uint32_t above = __shfl_sync(0xffffffffu, above_s, cs_);
            constexpr int SPL = SL / 32;
            uint32_t c[SPL];
            const uint32_t a = cluster_map(smem_addr(&sm.ssum[lane * SPL]), (uint32_t)cs_);
#pragma unroll
            for (int i = 0; i < SPL; ++i) c[i] = ld_cluster_u32(a + 4 * i);
            uint32_t ls = 0;
#pragma unroll
            for (int i = 0; i < SPL; ++i) ls += c[i];
            uint32_t lsuf = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, lsuf, o);
                if (lane + o < 32) lsuf += y;
            }
            uint32_t g = above + lsuf - ls;   // keys above this lane's buckets
#pragma unroll
            for (int i = SPL - 1; i >= 0; --i) {
                if (g < (uint32_t)keff && (uint32_t)keff <= g + c[i]) {
                    sm.bc[0] = (uint32_t)(cs_ * SL + lane * SPL + i);
                    sm.bc[1] = g;
                    sm.bc[2] = c[i];
                }
                g += c[i];
            }
        }
        __syncthreads();
        const int B = (int)sm.bc[0];
        const int take = keff - (int)sm.bc[1];   // 1 .. cnt
        const int cnt = (int)sm.bc[2];
        uint64_t inb = 0;
        uint32_t nb = 0;
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
            sel |= (uint64_t)(bk[e] > B) << e;
            inb |= (uint64_t)(bk[e] == B) << e;
            nb += bk[e] == B;
        }
        if (APPROX || cnt <= kBkCap) {
            // the boundary bucket's keys in column order over the cluster:
            // this CTA's after those of lower ranks
            uint32_t nbc = 0;
            const uint32_t lbase = bk_scan<NT>(nb, sm.red, &nbc);
            if (!APPROX) {
                uint32_t pos = lbase;
#pragma unroll
                for (int e = 0; e < KPT; ++e)
                    if ((inb >> e) & 1ull) sm.ck[pos++] = keys[e];
            }
            if (tid == 0) sm.xch[2][0] = nbc;
            cluster_sync();
            if (tid < 32) {
                const uint32_t v =
                    lane < CS ? ld_cluster_u32(cluster_map(smem_addr(&sm.xch[2][0]), (uint32_t)lane)) : 0u;
                uint32_t incl = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);   // every lane takes part
                if (lane < CS) sm.off[lane] = incl - v;
                if (lane == 0) sm.off[CS] = total;
            }
            __syncthreads();
            const uint32_t cbase = sm.off[me];
            if (APPROX) {
                const uint32_t off = (uint32_t)(sample % (uint64_t)cnt);
                uint32_t pos = cbase + lbase;
#pragma unroll
                for (int e = 0; e < KPT; ++e) {
                    if ((inb >> e) & 1ull) {
                        if ((pos + (uint32_t)cnt - off) % (uint32_t)cnt < (uint32_t)take) sel |= (uint64_t)1 << e;
                        ++pos;
                    }
                }
            } else {
                // gather the cluster's boundary keys, then rank this CTA's
                for (int gi = tid; gi < cnt; gi += NT) {
                    int owner = 0;
#pragma unroll
                    for (int c = 1; c < CS; ++c) owner += (uint32_t)gi >= sm.off[c];
                    sm.ckall[gi] = ld_cluster_u32(
                        cluster_map(smem_addr(&sm.ck[gi - (int)sm.off[owner]]), (uint32_t)owner));
                }
                __syncthreads();
                for (int i = tid; i < (int)nbc; i += NT) {
                    const int gi = (int)cbase + i;
                    const uint32_t mine = sm.ckall[gi];
                    int rank = 0;
                    for (int j = 0; j < cnt; ++j) {
                        const uint32_t y = sm.ckall[j];
                        rank += (y > mine) || (y == mine && j < gi);
                    }
                    sm.pick[i] = rank < take ? 1 : 0;
                }
                __syncthreads();
                uint32_t pos = lbase;
#pragma unroll
                for (int e = 0; e < KPT; ++e) {
                    if ((inb >> e) & 1ull) {
                        if (sm.pick[pos]) sel |= (uint64_t)1 << e;
                        ++pos;
                    }
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
        }
    }
    // ---- output positions in column order over the cluster
    __syncthreads();
    uint32_t tot = 0;
    uint32_t lpos = bk_scan<NT>((uint32_t)__popcll(sel), sm.red, &tot);
    if (tid == 0) sm.xch[6][0] = tot;
    cluster_sync();
    __syncthreads();   // bk_scan's reads of red are done before it is reused
    uint32_t below = 0;
    cl_gather_sum<NT, CS>(sm, 6, 0, &below);
    uint32_t pos = below + lpos;
#pragma unroll
    for (int e = 0; e < KPT; ++e)
        if ((sel >> e) & 1ull) out((int)pos++, col0 + e);
    cluster_sync();   // no CTA leaves, or reuses the scratch, while another reads it
    return keff;
}

}  // namespace
}  // namespace lsa

// Block scoring, exact radix top-k, and the FP8 fine rescoring of the
// coarse-to-fine variant.
//
// Scores: s_j = q . k_bar_j (Vortex blog post, block top-k equation),
// summed over the query heads of one KV head's group.  Because the score is
// linear in q, the group's queries are summed once (q_sum = sum_g q_g, fp32)
// and each summary row is read once with 16-byte loads and dotted with q_sum.
//
// Top-k of wide rows or large k: one CTA per row buckets the scores by a
// monotone remap of their values and ranks the boundary bucket exactly
// (topk_bucket.cuh; Vortex, "Making it fast").  Ties go to the lower index
// and the output is ascending, so the result is bit-exact.
#include <math.h>

#include <mutex>
#include <type_traits>

#include "lsa_device.cuh"
#include "topk_bucket.cuh"
#include "topk_cluster.cuh"

namespace lsa {
namespace {

// ============================================================ scoring

constexpr int kScoreWarps = 8;
constexpr int kScoreMaxChunk = 1024;   // blocks per CTA at most
constexpr int kPtPerThread = kScoreMaxChunk / (kScoreWarps * 32);

// One CTA scores a contiguous chunk of one request's blocks; each warp takes
// a contiguous share of the chunk.  The prologue is one memory round trip:
// the request length, the chunk's page ids and the group's queries are all
// loaded before anything is stored; the group's query sum goes to shared
// memory once per CTA.  The main loop keeps U summary rows in flight per
// warp at all times: each row's registers are refilled with the row U ahead
// as soon as its dot products are done.
template <int DK, int HKV>
__global__ void __launch_bounds__(kScoreWarps * 32, 2) k_score(ScoreArgs a)
{
    pdl_enter();
    constexpr int NCH = HKV * DK / 8;      // 16-byte chunks of one page's summary row
    constexpr int NI = (NCH + 31) / 32;    // chunks per lane
    constexpr int CPH = DK / 8;            // chunks per head
    constexpr int U = NI <= 4 ? 4 : 2;     // rows in flight per warp
    constexpr bool kGroupReduce = (CPH <= 32) && (32 % CPH == 0);
    static_assert(kGroupReduce || HKV == 1, "head rows must tile the warp");
    __shared__ int s_page[kScoreMaxChunk];
    __shared__ __align__(16) float s_qs[HKV * DK];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.y;
    const int G = a.hq / HKV;
    const int j0 = blockIdx.x * a.chunk;
    const int j1 = min(j0 + a.chunk, a.max_blocks);

    // ---- prologue: every load first (one round trip), then the stores
    const int L = a.lens[r];
    int praw[kPtPerThread];
#pragma unroll
    for (int i = 0; i < kPtPerThread; ++i) {
        const int j = j0 + tid + i * kScoreWarps * 32;
        praw[i] = j < j1 ? a.pt[(int64_t)r * a.max_blocks + j] : -1;
    }
    // the group's query sum, one 8-dim slice of one head per thread (NCH <=
    // threads for every supported shape).  Up to 8 heads a thread adds them
    // in head order; larger groups are cut into QSL slices of heads whose
    // loads are all issued at once, and the slices are added in slice order
    constexpr int QSL = (kScoreWarps * 32) / NCH;
    static_assert(QSL >= 1, "one thread per 16-byte chunk of the summary row");
    __shared__ __align__(16) float s_qpart[QSL > 1 ? QSL * NCH * 8 : 1];
    float qacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int qc = tid % NCH, qsl = tid / NCH;   // chunk, slice
    const int qh = qc / CPH, qd = (qc % CPH) * 8;
    const bool sliced = G > 8 && QSL > 1;
    if (!sliced && tid < NCH) {
        const uint16_t *qp = a.q + ((int64_t)r * a.hq + qh * G) * DK + qd;
        for (int g0 = 0; g0 < G; g0 += 4) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = g0 + u < G ? *reinterpret_cast<const uint4 *>(qp + (int64_t)(g0 + u) * DK) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = bf2_to_f2(w[e]);
                    qacc[2 * e] += f.x;
                    qacc[2 * e + 1] += f.y;
                }
            }
        }
    } else if (sliced && qsl < QSL) {
        // heads qsl, qsl + QSL, ...: at most 32 per thread (G <= 32 * QSL)
        const uint16_t *qp = a.q + ((int64_t)r * a.hq + qh * G) * DK + qd;
        for (int g0 = qsl; g0 < G; g0 += 8 * QSL) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int g = g0 + u * QSL;
                v[u] = g < G ? *reinterpret_cast<const uint4 *>(qp + (int64_t)g * DK) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = bf2_to_f2(w[e]);
                    qacc[2 * e] += f.x;
                    qacc[2 * e + 1] += f.y;
                }
            }
        }
        if constexpr (QSL > 1) {
#pragma unroll
            for (int e = 0; e < 8; ++e) s_qpart[(qsl * NCH + qc) * 8 + e] = qacc[e];
        }
    }
    const bool len_ok = L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * a.b;
    if (!len_ok && tid == 0 && blockIdx.x == 0) flag_error(a.status, LSA_ERR_BOUNDS);
    const int se = len_ok ? min(a.sink, L) : 0;
    const int rs = len_ok ? max(L - a.recent, se) : 0;
#pragma unroll
    for (int i = 0; i < kPtPerThread; ++i) {
        const int j = j0 + tid + i * kScoreWarps * 32;
        if (j >= j1) continue;
        const bool cand = len_ok && (int64_t)j * a.b >= se && (int64_t)(j + 1) * a.b <= rs;
        int p = cand ? praw[i] : -1;
        if (cand && (p < 0 || p >= a.num_pages)) {
            flag_error(a.status, LSA_ERR_BOUNDS);
            p = -1;
        }
        s_page[j - j0] = p;
        if (p < 0) {
#pragma unroll
            for (int h = 0; h < HKV; ++h) a.scores[((int64_t)r * HKV + h) * a.max_blocks + j] = -INFINITY;
        }
    }
    if (!sliced && tid < NCH) {
#pragma unroll
        for (int e = 0; e < 8; ++e) s_qs[qh * DK + qd + e] = qacc[e];
    }
    if constexpr (QSL > 1) {
        if (sliced) {
            __syncthreads();
            if (tid < NCH) {
                float t8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int sl = 0; sl < QSL; ++sl)
#pragma unroll
                    for (int e = 0; e < 8; ++e) t8[e] += s_qpart[(sl * NCH + tid) * 8 + e];
#pragma unroll
                for (int e = 0; e < 8; ++e) s_qs[qh * DK + qd + e] = t8[e];
            }
        }
    }
    __syncthreads();

    // ---- this lane's slice of the query sum.  Rows narrower than a warp
    // (NCH < 32 chunks) are taken R at a time, NCH lanes each.
    constexpr int R = NCH < 32 ? 32 / NCH : 1;
    static_assert(R == 1 || (NI == 1 && 32 % NCH == 0), "narrow rows tile the warp");
    constexpr int UR = (NI == 1 ? 8 : U);   // row groups in flight per warp
    const int sr = R > 1 ? lane / NCH : 0;  // this lane's row within a group
    const int lc = R > 1 ? lane % NCH : lane;
    float qs[NI][8];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int ch = lc + 32 * i;
#pragma unroll
        for (int e = 0; e < 8; ++e) qs[i][e] = ch < NCH ? s_qs[(ch / CPH) * DK + (ch % CPH) * 8 + e] : 0.f;
    }

    // ---- main loop over the warp's share [w0, w1) of the chunk
    const int n = j1 - j0;
    const int w0 = (int)((int64_t)n * warp / kScoreWarps), w1 = (int)((int64_t)n * (warp + 1) / kScoreWarps);
    const uint8_t *summ = reinterpret_cast<const uint8_t *>(a.summ);
    const uint64_t pol = l2_evict_first();
    uint4 v[UR][NI];
    // row group gi covers rows w0 + gi * R + [0, R)
    auto issue = [&](int i, uint4(&dst)[NI]) {
        const int p = i < w1 ? s_page[i] : -1;
#pragma unroll
        for (int c = 0; c < NI; ++c) {
            const int ch = lc + 32 * c;
            dst[c] = (p >= 0 && ch < NCH) ? ldg_stream_v4(summ + (int64_t)p * HKV * DK * 2 + ch * 16, pol)
                                          : make_uint4(0, 0, 0, 0);
        }
    };
#pragma unroll
    for (int u = 0; u < UR; ++u) issue(w0 + u * R + sr, v[u]);
    for (int base = w0; base < w1; base += UR * R) {
#pragma unroll
        for (int u = 0; u < UR; ++u) {
            const int i = base + u * R + sr;
            const int p = i < w1 ? s_page[i] : -1;      // warp-uniform when R == 1
            const bool any = R > 1 ? __any_sync(0xffffffffu, p >= 0) : p >= 0;
            if (any) {
                const int j = j0 + i;
                float part[NI];
#pragma unroll
                for (int c = 0; c < NI; ++c) {
                    const uint32_t w[4] = {v[u][c].x, v[u][c].y, v[u][c].z, v[u][c].w};
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc = __ffma2_rn(make_float2(qs[c][2 * e], qs[c][2 * e + 1]), bf2_to_f2(w[e]), acc);
                    part[c] = acc.x + acc.y;
                }
                if constexpr (kGroupReduce) {
#pragma unroll
                    for (int c = 0; c < NI; ++c) {
#pragma unroll
                        for (int off = CPH / 2; off > 0; off >>= 1)
                            part[c] += __shfl_xor_sync(0xffffffffu, part[c], off);
                        const int ch = lc + 32 * c;
                        if (p >= 0 && ch < NCH && (lane % CPH) == 0)
                            a.scores[((int64_t)r * HKV + ch / CPH) * a.max_blocks + j] = part[c];
                    }
                } else {
                    float tot = 0.f;
#pragma unroll
                    for (int c = 0; c < NI; ++c) tot += part[c];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
                    if (lane == 0) a.scores[(int64_t)r * a.max_blocks + j] = tot;
                }
            }
            issue(i + UR * R, v[u]);
        }
    }
}

// ============================================================ Quest scores

// Halves per-lane partials across the lane pair that differs in `bit`:
// the lane with the bit clear keeps the lower half of the entries (summed
// with its partner's), the other lane the upper half.
template <int N>
__device__ __forceinline__ void halve_sum(const float (&v)[N], float (&out)[N / 2], int bit)
{
    const bool up = (threadIdx.x & bit) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float send = up ? v[i] : v[N / 2 + i];
        out[i] = (up ? v[N / 2 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, send, bit);
    }
}

// The maximum over G heads of each head's sum over an aligned group of T
// lanes (T a power of two, G <= T): log2 G reduce-scatter steps on the
// group's top lane bits leave each lane one head's partial, the remaining
// bits finish the sums, and a max across the scatter bits combines the
// heads.  Every lane of the group gets the result.
template <int G, int T>
__device__ __forceinline__ float group_heads_sum_max(const float (&v)[G])
{
    static_assert(G <= T && (T & (T - 1)) == 0 && T <= 32, "head groups");
    float s;
    int sbits;   // lane bits used by the scatter
    if constexpr (G == 1) {
        s = v[0];
        sbits = 0;
    } else if constexpr (G == 2) {
        float a1[1];
        halve_sum<2>(v, a1, T / 2);
        s = a1[0];
        sbits = T / 2;
    } else if constexpr (G == 4) {
        float a2[2], a1[1];
        halve_sum<4>(v, a2, T / 2);
        halve_sum<2>(a2, a1, T / 4);
        s = a1[0];
        sbits = T / 2 | T / 4;
    } else {
        static_assert(G == 8, "groups of 1, 2, 4 or 8 query heads");
        float a4[4], a2[2], a1[1];
        halve_sum<8>(v, a4, T / 2);
        halve_sum<4>(a4, a2, T / 4);
        halve_sum<2>(a2, a1, T / 8);
        s = a1[0];
        sbits = T / 2 | T / 4 | T / 8;
    }
#pragma unroll
    for (int off = 1; off < T; off <<= 1)
        if (!(sbits & off)) s += __shfl_xor_sync(0xffffffffu, s, off);
#pragma unroll
    for (int off = 1; off < T; off <<= 1)
        if (sbits & off) s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, off));
    return s;
}

// s_j = max over the group's query heads g of sum_i max(q_gi * max_ji,
// q_gi * min_ji) for every candidate block j: the Quest bound on q_g . k_t
// over the block's tokens t (Vortex blog post, end of "Why Long
// Generations Are Expensive"; the Quest listing in "Writing an algorithm:
// vFlow" takes Max over heads of Sum over dims of Maximum(q * max, q * min)).
// Since max_ji >= min_ji, max(q * max, q * min) is q * max where q >= 0 and
// q * min where q < 0, so the head's bound is the exact identity
//   sum_i max(q_gi max_ji, q_gi min_ji) = q+_g . max_j + q-_g . min_j,
// q+ = max(q, 0), q- = min(q, 0): two multiply-adds per dim and head, with
// q+ and q- (fixed over the blocks) in registers.
//
// A CTA scores a contiguous chunk of one request's blocks.  The blocks'
// summary rows ([num_pages, HKV, 2, DK] bf16, maximum then minimum; ROW
// bytes a page) are staged in shared memory by 16-byte cp.async, NB pages a
// tile, kQsStages tiles in flight.  A thread owns DPT dims of one KV head's
// rows (TPB threads a row) and scores BPP blocks per pass.
constexpr int kQsThreads = 256;
constexpr int kQsStages = 3;
constexpr int kQsTileBytes = 32 * 1024;

template <int DK, int HKV, int G>
struct QsCfg {
    static constexpr int DPT = G <= 4 ? 8 : 4;              // dims per thread
    static constexpr int TPB = DK / DPT;                     // threads per (block, KV head)
    static constexpr int BPP = kQsThreads / (TPB * HKV);     // blocks per pass
    static constexpr int ROW = HKV * 2 * DK * 2;             // summary bytes of one page
    static constexpr int NB = kQsTileBytes / ROW;            // pages per tile
    static constexpr int PASSES = NB / BPP;
    static constexpr int SMEM = kQsStages * kQsTileBytes;
    static_assert(BPP >= 1 && PASSES >= 1 && NB % BPP == 0, "tile layout");
};

template <int DK, int HKV, int G>
__global__ void __launch_bounds__(kQsThreads, 2) k_score_quest(ScoreArgs a)
{
    using C = QsCfg<DK, HKV, G>;
    constexpr int DPT = C::DPT, TPB = C::TPB, BPP = C::BPP, ROW = C::ROW, NB = C::NB;
    extern __shared__ __align__(128) uint8_t qsm[];
    __shared__ int s_page[kScoreMaxChunk];
    pdl_enter();
    const int tid = threadIdx.x;
    const int r = blockIdx.y;
    const int sl = tid % TPB, h = (tid / TPB) % HKV, bp = tid / (TPB * HKV);
    const int j0 = blockIdx.x * a.chunk;
    const int j1 = min(j0 + a.chunk, a.max_blocks);

    // ---- prologue: lengths, page ids and the query, all loaded first
    const int L = a.lens[r];
    int praw[kPtPerThread];
#pragma unroll
    for (int i = 0; i < kPtPerThread; ++i) {
        const int j = j0 + tid + i * kQsThreads;
        praw[i] = j < j1 ? a.pt[(int64_t)r * a.max_blocks + j] : -1;
    }
    float qp[G][DPT], qn[G][DPT];
    {
        const uint16_t *q0 = a.q + ((int64_t)r * a.hq + h * G) * DK + sl * DPT;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            uint32_t w[DPT / 2];
            if constexpr (DPT == 8) {
                const uint4 v = *reinterpret_cast<const uint4 *>(q0 + (int64_t)g * DK);
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            } else {
                const uint2 v = *reinterpret_cast<const uint2 *>(q0 + (int64_t)g * DK);
                w[0] = v.x; w[1] = v.y;
            }
#pragma unroll
            for (int e = 0; e < DPT / 2; ++e) {
                const float2 f = bf2_to_f2(w[e]);
                qp[g][2 * e] = fmaxf(f.x, 0.f);
                qn[g][2 * e] = fminf(f.x, 0.f);
                qp[g][2 * e + 1] = fmaxf(f.y, 0.f);
                qn[g][2 * e + 1] = fminf(f.y, 0.f);
            }
        }
    }
    const bool len_ok = L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * a.b;
    if (!len_ok && tid == 0 && blockIdx.x == 0) flag_error(a.status, LSA_ERR_BOUNDS);
    const int se = len_ok ? min(a.sink, L) : 0;
    const int rs = len_ok ? max(L - a.recent, se) : 0;
#pragma unroll
    for (int i = 0; i < kPtPerThread; ++i) {
        const int j = j0 + tid + i * kQsThreads;
        if (j >= j1) continue;
        const bool cand = len_ok && (int64_t)j * a.b >= se && (int64_t)(j + 1) * a.b <= rs;
        int p = cand ? praw[i] : -1;
        if (cand && (p < 0 || p >= a.num_pages)) {
            flag_error(a.status, LSA_ERR_BOUNDS);
            p = -1;
        }
        s_page[j - j0] = p;
        if (p < 0) {
#pragma unroll
            for (int hh = 0; hh < HKV; ++hh) a.scores[((int64_t)r * HKV + hh) * a.max_blocks + j] = -INFINITY;
        }
    }
    __syncthreads();

    // ---- the chunk's tiles through a kQsStages-deep cp.async ring
    const int n = j1 - j0;
    const int ntiles = (n + NB - 1) / NB;
    const uint8_t *summ = reinterpret_cast<const uint8_t *>(a.summ);
    const uint64_t pol = l2_evict_first();
    const uint32_t sbase = smem_addr(qsm);
    auto issue = [&](int t) {
        if (t < ntiles) {
            const uint32_t dst = sbase + (uint32_t)((t % kQsStages) * kQsTileBytes);
            constexpr int CPR = ROW / 16;   // 16-byte chunks per page row
            for (int c = tid; c < NB * CPR; c += kQsThreads) {
                const int bi = c / CPR, off = c - bi * CPR;
                const int i = t * NB + bi;
                const int p = i < n ? s_page[i] : -1;
                if (p >= 0) cp_async16_policy(dst + (uint32_t)(bi * ROW + off * 16), summ + (int64_t)p * ROW + off * 16, pol);
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int t = 0; t < kQsStages - 1; ++t) issue(t);
    for (int t = 0; t < ntiles; ++t) {
        cp_async_wait<kQsStages - 2>();
        __syncthreads();                      // tile t is in; tile t - 1's stage is free
        issue(t + kQsStages - 1);
        const uint8_t *tile = qsm + (t % kQsStages) * kQsTileBytes;
#pragma unroll
        for (int ps = 0; ps < C::PASSES; ++ps) {
            const int bi = ps * BPP + bp;
            const int i = t * NB + bi;
            const bool have = i < n && s_page[i] >= 0;
            const uint8_t *row = tile + bi * ROW + h * (2 * DK * 2) + sl * DPT * 2;
            uint32_t wM[DPT / 2], wm[DPT / 2];
            if constexpr (DPT == 8) {
                const uint4 x = *reinterpret_cast<const uint4 *>(row);
                const uint4 y = *reinterpret_cast<const uint4 *>(row + DK * 2);
                wM[0] = x.x; wM[1] = x.y; wM[2] = x.z; wM[3] = x.w;
                wm[0] = y.x; wm[1] = y.y; wm[2] = y.z; wm[3] = y.w;
            } else {
                const uint2 x = *reinterpret_cast<const uint2 *>(row);
                const uint2 y = *reinterpret_cast<const uint2 *>(row + DK * 2);
                wM[0] = x.x; wM[1] = x.y;
                wm[0] = y.x; wm[1] = y.y;
            }
            float M[DPT], m[DPT];
#pragma unroll
            for (int e = 0; e < DPT / 2; ++e) {
                const float2 fM = bf2_to_f2(wM[e]), fm = bf2_to_f2(wm[e]);
                M[2 * e] = fM.x;
                M[2 * e + 1] = fM.y;
                m[2 * e] = fm.x;
                m[2 * e + 1] = fm.y;
            }
            float part[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float acc = 0.f;
#pragma unroll
                for (int d = 0; d < DPT; ++d) {
                    acc = fmaf(qp[g][d], M[d], acc);
                    acc = fmaf(qn[g][d], m[d], acc);
                }
                part[g] = acc;
            }
            const float sc = group_heads_sum_max<G, TPB>(part);
            if (have && sl == 0) a.scores[((int64_t)r * HKV + h) * a.max_blocks + j0 + i] = sc;
        }
    }
    cp_async_wait<0>();
}

template <int DK, int HKV, int G>
cudaError_t launch_score_quest_t(const ScoreArgs &a, cudaStream_t s)
{
    auto kern = k_score_quest<DK, HKV, G>;
    cudaError_t le = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, QsCfg<DK, HKV, G>::SMEM);
    if (le != cudaSuccess) return le;
    dim3 grid((a.max_blocks + a.chunk - 1) / a.chunk, a.batch);
    le = launch_step_kernel(kern, grid, dim3(kQsThreads), QsCfg<DK, HKV, G>::SMEM, s, a);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

// ============================================================ top-k

constexpr int kTopkThreads = 1024;
constexpr int kTopkMaxCols = 32768;

// Output index of column `col` of row `row`: the column, or for the fine
// pass of coarse-to-fine the token position it stands for.
__device__ __forceinline__ int32_t topk_out(const TopkArgs &a, int row, int col)
{
    if (!a.cand) return col;
    const int cb = a.cand[(int64_t)row * a.ncand + col / a.b];
    return cb * a.b + col % a.b;
}

// One block of NT threads per row (256 for rows of up to 2048 columns, else
// 1024), KPT columns per thread: the bucketed top-k of topk_bucket.cuh.
template <int KPT, bool APPROX = false, int NT = kTopkThreads>
__global__ void __launch_bounds__(NT) k_topk_rows(TopkArgs a)
{
    pdl_enter();
    __shared__ BucketScratch<NT> sm;
    const int row = blockIdx.x, tid = threadIdx.x;
    int n = a.num_cols ? a.num_cols[row] : a.cols;
    n = max(0, min(n, a.cols));
    const float *srow = a.scores + (int64_t)row * a.cols;
    const int c0 = tid * KPT;
    float v[KPT];
    const bool vec = (a.cols & 3) == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0 && c0 + KPT <= n;
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
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
        nan |= isnan(v[e]);
        keys[e] = (isnan(v[e]) || v[e] == -INFINITY) ? 0u : float_to_key(v[e]);
    }
    if (nan) flag_error(a.status, LSA_ERR_NAN);
    int32_t *orow = a.idx + (int64_t)row * a.k;
    const int keff = block_bucket_topk<NT, KPT, APPROX>(
        keys, a.k, sm, [&](int pos, int col) { orow[pos] = topk_out(a, row, col); },
        APPROX ? splitmix64(a.seed, (uint64_t)row + 1) : 0ull);
    for (int i = keff + tid; i < a.k; i += NT) orow[i] = -1;
}

// Few long rows: a cluster of CS CTAs of kClThreads threads per row, KPT
// columns per thread (topk_cluster.cuh), so that a handful of rows still
// spread over many SMs.  CTA c of the row's cluster holds columns
// [c * kClThreads * KPT, (c + 1) * kClThreads * KPT).
constexpr int kClThreads = 512;

template <int CS, int KPT, bool APPROX = false>
__global__ void __launch_bounds__(kClThreads, 1) k_topk_cluster(TopkArgs a)
{
    pdl_enter();
    __shared__ ClusterTopkScratch<kClThreads, CS> sm;
    const int rank = (int)cluster_rank();
    const int row = blockIdx.y, tid = threadIdx.x;
    int n = a.num_cols ? a.num_cols[row] : a.cols;
    n = max(0, min(n, a.cols));
    const float *srow = a.scores + (int64_t)row * a.cols;
    const int c0 = (rank * kClThreads + tid) * KPT;
    float v[KPT];
    const bool vec = KPT >= 2 && (a.cols % KPT) == 0 && (reinterpret_cast<uintptr_t>(a.scores) % (4 * KPT)) == 0 &&
                     c0 + KPT <= n;
    if constexpr (KPT == 2) {
        if (vec) {
            const float2 f = *reinterpret_cast<const float2 *>(srow + c0);
            v[0] = f.x;
            v[1] = f.y;
        }
    } else if constexpr (KPT >= 4) {
        if (vec) {
#pragma unroll
            for (int e = 0; e < KPT; e += 4) {
                const float4 f = *reinterpret_cast<const float4 *>(srow + c0 + e);
                v[e] = f.x;
                v[e + 1] = f.y;
                v[e + 2] = f.z;
                v[e + 3] = f.w;
            }
        }
    }
    if (!vec) {
#pragma unroll
        for (int e = 0; e < KPT; ++e) v[e] = c0 + e < n ? srow[c0 + e] : -INFINITY;
    }
    uint32_t keys[KPT];
    bool nan = false;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
        nan |= isnan(v[e]);
        keys[e] = (isnan(v[e]) || v[e] == -INFINITY) ? 0u : float_to_key(v[e]);
    }
    if (nan) flag_error(a.status, LSA_ERR_NAN);
    int32_t *orow = a.idx + (int64_t)row * a.k;
    const int keff = cluster_bucket_topk<kClThreads, KPT, CS, APPROX>(
        keys, a.k, c0, sm, [&](int pos, int col) { orow[pos] = topk_out(a, row, col); },
        APPROX ? splitmix64(a.seed, (uint64_t)row + 1) : 0ull);
    if (rank == 0)
        for (int i = keff + tid; i < a.k; i += kClThreads) orow[i] = -1;
}

// Cluster size the cluster top-k runs with on this device: 16 CTAs where a
// cluster of 16 can be resident, else 8 (0: neither).
int topk_cluster_size()
{
    static std::mutex mu;
    static int cs[64] = {};
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!done[dev]) {
        int c = 0;
        if (max_active_clusters(k_topk_cluster<16, 1>, 16, dim3(kClThreads), 0) > 0 &&
            max_active_clusters(k_topk_cluster<16, 2>, 16, dim3(kClThreads), 0) > 0 &&
            max_active_clusters(k_topk_cluster<16, 4>, 16, dim3(kClThreads), 0) > 0)
            c = 16;
        else if (max_active_clusters(k_topk_cluster<8, 8>, 8, dim3(kClThreads), 0) > 0)
            c = 8;
        cs[dev] = c;
        done[dev] = true;
    }
    return cs[dev];
}

template <int CS, int KPT>
cudaError_t launch_topk_cluster_t(const TopkArgs &a, cudaStream_t s)
{
    if (a.approx && CS > 8) {
        cudaError_t e = cudaFuncSetAttribute(k_topk_cluster<CS, KPT, true>,
                                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    return a.approx ? launch_cluster_kernel(pdl_enabled(), CS, k_topk_cluster<CS, KPT, true>, dim3(CS, a.rows),
                                            dim3(kClThreads), 0, s, a)
                    : launch_cluster_kernel(pdl_enabled(), CS, k_topk_cluster<CS, KPT>, dim3(CS, a.rows),
                                            dim3(kClThreads), 0, s, a);
}

// The cluster top-k when the rows are few and long enough for it to pay
// (LSA_TOPK_PATH=rows / cluster forces one or the other); false: not taken.
bool launch_topk_cluster(const TopkArgs &a, cudaStream_t s, cudaError_t *err)
{
    const char *env = getenv("LSA_TOPK_PATH");
    const int mode = !env ? 0 : strcmp(env, "rows") == 0 ? 1 : strcmp(env, "cluster") == 0 ? 2 : 0;
    if (mode == 1) return false;
    const int cs = topk_cluster_size();
    if (cs == 0) return false;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (mode == 0 && !(a.cols > 4096 && (int64_t)a.rows * cs <= sms)) return false;
    const int per = cs * kClThreads;
    const int kpt = a.cols <= per ? 1 : a.cols <= 2 * per ? 2 : a.cols <= 4 * per ? 4 : 8;
    cudaError_t e;
    if (cs == 16) {
        if (kpt > 4) return false;
        e = kpt == 1 ? launch_topk_cluster_t<16, 1>(a, s)
          : kpt == 2 ? launch_topk_cluster_t<16, 2>(a, s)
                     : launch_topk_cluster_t<16, 4>(a, s);
    } else {
        e = kpt == 1 ? launch_topk_cluster_t<8, 1>(a, s)
          : kpt == 2 ? launch_topk_cluster_t<8, 2>(a, s)
          : kpt == 4 ? launch_topk_cluster_t<8, 4>(a, s)
                     : launch_topk_cluster_t<8, 8>(a, s);
    }
    *err = e != cudaSuccess ? e : cudaGetLastError();
    return true;
}

// ============================================================ fine pass

constexpr int kFineWarps = 8;
constexpr int kFineBlocksPerCta = 4;

// f_t = scale_t * q_sum . e4m3(k8_t) for every token of the candidate
// blocks (LeanSparse, Section 5: exact rescoring of the retained candidates
// with their original FP8 indexer keys).  8 lanes per token, 16 dims each.
__global__ void __launch_bounds__(kFineWarps * 32) k_fine_scores(FineArgs a)
{
    pdl_enter();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.y;                 // r * hkv + h
    const int hkv = a.ic.hkv;
    const int r = row / hkv, h = row % hkv;
    const int G = a.hq / hkv;
    const int b = a.ic.b;
    const int sub = lane & 7, tq = lane >> 3;   // 16 dims per lane, 4 tokens per warp

    // the group's query sum over all 256 threads: thread (slice sl, 8-dim
    // chunk c) adds heads sl, sl + 16, ... of its chunk, all loads issued at
    // once; the 16 slices are then added in slice order
    __shared__ float s_part[16][128];
    __shared__ float s_qsum[128];
    {
        const int c = threadIdx.x & 15, sl = threadIdx.x >> 4;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint16_t *qb = a.q + ((int64_t)r * a.hq + h * G) * 128 + c * 8;
        for (int g0 = sl; g0 < G; g0 += 4 * 16) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int g = g0 + 16 * u;
                v[u] = g < G ? *reinterpret_cast<const uint4 *>(qb + (int64_t)g * 128) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = bf2_to_f2(w[e]);
                    acc[2 * e] += f.x;
                    acc[2 * e + 1] += f.y;
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) s_part[sl][c * 8 + e] = acc[e];
        __syncthreads();
        if (threadIdx.x < 128) {
            float t = 0.f;
            for (int k = 0; k < 16; ++k) t += s_part[k][threadIdx.x];
            s_qsum[threadIdx.x] = t;
        }
        __syncthreads();
    }
    float qs[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) qs[e] = s_qsum[sub * 16 + e];

    const int L = a.lens[r];
    const int nfull = (L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * b) ? L / b : 0;
    const int64_t ntok_row = (int64_t)a.ncand * b;
    float *frow = a.fscores + (int64_t)row * ntok_row;
    const int c0 = blockIdx.x * kFineBlocksPerCta;
    const int nb = min(kFineBlocksPerCta, a.ncand - c0);
    // the CTA's candidate blocks -> page ids (two dependent round trips,
    // once for all of them); -1 for padding and invalid entries
    __shared__ int s_pg[kFineBlocksPerCta];
    if (threadIdx.x < nb) {
        const int j = a.cand[(int64_t)row * a.ncand + c0 + threadIdx.x];
        int p = -1;
        if (j >= 0 && j < nfull) p = a.pt[(int64_t)r * a.max_blocks + j];
        const bool ok = p >= 0 && p < a.ic.num_pages;
        if (!ok && j != -1) flag_error(a.status, LSA_ERR_BOUNDS);
        s_pg[threadIdx.x] = ok ? p : -1;
    }
    __syncthreads();
    // every (block, token) of the CTA: 8 lanes per token, 16 dims each; a
    // warp takes 4 tokens per step and all its steps' loads go out at once
    constexpr int kSteps = kFineBlocksPerCta * 64 / (kFineWarps * 4);
    static_assert(kSteps <= 16, "loads in flight per lane");
    const int ntok = nb * b;
    uint4 kv[kSteps];
    float sc[kSteps];
#pragma unroll
    for (int it = 0; it < kSteps; ++it) {
        const int t = (it * kFineWarps + warp) * 4 + tq;   // token of the CTA, block-major
        const int bi = t / b, slot = t - bi * b;
        const int p = t < ntok ? s_pg[bi] : -1;
        kv[it] = make_uint4(0, 0, 0, 0);
        sc[it] = 0.f;
        if (p >= 0) {
            kv[it] = ldg_nc_v4(a.ic.k + (int64_t)p * a.ic.kps + (int64_t)h * a.ic.khs + (int64_t)slot * a.ic.kts +
                               sub * 16);
            sc[it] = a.ic.kscale[(int64_t)p * a.ic.sps + (int64_t)h * a.ic.shs + slot];
        }
    }
#pragma unroll
    for (int it = 0; it < kSteps; ++it) {
        const int t = (it * kFineWarps + warp) * 4 + tq;
        const int bi = t / b;
        const bool have = t < ntok && s_pg[bi] >= 0;
        float acc = 0.f;
        const uint32_t w[4] = {kv[it].x, kv[it].y, kv[it].z, kv[it].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float2 lo = e4m3x2_to_f2((uint16_t)(w[e] & 0xffffu));
            float2 hi = e4m3x2_to_f2((uint16_t)(w[e] >> 16));
            acc = fmaf(qs[4 * e + 0], lo.x, acc);
            acc = fmaf(qs[4 * e + 1], lo.y, acc);
            acc = fmaf(qs[4 * e + 2], hi.x, acc);
            acc = fmaf(qs[4 * e + 3], hi.y, acc);
        }
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (t < ntok && sub == 0) frow[(int64_t)c0 * b + t] = have ? sc[it] * acc : -INFINITY;
    }

}

// The weighted-ReLU indexer score of the fine pass: f_t = sum_g w[r, g] *
// ReLU(q_g . k_t), k_t = scale_t * e4m3(k8_t) (LeanSparse, Section 5: Eq. 6's
// weighted head aggregation, applied to the exact keys).  The ReLU acts per
// head, so the queries cannot be summed first: for the CTA's tokens the dots
// of all 64 heads are a dense [64 x 128] x [128 x tokens] product, run as
// m16n8k16 MMAs (bf16 queries; the e4m3 keys widened to bf16, exactly, in
// shared memory).  Warp w takes the 16 heads of M-tile w % 4 over half of
// the tokens; per token the weighted ReLUs of its heads are summed across
// lanes and then across the four M-tiles in shared memory, and scaled by
// scale_t (>= 0, so scale_t ReLU(x) = ReLU(scale_t x)).
constexpr int kWrTok = kFineBlocksPerCta * 64;        // tokens per CTA at most
constexpr int kWrSmem = kWrTok * 128 * 2;              // the widened key tile

__global__ void __launch_bounds__(kFineWarps * 32) k_fine_scores_wrelu(FineArgs a)
{
    pdl_enter();
    extern __shared__ __align__(1024) uint8_t wsm[];   // [kWrTok / 16] tiles of 16 tokens x 128 dims, swizzled
    __shared__ float s_part[4][kWrTok];
    __shared__ int s_pg[kFineBlocksPerCta];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.y;
    const int hkv = a.ic.hkv;
    const int r = row / hkv, h = row % hkv;
    const int G = a.hq / hkv;   // 64 (host-checked)
    const int b = a.ic.b;
    const int mt = warp & 3, th = warp >> 2;
    const int rr = lane >> 2, cc = lane & 3;

    // this warp's A fragments: heads 16 mt .. 16 mt + 15, all 128 dims
    uint32_t qa[8][4];
    {
        const uint16_t *q0 = a.q + ((int64_t)r * a.hq + h * G + 16 * mt + rr) * 128;
        const uint16_t *q8 = q0 + 8 * 128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qa[ks][0] = *reinterpret_cast<const uint32_t *>(q0 + 16 * ks + 2 * cc);
            qa[ks][1] = *reinterpret_cast<const uint32_t *>(q8 + 16 * ks + 2 * cc);
            qa[ks][2] = *reinterpret_cast<const uint32_t *>(q0 + 16 * ks + 8 + 2 * cc);
            qa[ks][3] = *reinterpret_cast<const uint32_t *>(q8 + 16 * ks + 8 + 2 * cc);
        }
    }
    const float w_lo = a.weights[(int64_t)r * a.hq + h * G + 16 * mt + rr];
    const float w_hi = a.weights[(int64_t)r * a.hq + h * G + 16 * mt + rr + 8];

    const int L = a.lens[r];
    const int nfull = (L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * b) ? L / b : 0;
    const int64_t ntok_row = (int64_t)a.ncand * b;
    float *frow = a.fscores + (int64_t)row * ntok_row;
    const int c0 = blockIdx.x * kFineBlocksPerCta;
    const int nb = min(kFineBlocksPerCta, a.ncand - c0);
    if (threadIdx.x < nb) {
        const int j = a.cand[(int64_t)row * a.ncand + c0 + threadIdx.x];
        int p = -1;
        if (j >= 0 && j < nfull) p = a.pt[(int64_t)r * a.max_blocks + j];
        const bool ok = p >= 0 && p < a.ic.num_pages;
        if (!ok && j != -1) flag_error(a.status, LSA_ERR_BOUNDS);
        s_pg[threadIdx.x] = ok ? p : -1;
    }
    __syncthreads();
    const int ntok = nb * b;

    // ---- the keys, widened: task (token t, 16-dim chunk u) -> two swizzled
    // 16-byte chunks of bf16; tokens with nothing to score become zeros
    {
        constexpr int kTasks = kWrTok * 8;
        for (int task = threadIdx.x; task < kTasks; task += kFineWarps * 32) {
            const int t = task >> 3, u = task & 7;
            const int bi = t / b, slot = t - bi * b;
            const int p = t < ntok ? s_pg[bi] : -1;
            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
            if (p >= 0) {
                const uint4 v = ldg_nc_v4(a.ic.k + (int64_t)p * a.ic.kps + (int64_t)h * a.ic.khs +
                                          (int64_t)slot * a.ic.kts + u * 16);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f0 = e4m3x2_to_f2((uint16_t)(w[e] & 0xffffu));
                    const float2 f1 = e4m3x2_to_f2((uint16_t)(w[e] >> 16));
                    o[2 * e] = pack_bf16x2(f0.x, f0.y);       // exact: e4m3 values are bf16 values
                    o[2 * e + 1] = pack_bf16x2(f1.x, f1.y);
                }
                lo = make_uint4(o[0], o[1], o[2], o[3]);
                hi = make_uint4(o[4], o[5], o[6], o[7]);
            }
            uint8_t *tile = wsm + (t >> 4) * (16 * 256);
            *reinterpret_cast<uint4 *>(tile + swizzle_offset(t & 15, 2 * u)) = lo;
            *reinterpret_cast<uint4 *>(tile + swizzle_offset(t & 15, 2 * u + 1)) = hi;
        }
    }
    __syncthreads();

    // ---- dots of the warp's 16 heads with its half of the tokens
    const int mi = lane >> 3, r8 = lane & 7;
    const int tk = (mi >> 1) * 8 + r8, ck = mi & 1;
    const uint32_t wbase = smem_addr(wsm);
    for (int gi = 8 * th; gi < min(8 * th + 8, (ntok + 15) / 16); ++gi) {
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t tb = wbase + gi * (16 * 256);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t bb[4];
            ldsm_x4(bb, tb + swizzle_offset(tk, 2 * ks + ck));
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+f"(s0[0]), "+f"(s0[1]), "+f"(s0[2]), "+f"(s0[3])
                : "r"(qa[ks][0]), "r"(qa[ks][1]), "r"(qa[ks][2]), "r"(qa[ks][3]), "r"(bb[0]), "r"(bb[1]));
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                "{%0,%1,%2,%3};"
                : "+f"(s1[0]), "+f"(s1[1]), "+f"(s1[2]), "+f"(s1[3])
                : "r"(qa[ks][0]), "r"(qa[ks][1]), "r"(qa[ks][2]), "r"(qa[ks][3]), "r"(bb[2]), "r"(bb[3]));
        }
        // lane holds heads rr (s[0], s[1]) and rr + 8 (s[2], s[3]) of tokens
        // 2 cc, 2 cc + 1 of each 8-token n-tile: weight, ReLU, then the sum
        // over the 8 lanes sharing cc
        float t0 = w_lo * fmaxf(s0[0], 0.f) + w_hi * fmaxf(s0[2], 0.f);
        float t1 = w_lo * fmaxf(s0[1], 0.f) + w_hi * fmaxf(s0[3], 0.f);
        float t2 = w_lo * fmaxf(s1[0], 0.f) + w_hi * fmaxf(s1[2], 0.f);
        float t3 = w_lo * fmaxf(s1[1], 0.f) + w_hi * fmaxf(s1[3], 0.f);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            t0 += __shfl_xor_sync(0xffffffffu, t0, off);
            t1 += __shfl_xor_sync(0xffffffffu, t1, off);
            t2 += __shfl_xor_sync(0xffffffffu, t2, off);
            t3 += __shfl_xor_sync(0xffffffffu, t3, off);
        }
        if (rr == 0) {
            s_part[mt][gi * 16 + 2 * cc] = t0;
            s_part[mt][gi * 16 + 2 * cc + 1] = t1;
            s_part[mt][gi * 16 + 8 + 2 * cc] = t2;
            s_part[mt][gi * 16 + 8 + 2 * cc + 1] = t3;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < ntok; t += kFineWarps * 32) {
        const int bi = t / b, slot = t - bi * b;
        const int p = s_pg[bi];
        float f = -INFINITY;
        if (p >= 0) {
            const float sc = a.ic.kscale[(int64_t)p * a.ic.sps + (int64_t)h * a.ic.shs + slot];
            f = sc * ((s_part[0][t] + s_part[1][t]) + (s_part[2][t] + s_part[3][t]));
        }
        frow[(int64_t)c0 * b + t] = f;
    }
}

template <int DK, int HKV>
cudaError_t launch_score_t(const ScoreArgs &a, cudaStream_t s)
{
    dim3 grid((a.max_blocks + a.chunk - 1) / a.chunk, a.batch);
    cudaError_t le = launch_step_kernel(k_score<DK, HKV>, grid, dim3(kScoreWarps * 32), 0, s, a);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

}  // namespace

bool score_supported(int dk, int hkv)
{
    switch (dk) {
    case 64: case 128: case 256: return hkv == 1 || hkv == 2 || hkv == 4 || hkv == 8;
    case 576: return hkv == 1;
    default: return false;
    }
}

cudaError_t launch_score(const ScoreArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = false;
    if (a.batch == 0 || a.max_blocks == 0) return cudaSuccess;
#define LSA_SCORE_CASE(D, H) \
    if (a.dk == D && a.hkv == H) return launch_score_t<D, H>(a, s);
    LSA_SCORE_CASE(64, 1) LSA_SCORE_CASE(64, 2) LSA_SCORE_CASE(64, 4) LSA_SCORE_CASE(64, 8)
    LSA_SCORE_CASE(128, 1) LSA_SCORE_CASE(128, 2) LSA_SCORE_CASE(128, 4) LSA_SCORE_CASE(128, 8)
    LSA_SCORE_CASE(256, 1) LSA_SCORE_CASE(256, 2) LSA_SCORE_CASE(256, 4) LSA_SCORE_CASE(256, 8)
    LSA_SCORE_CASE(576, 1)
#undef LSA_SCORE_CASE
    *unsupported = true;
    return cudaSuccess;
}

bool score_quest_supported(int dk, int hkv, int group)
{
    return (dk == 64 || dk == 128) && (hkv == 1 || hkv == 2 || hkv == 4 || hkv == 8) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t launch_score_quest(const ScoreArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = false;
    if (a.batch == 0 || a.max_blocks == 0) return cudaSuccess;
    const int G = a.hq / a.hkv;
#define LSA_QUEST_G(D, H)                                                    \
    if (a.dk == D && a.hkv == H) {                                           \
        if (G == 1) return launch_score_quest_t<D, H, 1>(a, s);               \
        if (G == 2) return launch_score_quest_t<D, H, 2>(a, s);               \
        if (G == 4) return launch_score_quest_t<D, H, 4>(a, s);               \
        if (G == 8) return launch_score_quest_t<D, H, 8>(a, s);               \
    }
    LSA_QUEST_G(64, 1) LSA_QUEST_G(64, 2) LSA_QUEST_G(64, 4) LSA_QUEST_G(64, 8)
    LSA_QUEST_G(128, 1) LSA_QUEST_G(128, 2) LSA_QUEST_G(128, 4) LSA_QUEST_G(128, 8)
#undef LSA_QUEST_G
    *unsupported = true;
    return cudaSuccess;
}

int topk_max_cols() { return kTopkMaxCols; }

int score_chunk(int batch, int max_blocks, int sms)
{
    // one wave of two CTAs per SM with equal chunks (a multiple of 4 blocks)
    const int64_t target = 2LL * sms;
    int64_t per = ((int64_t)batch * max_blocks + target - 1) / target;
    per = ((per + 3) / 4) * 4;
    if (per < 4) per = 4;
    if (per > kScoreMaxChunk) per = kScoreMaxChunk;
    return (int)per;
}

cudaError_t launch_topk(const TopkArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = a.cols > kTopkMaxCols;
    if (*unsupported || a.rows == 0 || a.k == 0) return cudaSuccess;
    cudaError_t fe = cudaSuccess;
    // rows of up to 8192 columns with k <= 64: the block top-k (a bound from
    // the threads' maxima, then an exact rank of the few keys above it);
    // wider rows and larger k: the radix select
    if (!a.approx && a.k <= 64 && launch_topk_fast(a, s, &fe)) return fe;
    if (launch_topk_cluster(a, s, &fe)) return fe;
    cudaError_t e;
    const dim3 g(a.rows), blk(kTopkThreads);
    if (a.approx) {
        if (a.cols <= 256 * 8) e = launch_step_kernel(k_topk_rows<8, true, 256>, g, dim3(256), 0, s, a);
        else if (a.cols <= kTopkThreads * 8) e = launch_step_kernel(k_topk_rows<8, true>, g, blk, 0, s, a);
        else if (a.cols <= kTopkThreads * 16) e = launch_step_kernel(k_topk_rows<16, true>, g, blk, 0, s, a);
        else e = launch_step_kernel(k_topk_rows<32, true>, g, blk, 0, s, a);
    } else {
        if (a.cols <= 256 * 8) e = launch_step_kernel(k_topk_rows<8, false, 256>, g, dim3(256), 0, s, a);
        else if (a.cols <= kTopkThreads * 8) e = launch_step_kernel(k_topk_rows<8>, g, blk, 0, s, a);
        else if (a.cols <= kTopkThreads * 16) e = launch_step_kernel(k_topk_rows<16>, g, blk, 0, s, a);
        else e = launch_step_kernel(k_topk_rows<32>, g, blk, 0, s, a);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_fine_scores(const FineArgs &a, cudaStream_t s, bool *unsupported)
{
    // a CTA scores kFineBlocksPerCta blocks of at most 64 tokens each
    *unsupported = a.ic.dk != 128 || !a.ic.e4m3 || a.ic.b > 64 || a.ic.b % 16 != 0 ||
                   (a.weights && a.hq / a.ic.hkv != 64);
    if (*unsupported || a.batch == 0 || a.ncand == 0) return cudaSuccess;
    dim3 grid((a.ncand + kFineBlocksPerCta - 1) / kFineBlocksPerCta, a.batch * a.ic.hkv);
    cudaError_t le;
    if (a.weights) {
        le = cudaFuncSetAttribute(k_fine_scores_wrelu, cudaFuncAttributeMaxDynamicSharedMemorySize, kWrSmem);
        if (le != cudaSuccess) return le;
        le = launch_step_kernel(k_fine_scores_wrelu, grid, dim3(kFineWarps * 32), kWrSmem, s, a);
    } else {
        le = launch_step_kernel(k_fine_scores, grid, dim3(kFineWarps * 32), 0, s, a);
    }
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

}  // namespace lsa

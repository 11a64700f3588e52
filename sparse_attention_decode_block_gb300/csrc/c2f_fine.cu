// The fine half of the coarse-to-fine decode step in one kernel: per
// request, one thread-block cluster of CS CTAs
//   1. selects the top C candidate blocks of the request's coarse scores
//      (the index-key summary scores of the kernel before it),
//   2. rescores every token of its share of those blocks exactly against the
//      FP8 e4m3 index keys (head-sum score, or the weighted-ReLU indexer
//      score), and
//   3. selects the request's top tokens over all of the cluster's scores
// (LeanSparse, Section 5 "Coarse-to-fine decode indexing": a coarse pass
// keeps candidates, an exact pass over their original FP8 keys keeps the
// final tokens).  Both selections are the exact cluster top-k of
// topk_cluster.cuh; the candidates travel to the CTAs that rescore them,
// and the fine scores stay, through distributed shared memory.  Nothing
// waits on a flag, and nothing but the two selections goes to memory.
#include <math.h>

#include <mutex>

#include "lsa_device.cuh"
#include "fine_tile.cuh"
#include "topk_cluster.cuh"

namespace lsa {
namespace {

constexpr int kCfThreads = kFtThreads;
constexpr int kCfWarps = kFtWarps;
constexpr int kCfTok = kFtTok;               // tokens one CTA rescores at most
constexpr int kCfMaxCand = 64;               // candidate blocks one CTA takes at most
constexpr int kCfKpt = kCfTok / kCfThreads;  // fine-score columns per thread

// Dynamic shared memory of a CTA.
struct CfLayout {
    static constexpr int KEYS = 0;                        // [kCfTok][128] e4m3, 16-byte chunks swizzled
    static constexpr int PART = KEYS + kCfTok * 128;      // [4][kCfTok] fp32: query-sum partials, then head-tile partials
    static constexpr int FS = PART + 4 * kCfTok * 4;      // [kCfTok] fp32 fine scores
    static constexpr int SC = FS + kCfTok * 4;            // [kCfTok] fp32 token scales
    static constexpr int QS = SC + kCfTok * 4;            // [128] fp32 query sum
    static constexpr int CAND = QS + 128 * 4;             // [kCfMaxCand] int32 candidate blocks
    static constexpr int PG = CAND + kCfMaxCand * 4;      // [kCfMaxCand] int32 their pages
    static constexpr int SMEM = PG + kCfMaxCand * 4;
};
static_assert(CfLayout::SMEM + sizeof(ClusterTopkScratch<kCfThreads, 8>) <= 227 * 1024, "shared memory");

template <int CS, int KPT1, bool WRELU>
__global__ void __launch_bounds__(kCfThreads, 1) k_c2f_fine(FineArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ ClusterTopkScratch<kCfThreads, CS> tsm;
    using LY = CfLayout;
    const int rank = (int)cluster_rank();
    const int r = blockIdx.y;   // the request (one KV head)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.hq;
    const int b = a.ic.b;
    const int CB = (a.ncand + CS - 1) / CS;   // candidate positions per CTA
    const int nb = min(CB, max(0, a.ncand - rank * CB));
    float *s_part = reinterpret_cast<float *>(smem + LY::PART);
    float *s_fs = reinterpret_cast<float *>(smem + LY::FS);
    float *s_sc = reinterpret_cast<float *>(smem + LY::SC);
    float *s_qs = reinterpret_cast<float *>(smem + LY::QS);
    int *s_cand = reinterpret_cast<int *>(smem + LY::CAND);
    int *s_pg = reinterpret_cast<int *>(smem + LY::PG);

    // ---- prologue, before the coarse scores are final: the query side
    WreluQ Q;               // WRELU: this warp's A fragments and weights (fine_tile.cuh)
    float qs[16];           // head sum: this lane's 16 dims of the query sum
    if constexpr (WRELU) {
        // a query element outside f16's exact range is flagged
        // (LSA_ERR_BOUNDS) and the request scores nothing
        const bool big = wrelu_load_q(a.q + (int64_t)r * a.hq * 128, a.weights + (int64_t)r * a.hq, Q);
        if (big) flag_error(a.status, LSA_ERR_BOUNDS);
        if (__syncthreads_or(big ? 1 : 0)) wrelu_zero(Q);   // the selections still run (on empty rows)
    } else {
        // the group's query sum: thread (slice sl, 8-dim chunk c) adds heads
        // sl, sl + 32, ... of its chunk; the slices are then added in order
        const int c = tid & 15, sl = tid >> 4;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint16_t *qb = a.q + (int64_t)r * a.hq * 128 + c * 8;
        for (int g0 = sl; g0 < G; g0 += 4 * 32) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int g = g0 + 32 * u;
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
        for (int e = 0; e < 8; ++e) s_part[sl * 128 + c * 8 + e] = acc[e];
        __syncthreads();
        if (tid < 128) {
            float t = 0.f;
            for (int k = 0; k < 32; ++k) t += s_part[k * 128 + tid];
            s_qs[tid] = t;
        }
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 16; ++e) qs[e] = s_qs[(lane & 7) * 16 + e];
    }
    for (int i = tid; i < kCfMaxCand; i += kCfThreads) s_cand[i] = -1;

    // ---- 1. the coarse selection (the scores of the kernel before)
    pdl_wait();
    pdl_launch_dependents();
    {
        const float *crow = a.coarse + (int64_t)r * a.max_blocks;
        const int c0 = (rank * kCfThreads + tid) * KPT1;
        uint32_t keys[KPT1];
        bool nan = false;
#pragma unroll
        for (int e = 0; e < KPT1; ++e) {
            const float x = c0 + e < a.max_blocks ? __ldcg(crow + c0 + e) : -INFINITY;
            nan |= isnan(x);
            keys[e] = (isnan(x) || x == -INFINITY) ? 0u : float_to_key(x);
        }
        if (nan) flag_error(a.status, LSA_ERR_NAN);
        int32_t *cout = a.cand_out ? a.cand_out + (int64_t)r * a.ncand : nullptr;
        const int keff = cluster_bucket_topk<kCfThreads, KPT1, CS>(keys, a.ncand, c0, tsm, [&](int pos, int col) {
            const int owner = pos / CB;
            st_cluster_u32(cluster_map(smem_addr(&s_cand[pos - owner * CB]), (uint32_t)owner), (uint32_t)col);
            if (cout) cout[pos] = col;
        });
        if (cout && rank == 0)
            for (int i = keff + tid; i < a.ncand; i += kCfThreads) cout[i] = -1;
    }

    // ---- 2. exact rescoring of this CTA's candidate blocks
    const int L = a.lens[r];
    const int nfull = (L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * b) ? L / b : 0;
    if (tid < nb) {
        const int j = s_cand[tid];
        int p = -1;
        if (j >= 0 && j < nfull) p = a.pt[(int64_t)r * a.max_blocks + j];
        const bool ok = p >= 0 && p < a.ic.num_pages;
        if (!ok && j != -1) flag_error(a.status, LSA_ERR_BOUNDS);
        s_pg[tid] = ok ? p : -1;
    }
    __syncthreads();
    const int ntok = nb * b;
    {
        // every key row of the CTA's tokens by 16-byte cp.async, all in
        // flight at once; rows with nothing to score are zeros
        const uint32_t kbase = smem_addr(smem + LY::KEYS);
        for (int task = tid; task < ntok * 8; task += kCfThreads) {
            const int t = task >> 3, u = task & 7;
            const int bi = t / b, slot = t - bi * b;
            const int p = s_pg[bi];
            if (p >= 0)
                cp_async16(kbase + cf_key_off(t, u),
                           a.ic.k + (int64_t)p * a.ic.kps + (int64_t)slot * a.ic.kts + u * 16);
            else
                *reinterpret_cast<uint4 *>(smem + LY::KEYS + cf_key_off(t, u)) = make_uint4(0u, 0u, 0u, 0u);
        }
        cp_async_commit();
        for (int t = tid; t < ntok; t += kCfThreads) {
            const int bi = t / b, slot = t - bi * b;
            const int p = s_pg[bi];
            s_sc[t] = p >= 0 ? a.ic.kscale[(int64_t)p * a.ic.sps + slot] : 0.f;
        }
        cp_async_wait<0>();
        __syncthreads();
    }
    if constexpr (WRELU) {
        wrelu_tile_partials(smem_addr(smem + LY::KEYS), ntok, Q, s_part);
        __syncthreads();
        for (int t = tid; t < ntok; t += kCfThreads)
            s_fs[t] = s_pg[t / b] >= 0 ? s_sc[t] * wrelu_combine(s_part, t) : -INFINITY;
    } else {
        // 8 lanes per token, 16 dims each
        const int sub = lane & 7, tq = lane >> 3;
        for (int t0 = warp * 4; t0 < ntok; t0 += kCfWarps * 4) {
            const int t = min(t0 + tq, ntok - 1);
            const float acc = headsum_dot(smem + LY::KEYS, t, qs);
            if (t0 + tq < ntok && sub == 0) s_fs[t] = s_pg[t / b] >= 0 ? s_sc[t] * acc : -INFINITY;
        }
    }
    __syncthreads();

    // ---- 3. the request's top tokens over the cluster's fine scores
    {
        uint32_t keys[kCfKpt];
        bool nan = false;
#pragma unroll
        for (int e = 0; e < kCfKpt; ++e) {
            const int t = tid * kCfKpt + e;
            const float x = t < ntok ? s_fs[t] : -INFINITY;
            nan |= isnan(x);
            keys[e] = (isnan(x) || x == -INFINITY) ? 0u : float_to_key(x);
        }
        if (nan) flag_error(a.status, LSA_ERR_NAN);
        const int cbase = rank * CB * b;
        int32_t *orow = a.tok_idx + (int64_t)r * a.tok_k;
        const int keff = cluster_bucket_topk<kCfThreads, kCfKpt, CS>(
            keys, a.tok_k, cbase + tid * kCfKpt, tsm, [&](int pos, int col) {
                const int lt = col - cbase;
                const int bi = lt / b;
                orow[pos] = s_cand[bi] * b + (lt - bi * b);
            });
        if (rank == 0)
            for (int i = keff + tid; i < a.tok_k; i += kCfThreads) orow[i] = -1;
    }
}

template <int CS, int KPT1, bool WRELU>
cudaError_t launch_c2f_t(const FineArgs &a, cudaStream_t s)
{
    auto kern = k_c2f_fine<CS, KPT1, WRELU>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CfLayout::SMEM);
    if (e != cudaSuccess) return e;
    if (CS > 8 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
        return e;
    e = launch_cluster_kernel(pdl_step_dependent(), CS, kern, dim3(CS, a.batch), dim3(kCfThreads),
                              (size_t)CfLayout::SMEM, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int CS, bool WRELU>
cudaError_t launch_c2f_kpt(const FineArgs &a, int kpt, cudaStream_t s)
{
    if (kpt == 1) return launch_c2f_t<CS, 1, WRELU>(a, s);
    if (kpt == 2) return launch_c2f_t<CS, 2, WRELU>(a, s);
    return launch_c2f_t<CS, 4, WRELU>(a, s);
}

// 16 CTAs per cluster where such a cluster of this kernel can be resident
// on the device, else 8 (0: neither).
int c2f_cluster_size()
{
    static std::mutex mu;
    static int cs[64] = {};
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!done[dev]) {
        int c = 0;
        const dim3 blk(kCfThreads);
        if (max_active_clusters(k_c2f_fine<16, 4, true>, 16, blk, CfLayout::SMEM) > 0 &&
            max_active_clusters(k_c2f_fine<16, 4, false>, 16, blk, CfLayout::SMEM) > 0)
            c = 16;
        else if (max_active_clusters(k_c2f_fine<8, 4, true>, 8, blk, CfLayout::SMEM) > 0 &&
                 max_active_clusters(k_c2f_fine<8, 4, false>, 8, blk, CfLayout::SMEM) > 0)
            c = 8;
        cs[dev] = c;
        done[dev] = true;
    }
    return cs[dev];
}

}  // namespace

bool c2f_fine_supported(const CacheView &iv, int hq, int max_blocks, int ncand, int tok_k, bool weighted)
{
    if (!(iv.e4m3 && iv.dk == 128 && iv.hkv == 1 && iv.b >= 16 && iv.b <= 64 && iv.b % 16 == 0)) return false;
    if (tok_k <= 0 || ncand <= 0 || (weighted && hq != 64)) return false;
    if ((iv.kts & 15) || (iv.kps & 15) || (reinterpret_cast<uintptr_t>(iv.k) & 15)) return false;
    const int cs = c2f_cluster_size();
    if (cs == 0) return false;
    const int cb = (ncand + cs - 1) / cs;
    return cb <= kCfMaxCand && cb * iv.b <= kCfTok && (int64_t)max_blocks <= (int64_t)cs * kCfThreads * 4;
}

cudaError_t launch_c2f_fine(const FineArgs &a, cudaStream_t s, bool *unsupported)
{
    const bool w = a.weights != nullptr;
    *unsupported = !c2f_fine_supported(a.ic, a.hq, a.max_blocks, a.ncand, a.tok_k, w);
    if (*unsupported || a.batch == 0) return cudaSuccess;
    const int cs = c2f_cluster_size();
    const int per = cs * kCfThreads;
    const int kpt = a.max_blocks <= per ? 1 : a.max_blocks <= 2 * per ? 2 : 4;
    if (cs == 16) return w ? launch_c2f_kpt<16, true>(a, kpt, s) : launch_c2f_kpt<16, false>(a, kpt, s);
    return w ? launch_c2f_kpt<8, true>(a, kpt, s) : launch_c2f_kpt<8, false>(a, kpt, s);
}

}  // namespace lsa

// Block scoring, exact radix top-k, and the FP8 fine rescoring of the
// coarse-to-fine variant.
//
// Scores: s_j = q . k_bar_j (Vortex blog post, block top-k equation),
// summed over the query heads of one KV head's group.  Because the score is
// linear in q, the group's queries are summed once (q_sum = sum_g q_g, fp32)
// and each summary row is read once with 16-byte loads and dotted with q_sum.
//
// Top-k: exact radix select on order-preserving 32-bit keys, 8 bits per
// pass, one CTA per row with the keys in shared memory (Vortex, "Making it
// fast": radix-based top-k buckets values by their digits).  Ties go to the
// lower index and the output is ascending, so the result is bit-exact.
#include <math.h>

#include "lsa_device.cuh"

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
    float qacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const bool qthread = tid < NCH;        // one 8-dim slice of one head per thread
    const int qh = tid / CPH, qd = (tid % CPH) * 8;
    if (qthread) {
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
    }
    for (int c = tid; c < NCH; c += kScoreWarps * 32) {   // NCH > threads only for wide rows
        if (c != tid) {
            const int h = c / CPH, d0 = (c % CPH) * 8;
            float t8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int g = 0; g < G; ++g) {
                const uint4 v = *reinterpret_cast<const uint4 *>(a.q + ((int64_t)r * a.hq + h * G + g) * DK + d0);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = bf2_to_f2(w[e]);
                    t8[2 * e] += f.x;
                    t8[2 * e + 1] += f.y;
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) s_qs[h * DK + d0 + e] = t8[e];
        }
    }
    if (qthread) {
#pragma unroll
        for (int e = 0; e < 8; ++e) s_qs[qh * DK + qd + e] = qacc[e];
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
    __syncthreads();

    // ---- this lane's slice of the query sum
    float qs[NI][8];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int ch = lane + 32 * i;
#pragma unroll
        for (int e = 0; e < 8; ++e) qs[i][e] = ch < NCH ? s_qs[(ch / CPH) * DK + (ch % CPH) * 8 + e] : 0.f;
    }

    // ---- main loop over the warp's share [w0, w1) of the chunk
    const int n = j1 - j0;
    const int w0 = (int)((int64_t)n * warp / kScoreWarps), w1 = (int)((int64_t)n * (warp + 1) / kScoreWarps);
    const uint8_t *summ = reinterpret_cast<const uint8_t *>(a.summ);
    const uint64_t pol = l2_evict_first();
    uint4 v[U][NI];
    auto issue = [&](int i, uint4(&dst)[NI]) {
        const int p = i < w1 ? s_page[i] : -1;
#pragma unroll
        for (int c = 0; c < NI; ++c) {
            const int ch = lane + 32 * c;
            dst[c] = (p >= 0 && ch < NCH) ? ldg_stream_v4(summ + (int64_t)p * HKV * DK * 2 + ch * 16, pol)
                                          : make_uint4(0, 0, 0, 0);
        }
    };
#pragma unroll
    for (int u = 0; u < U; ++u) issue(w0 + u, v[u]);
    for (int base = w0; base < w1; base += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u;
            const int p = i < w1 ? s_page[i] : -1;      // warp-uniform
            if (p >= 0) {
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
                        const int ch = lane + 32 * c;
                        if (ch < NCH && (lane % CPH) == 0)
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
            issue(i + U, v[u]);
        }
    }
}

// ============================================================ top-k

constexpr int kTopkThreads = 1024;
constexpr int kTopkMaxCols = 32768;

// Block-wide exclusive scan of one uint32 per thread.
__device__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_sums)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        uint32_t s = lane < nw ? warp_sums[lane] : 0u;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        if (lane < nw) warp_sums[lane] = s;   // inclusive
    }
    __syncthreads();
    const uint32_t before_warp = warp ? warp_sums[warp - 1] : 0u;
    const uint32_t r = before_warp + x - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kTopkThreads) k_topk_rows(TopkArgs a)
{
    pdl_enter();
    extern __shared__ uint32_t keys[];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t warp_sums[32];
    __shared__ uint32_t s_nvalid, s_digit, s_gt;

    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31;
    int n = a.num_cols ? a.num_cols[row] : a.cols;
    n = max(0, min(n, a.cols));
    if (tid == 0) s_nvalid = 0;
    __syncthreads();

    uint32_t cnt = 0;
    const float *srow = a.scores + (int64_t)row * a.cols;
    for (int i = tid; i < n; i += kTopkThreads) {
        const float s = srow[i];
        uint32_t key = 0;
        if (isnan(s)) {
            flag_error(a.status, LSA_ERR_NAN);
        } else if (s != -INFINITY) {
            key = float_to_key(s);
            ++cnt;
        }
        keys[i] = key;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    if (lane == 0 && cnt) atomicAdd(&s_nvalid, cnt);
    __syncthreads();
    const uint32_t nvalid = s_nvalid;
    const uint32_t keff = min((uint32_t)max(a.k, 0), nvalid);

    uint32_t thresh = 0, take_eq = 0;   // select key > thresh, and the first take_eq with key == thresh
    if (keff > 0 && keff < nvalid) {
        uint32_t prefix = 0, mask = 0, remaining = keff;
        for (int shift = 24; shift >= 0; shift -= 8) {
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
            for (int base = 0; base < n; base += kTopkThreads) {
                const int i = base + tid;
                const uint32_t key = i < n ? keys[i] : 0u;
                const bool in = key != 0 && (key & mask) == prefix;
                const uint32_t digit = (key >> shift) & 0xffu;
                const uint32_t act = __ballot_sync(0xffffffffu, in);
                if (in) {
                    const uint32_t peers = __match_any_sync(act, digit);
                    if ((__ffs(peers) - 1) == lane) atomicAdd(&hist[digit], __popc(peers));
                }
            }
            __syncthreads();
            if (tid < 32) {
                // lane l owns digits 8l .. 8l+7; find the digit whose bucket
                // holds the remaining-th largest key
                uint32_t c[8], tot = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    c[e] = hist[8 * lane + e];
                    tot += c[e];
                }
                // above = sum of the totals of lanes > lane
                uint32_t incl = tot;   // inclusive suffix scan over lanes
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    uint32_t y = __shfl_down_sync(0xffffffffu, incl, off);
                    if (lane + off < 32) incl += y;
                }
                uint32_t gt = incl - tot;
#pragma unroll
                for (int e = 7; e >= 0; --e) {
                    if (gt < remaining && remaining <= gt + c[e]) {
                        s_digit = 8 * lane + e;
                        s_gt = gt;
                    }
                    gt += c[e];
                }
            }
            __syncthreads();
            prefix |= s_digit << shift;
            mask |= 0xffu << shift;
            remaining -= s_gt;
            __syncthreads();
        }
        thresh = prefix;
        take_eq = remaining;
    }

    // compact the selected columns in index order
    const int per = (n + kTopkThreads - 1) / kTopkThreads;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    uint32_t ngt = 0, neq = 0;
    if (keff > 0) {
        for (int i = lo; i < hi; ++i) {
            const uint32_t key = keys[i];
            ngt += key != 0 && key > thresh;
            neq += key != 0 && key == thresh;
        }
    }
    const uint32_t packed = block_excl_scan((ngt << 16) | neq, warp_sums);
    uint32_t gt_before = packed >> 16, eq_before = packed & 0xffffu;
    int32_t *orow = a.idx + (int64_t)row * a.k;
    if (keff > 0) {
        for (int i = lo; i < hi; ++i) {
            const uint32_t key = keys[i];
            if (key == 0) continue;
            int pos = -1;
            if (key > thresh) {
                pos = (int)(gt_before + min(eq_before, take_eq));
                ++gt_before;
            } else if (key == thresh) {
                if (eq_before < take_eq) pos = (int)(gt_before + eq_before);
                ++eq_before;
            }
            if (pos >= 0) {
                int out = i;
                if (a.cand) {
                    const int cb = a.cand[(int64_t)row * a.ncand + i / a.b];
                    out = cb * a.b + i % a.b;
                }
                orow[pos] = out;
            }
        }
    }
    for (int i = (int)keff + tid; i < a.k; i += kTopkThreads) orow[i] = -1;
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

    float qs[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) qs[e] = 0.f;
    for (int g = 0; g < G; ++g) {
        const uint16_t *qg = a.q + ((int64_t)r * a.hq + h * G + g) * 128 + sub * 16;
        const uint4 v0 = *reinterpret_cast<const uint4 *>(qg);
        const uint4 v1 = *reinterpret_cast<const uint4 *>(qg + 8);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float2 f = bf2_to_f2(w[e]);
            qs[2 * e] += f.x;
            qs[2 * e + 1] += f.y;
        }
    }

    const int L = a.lens[r];
    const int nfull = (L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * b) ? L / b : 0;
    const int64_t ntok_row = (int64_t)a.ncand * b;
    float *frow = a.fscores + (int64_t)row * ntok_row;
    const int c0 = blockIdx.x * kFineBlocksPerCta;
    const int c1 = min(c0 + kFineBlocksPerCta, a.ncand);
    for (int ci = c0; ci < c1; ++ci) {
        const int j = a.cand[(int64_t)row * a.ncand + ci];
        int p = -1;
        if (j >= 0 && j < nfull) p = a.pt[(int64_t)r * a.max_blocks + j];
        const bool ok = p >= 0 && p < a.ic.num_pages;
        if (!ok) {
            if (j != -1 && warp == 0 && lane == 0) flag_error(a.status, LSA_ERR_BOUNDS);
            for (int t = threadIdx.x; t < b; t += blockDim.x) frow[(int64_t)ci * b + t] = -INFINITY;
            continue;
        }
        const uint8_t *kb = a.ic.k + (int64_t)p * a.ic.kps + (int64_t)h * a.ic.khs;
        const float *sb = a.ic.kscale + (int64_t)p * a.ic.sps + (int64_t)h * a.ic.shs;
        for (int t0 = warp * 4; t0 < b; t0 += kFineWarps * 4) {
            const int t = t0 + tq;
            float acc = 0.f;
            if (t < b) {
                const uint4 v = ldg_nc_v4(kb + (int64_t)t * a.ic.kts + sub * 16);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 lo = e4m3x2_to_f2((uint16_t)(w[e] & 0xffffu));
                    float2 hi = e4m3x2_to_f2((uint16_t)(w[e] >> 16));
                    acc = fmaf(qs[4 * e + 0], lo.x, acc);
                    acc = fmaf(qs[4 * e + 1], lo.y, acc);
                    acc = fmaf(qs[4 * e + 2], hi.x, acc);
                    acc = fmaf(qs[4 * e + 3], hi.y, acc);
                }
            }
#pragma unroll
            for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (t < b && sub == 0) frow[(int64_t)ci * b + t] = sb[t] * acc;
        }
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
    if (launch_topk_fast(a, s, &fe)) return fe;   // rows of up to 8192 columns
    const size_t smem = (size_t)max(a.cols, 1) * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(k_topk_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_step_kernel(k_topk_rows, dim3(a.rows), dim3(kTopkThreads), smem, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_fine_scores(const FineArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = a.ic.dk != 128 || !a.ic.e4m3 || a.ic.b % 4 != 0;
    if (*unsupported || a.batch == 0 || a.ncand == 0) return cudaSuccess;
    dim3 grid((a.ncand + kFineBlocksPerCta - 1) / kFineBlocksPerCta, a.batch * a.ic.hkv);
    cudaError_t le = launch_step_kernel(k_fine_scores, grid, dim3(kFineWarps * 32), 0, s, a);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

}  // namespace lsa

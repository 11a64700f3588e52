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
constexpr int kScoreUnroll = 4;     // summary rows in flight per warp
constexpr int kScoreMaxChunk = 1024;

template <int DK, int HKV>
__global__ void __launch_bounds__(kScoreWarps * 32) k_score(ScoreArgs a)
{
    constexpr int NCH = HKV * DK / 8;      // 16-byte chunks of one page's summary row
    constexpr int NI = (NCH + 31) / 32;    // chunks per lane
    constexpr int CPH = DK / 8;            // chunks per head
    constexpr bool kGroupReduce = (CPH <= 32) && (32 % CPH == 0);
    static_assert(kGroupReduce || HKV == 1, "head rows must tile the warp");
    __shared__ int s_page[kScoreMaxChunk];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.y;
    const int G = a.hq / HKV;

    const int L = a.lens[r];
    const bool len_ok = L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * a.b;
    if (!len_ok && threadIdx.x == 0 && blockIdx.x == 0) flag_error(a.status, LSA_ERR_BOUNDS);
    const int se = min(a.sink, max(L, 0));
    const int rs = max(L - a.recent, se);
    const int j0 = blockIdx.x * a.chunk;
    const int j1 = min(j0 + a.chunk, a.max_blocks);

    // page ids of the chunk's candidate blocks (-1: not a candidate); the
    // other blocks get -inf right away
    for (int j = j0 + threadIdx.x; j < j1; j += blockDim.x) {
        const bool cand = len_ok && (int64_t)j * a.b >= se && (int64_t)(j + 1) * a.b <= rs;
        int p = cand ? a.pt[(int64_t)r * a.max_blocks + j] : -1;
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

    // q_sum = sum of the group's queries, for this lane's chunks (fp32)
    float qs[NI][8];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int ch = lane + 32 * i;
#pragma unroll
        for (int e = 0; e < 8; ++e) qs[i][e] = 0.f;
        if (ch < NCH) {
            const int h = ch / CPH, d0 = (ch % CPH) * 8;
            for (int g = 0; g < G; ++g) {
                const uint4 v = *reinterpret_cast<const uint4 *>(a.q + ((int64_t)r * a.hq + h * G + g) * DK + d0);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 f = bf2_to_f2(w[e]);
                    qs[i][2 * e] += f.x;
                    qs[i][2 * e + 1] += f.y;
                }
            }
        }
    }
    __syncthreads();

    const uint8_t *summ = reinterpret_cast<const uint8_t *>(a.summ);
    for (int jb = j0 + warp * kScoreUnroll; jb < j1; jb += kScoreWarps * kScoreUnroll) {
        uint4 v[kScoreUnroll][NI];
        int pg[kScoreUnroll];
#pragma unroll
        for (int u = 0; u < kScoreUnroll; ++u) {
            const int j = jb + u;
            pg[u] = j < j1 ? s_page[j - j0] : -1;
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const int ch = lane + 32 * i;
                v[u][i] = make_uint4(0, 0, 0, 0);
                if (pg[u] >= 0 && ch < NCH) v[u][i] = ldg_nc_v4(summ + (int64_t)pg[u] * HKV * DK * 2 + ch * 16);
            }
        }
#pragma unroll
        for (int u = 0; u < kScoreUnroll; ++u) {
            if (pg[u] < 0) continue;       // warp-uniform
            const int j = jb + u;
            float part[NI];
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                const uint32_t w[4] = {v[u][i].x, v[u][i].y, v[u][i].z, v[u][i].w};
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 f = bf2_to_f2(w[e]);
                    acc = fmaf(qs[i][2 * e], f.x, acc);
                    acc = fmaf(qs[i][2 * e + 1], f.y, acc);
                }
                part[i] = acc;
            }
            if constexpr (kGroupReduce) {
#pragma unroll
                for (int i = 0; i < NI; ++i) {
#pragma unroll
                    for (int off = CPH / 2; off > 0; off >>= 1)
                        part[i] += __shfl_xor_sync(0xffffffffu, part[i], off);
                    const int ch = lane + 32 * i;
                    if (ch < NCH && (lane % CPH) == 0)
                        a.scores[((int64_t)r * HKV + ch / CPH) * a.max_blocks + j] = part[i];
                }
            } else {
                float tot = 0.f;
#pragma unroll
                for (int i = 0; i < NI; ++i) tot += part[i];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
                if (lane == 0) a.scores[(int64_t)r * a.max_blocks + j] = tot;
            }
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
    k_score<DK, HKV><<<grid, kScoreWarps * 32, 0, s>>>(a);
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
    // one wave of CTAs (two per SM), chunk a multiple of the warps' stride
    const int64_t target = 2LL * sms;
    int64_t per = ((int64_t)batch * max_blocks + target - 1) / target;
    const int step = kScoreWarps * kScoreUnroll;
    per = ((per + step - 1) / step) * step;
    if (per < step) per = step;
    if (per > kScoreMaxChunk) per = kScoreMaxChunk;
    return (int)per;
}

cudaError_t launch_topk(const TopkArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = a.cols > kTopkMaxCols;
    if (*unsupported || a.rows == 0 || a.k == 0) return cudaSuccess;
    const size_t smem = (size_t)max(a.cols, 1) * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(k_topk_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_topk_rows<<<a.rows, kTopkThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fine_scores(const FineArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = a.ic.dk != 128 || !a.ic.e4m3 || a.ic.b % 4 != 0;
    if (*unsupported || a.batch == 0 || a.ncand == 0) return cudaSuccess;
    dim3 grid((a.ncand + kFineBlocksPerCta - 1) / kFineBlocksPerCta, a.batch * a.ic.hkv);
    k_fine_scores<<<grid, kFineWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace lsa

// PQ32 coarse-to-fine index selection (LeanSparse, Section 5
// "Coarse-to-fine decode indexing", "Approximate scoring with PQ", Eq. 6,
// and "Retrieving and refining candidates").
//
// A 128-dim index key is split into 32 four-dim subvectors, each stored as a
// one-byte index into a codebook of 256 centroids per subspace (PQ32, 32
// bytes a token).  A decode step
//   1. scores every encoded token with the centroids in place of its
//      subvectors, inside the indexer's weighted head aggregation,
//        s~_t = sum_g w_g ReLU(sum_j q_{g,j} . C_j[c_{t,j}])     (k_pq_scores)
//   2. keeps the top C tokens by s~ (k_pq_hist, then k_pq_select),
//   3. keeps, of those, every one whose original index key is cached and
//      every other one whose s~ is at least the candidates' k-th largest s~
//      minus one sample standard deviation (the miss filter),
//   4. rescores the kept candidates and the unencoded tail (the partial
//      last block) exactly from their FP8 keys, and selects the top k
//      tokens (k_pq_select).
//
// k_pq_scores decodes the codes of 128 tokens at a time into a bf16 key
// tile (centroids exactly, from a shared-memory copy of the codebook) and
// forms the dots of all 64 heads as one tcgen05 product into tensor memory:
//   S^T [128 tokens x 64 heads] = K~_tile [128 x 128] . Q^T [128 x 64]
// -- bf16 operands, fp32 accumulation, exact products -- then each thread
// reads its token's 64 dots and applies the weighted ReLU.  The selection
// over rows of up to max_blocks * b tokens buckets the scores by a linear
// remap between the row's smallest and largest score (as the top-k of
// topk_bucket.cuh; the extremes are gathered by k_pq_scores, the counts by
// k_pq_hist), so that one cluster per request can find the C-th largest
// score's bucket without sorting the row.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "fine_tile.cuh"
#include "topk_cluster.cuh"

namespace lsa {
namespace {

// ---------------------------------------------------------------- encoding

// PQ32 codes of every token of every full block (the encoded history), by
// nearest centroid: per subspace, the smallest squared distance between the
// dequantised key scale_t * e4m3(k8_t) and a centroid, ties to the lower
// centroid.  The distance decides an integer, so it is taken in one fixed
// fp32 order with no fused multiply-add:
//   k = scale * e4m3, d_e = k_e - C_e, dist = ((d_0^2 + d_1^2) + d_2^2) + d_3^2.
// A warp takes 32 tokens of one subspace, so every lane reads the same
// centroid (a broadcast).  The codebook is held in shared memory as fp32.
constexpr int kPeThreads = 256;
constexpr int kPeSmem = 32 * 256 * 4 * 4;

__global__ void __launch_bounds__(kPeThreads) k_pq_encode(PqArgs a)
{
    pdl_enter();
    extern __shared__ __align__(16) uint8_t pesm[];
    float *cbf = reinterpret_cast<float *>(pesm);
    for (int i = threadIdx.x; i < 32 * 256 * 2; i += kPeThreads) {
        const float2 f = bf2_to_f2(reinterpret_cast<const uint32_t *>(a.codebook)[i]);
        cbf[2 * i] = f.x;
        cbf[2 * i + 1] = f.y;
    }
    __syncthreads();
    const int r = blockIdx.y;
    const int b = a.ic.b;
    const int L = a.lens[r];
    const bool len_ok = L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * b;
    if (!len_ok) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(a.status, LSA_ERR_BOUNDS);
        return;
    }
    const int nfull = L / b;
    for (int j = blockIdx.x; j < nfull; j += gridDim.x) {
        const int p = a.pt[(int64_t)r * a.max_blocks + j];
        if (p < 0 || p >= a.ic.num_pages) {
            if (threadIdx.x == 0) flag_error(a.status, LSA_ERR_BOUNDS);
            continue;
        }
        for (int task = threadIdx.x; task < b * 32; task += kPeThreads) {
            const int sub = task / b, t = task - sub * b;
            const uint32_t four =
                *reinterpret_cast<const uint32_t *>(a.ic.k + (int64_t)p * a.ic.kps + (int64_t)t * a.ic.kts + 4 * sub);
            const float sc = a.ic.kscale[(int64_t)p * a.ic.sps + t];
            const float2 lo = e4m3x2_to_f2((uint16_t)(four & 0xffffu)), hi = e4m3x2_to_f2((uint16_t)(four >> 16));
            const float k0 = __fmul_rn(sc, lo.x), k1 = __fmul_rn(sc, lo.y);
            const float k2 = __fmul_rn(sc, hi.x), k3 = __fmul_rn(sc, hi.y);
            const float4 *cj = reinterpret_cast<const float4 *>(cbf) + sub * 256;
            int best = 0;
            float bd = INFINITY;
            for (int c = 0; c < 256; ++c) {
                const float4 cv = cj[c];
                const float d0 = __fsub_rn(k0, cv.x), d1 = __fsub_rn(k1, cv.y);
                const float d2 = __fsub_rn(k2, cv.z), d3 = __fsub_rn(k3, cv.w);
                const float dist = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(d0, d0), __fmul_rn(d1, d1)), __fmul_rn(d2, d2)),
                                             __fmul_rn(d3, d3));
                if (dist < bd) {
                    bd = dist;
                    best = c;
                }
            }
            a.codes_out[((int64_t)p * b + t) * 32 + sub] = (uint8_t)best;
        }
    }
}

// ---------------------------------------------------------------- coarse scores

// Four warps a CTA, two CTAs an SM, tiles of 128 tokens strided over the
// grid.  Thread p owns token row p of a tile, which is TMEM lane p (warp w
// writes and reads lane quadrant w).  For tile i it decodes its token's 32
// centroids into 64 registers (two bf16 a 32-bit word, dims in order) and
// writes them into its lane of the A buffer i & 1 (tcgen05.st), once the
// product that last read that buffer has completed; thread 0 then issues
// the tile's product with A from tensor memory,
//   S^T [128 tokens x 64 heads] = K~ [128 x 128] . Q^T [128 x 64],
// Q^T the request's query tile in shared memory, into accumulator i & 1,
// and while it runs every thread reads the accumulator of tile i - 1 and
// applies the weighted ReLU.  The decoded keys never pass through shared
// memory: the only shared-memory traffic is the codebook lookups and the
// product's reads of the query tile.  Each thread loads its codes a tile
// ahead and its page id two tiles ahead.
constexpr int kPsThreads = 128;     // warps 0-3: every warp can reach its TMEM lane quadrant
constexpr int kPsCtasPerSm = 2;
constexpr int kPsTok = 128;         // tokens per tile (the MMA's M)
constexpr int kPsHeads = 64;        // query heads (the MMA's N)

struct PsLayout {
    static constexpr int CB = 0;                          // codebook, bf16 [32][256][4]
    static constexpr int QCOL = (kPsHeads / 8) * 1024;    // one 64-dim atom column of a query tile
    static constexpr int QS = 32 * 256 * 8;               // query tiles: 2 slots x 2 atom columns
    static constexpr int CRING = 3;                       // codes in flight: tiles i, i + 1, i + 2
    static constexpr int PRING = 4;                       // page ids: tiles i + 2, i + 3 (and two spare)
    static constexpr int CODES = QS + 4 * QCOL;           // [CRING][128 threads] 32 bytes of codes
    static constexpr int PGS = CODES + CRING * kPsThreads * 32;  // [PRING][128 threads] page ids
    static constexpr int BAR = PGS + PRING * kPsThreads * 4;     // mma[2], stored[2], TMEM base address
    static constexpr int SMEM = BAR + 48;
    static constexpr int TA = 0;                          // TMEM columns: A buffers 2 x 64 (128 dims, two a column)
    static constexpr int TD = 128;                        // accumulators 2 x 64 (64 heads)
    static constexpr int TCOLS = 256;
    static_assert(QS % 1024 == 0, "swizzled atoms are 1024-byte aligned");
    static_assert(kPsCtasPerSm * TCOLS <= 512, "tensor memory of one SM");
    static_assert(kPsCtasPerSm * SMEM <= 227 * 1024, "shared memory of one SM");
};

// Whether block j of a request is a candidate: full and outside the forced
// sink [0, se) and recent [rs, L) ranges.
__device__ __forceinline__ bool pq_block_candidate(int64_t j, int b, int64_t se, int64_t rs)
{
    return j * b >= se && (j + 1) * b <= rs;
}

// Adds a warp's extremes of request r's scores to the row's.
__device__ __forceinline__ void pq_flush_ext(uint32_t *row_ext, int r, uint32_t kmax, uint32_t kmin)
{
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    if ((threadIdx.x & 31) == 0 && kmax != 0u && row_ext) {
        atomicMax(row_ext + 2 * r, kmax);
        atomicMax(row_ext + 2 * r + 1, ~kmin);
    }
}


__global__ void __launch_bounds__(kPsThreads, kPsCtasPerSm) k_pq_scores(PqArgs a)
{
    pdl_enter();
    using LY = PsLayout;
    constexpr uint32_t IDESC = umma_idesc_bf16(kPsTok, kPsHeads, false, false);
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5;
    if ((smem_addr(smem) & 1023u) != 0) {
        if (tid == 0) flag_error(a.status, LSA_ERR_INVALID_ARG);
        return;
    }
    uint64_t *mma = reinterpret_cast<uint64_t *>(smem + LY::BAR);   // product of buffer b done
    uint64_t *stored = mma + 2;                                        // buffer b's rows (and query tile) in place
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + LY::BAR + 32);
    const uint32_t sbase = smem_addr(smem);
    if (warp == 0) {
        tmem_alloc(tslot, LY::TCOLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&mma[0], 1);
        mbar_init(&mma[1], 1);
        mbar_init(&stored[0], kPsThreads);
        mbar_init(&stored[1], kPsThreads);
        fence_barrier_init();
    }
    // the codebook, once per CTA
    for (int i = tid; i < 32 * 256 * 8 / 16; i += kPsThreads)
        cp_async16(sbase + LY::CB + i * 16, reinterpret_cast<const uint8_t *>(a.codebook) + i * 16);
    cp_async_commit();
    cp_async_wait<0>();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

    const int b = a.ic.b;
    const int T = a.max_blocks * b;
    const int tpr = (T + kPsTok - 1) / kPsTok;
    const int total = a.batch * tpr;
    const int ntiles = (int)blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto tile_of = [&](int i) { return (int)blockIdx.x + i * (int)gridDim.x; };
    const int p = tid;   // this thread's key row

    // this thread's token of tile i and whether it is scored (the request's
    // length is read once per request)
    int len_r = -1, len_v = 0;
    auto token_of = [&](int i, int &r, int &tok) -> bool {
        const int tile = tile_of(i);
        r = (int)fdiv((uint32_t)tile, a.fd_tpr);
        tok = (tile - r * tpr) * kPsTok + p;
        if (r != len_r) {
            len_r = r;
            len_v = a.lens[r];
            if (!(len_v >= 0 && (int64_t)len_v <= (int64_t)T) && p == 0) flag_error(a.status, LSA_ERR_BOUNDS);
        }
        const int L = len_v;
        const bool len_ok = L >= 0 && (int64_t)L <= (int64_t)T;
        const int64_t se = len_ok ? min(a.sink, L) : 0;
        const int64_t rs = len_ok ? max((int64_t)L - a.recent, se) : 0;
        const int nfull_tok = len_ok ? (int)fdiv((uint32_t)L, a.fd_b) * b : 0;
        return tok < nfull_tok && pq_block_candidate(fdiv((uint32_t)tok, a.fd_b), b, se, rs);
    };

    // this thread's prefetch ring (its own slots, so no barrier): the page
    // id of tile i + 3 and the codes of tile i + 2 are requested while tile
    // i decodes, by cp.async, so that no register waits on a load; stage
    // s % CRING (codes) and s % PRING (page ids) belong to tile s.  A tile whose token is not
    // scored (or whose page id is bad) loads nothing and decodes zeros.
    const uint32_t ring_codes = sbase + LY::CODES + p * 32;
    const uint32_t ring_pg = sbase + LY::PGS + p * 4;
    const int *pg_s = reinterpret_cast<const int *>(smem + LY::PGS) + p;
    auto codes_at = [&](int i) -> const uint4 * {
        return reinterpret_cast<const uint4 *>(smem + LY::CODES + ((i % LY::CRING) * kPsThreads + p) * 32);
    };
    auto request_pg = [&](int i, bool scored, int r, int tk) {   // page id of tile i's token
        if (scored)
            cp_async4(ring_pg + (i % LY::PRING) * kPsThreads * 4,
                      a.pt + (int64_t)r * a.max_blocks + fdiv((uint32_t)tk, a.fd_b));
        cp_async_commit();
    };
    auto request_codes = [&](int i, bool &scored, int tk) {      // codes of tile i's token, its page id in place
        if (scored) {
            const int pg = pg_s[(i % LY::PRING) * kPsThreads];
            if (pg < 0 || pg >= a.ic.num_pages) {
                flag_error(a.status, LSA_ERR_BOUNDS);
                scored = false;
            } else {
                const uint8_t *src = a.codes + ((int64_t)pg * b + (tk - (int)fdiv((uint32_t)tk, a.fd_b) * b)) * 32;
                const uint32_t dst = ring_codes + (i % LY::CRING) * kPsThreads * 32;
                cp_async16(dst, src);
                cp_async16(dst + 16, src + 16);
            }
        }
        cp_async_commit();
    };
    // tiles 0 .. 2: page ids of 0, 1, 2, then the codes of 0 and 1
    int rq[3] = {0, 0, 0}, tq[3] = {0, 0, 0};
    bool vq[3] = {false, false, false};
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        vq[k] = k < ntiles && token_of(k, rq[k], tq[k]);
        request_pg(k, vq[k], rq[k], tq[k]);
    }
    cp_async_wait<0>();
    request_codes(0, vq[0], tq[0]);
    request_codes(1, vq[1], tq[1]);
    // the ring's state entering iteration i: tile i's and i+1's codes are
    // requested (validity v, v1), tile i+2's page id is requested (v2)
    bool v = vq[0], v1 = vq[1], v2 = vq[2];
    int tok = tq[0], tok1 = tq[1], tok2 = tq[2];

    // No CTA barrier inside the loop, so that the warps drift apart and one
    // warp's codebook lookups overlap another's epilogue: a thread arrives
    // on stored[b] once its rows (and its part of a new query tile) are in
    // place, warp 0 waits for all of them and issues the product, and every
    // thread waits for the product's commit itself.  The request's head
    // weights live in each thread's registers.  A wait that gives up ends
    // the thread's loop; the others' waits then give up as well.
    int cur = -1;                // request of the weights in registers and of the row extremes
    float wreg[kPsHeads];
    uint32_t kmax = 0u, kmin = 0xffffffffu;
    int q_req0 = -1, q_req1 = -1;   // request of each query slot
    int slot = 0;
    int tokA = -1, tokB = -1;      // this thread's token (-1: not scored) of the tile in each accumulator
    int reqA = 0, reqB = 0;
    int issued0 = -1, issued1 = -1;
    bool ok = true;
    auto epilogue = [&](int i) -> bool {
        const int buf = i & 1;
        if (!mbar_wait(&mma[buf], (i >> 1) & 1, a.status, a.spin_budget)) return false;
        tc_fence_after();
        const int r = buf ? reqB : reqA;
        const int tk = buf ? tokB : tokA;
        if (r != cur) {
            if (cur >= 0) pq_flush_ext(a.row_ext, cur, kmax, kmin);
            kmax = 0u;
            kmin = 0xffffffffu;
            cur = r;
            const float4 *wr = reinterpret_cast<const float4 *>(a.weights + (int64_t)r * a.hq);
#pragma unroll
            for (int g = 0; g < kPsHeads / 4; ++g) {
                const float4 w4 = __ldg(wr + g);
                wreg[4 * g] = w4.x;
                wreg[4 * g + 1] = w4.y;
                wreg[4 * g + 2] = w4.z;
                wreg[4 * g + 3] = w4.w;
            }
        }
        float d[32];
        float2 s2 = make_float2(0.f, 0.f);   // even and odd heads, added at the end
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tmem_ld32(tmem + lane_base + LY::TD + 64 * buf + 32 * half, d);
#pragma unroll
            for (int g = 0; g < 32; g += 2)
                s2 = __ffma2_rn(make_float2(wreg[32 * half + g], wreg[32 * half + g + 1]),
                                make_float2(fmaxf(d[g], 0.f), fmaxf(d[g + 1], 0.f)), s2);
        }
        const float s = s2.x + s2.y;
        const bool valid = tk >= 0;
        if (valid) {
            if (isnan(s)) flag_error(a.status, LSA_ERR_NAN);
            else {
                const uint32_t key = float_to_key(s);
                kmax = max(kmax, key);
                kmin = min(kmin, key);
            }
        }
        const int tok_row = (tile_of(i) - r * tpr) * kPsTok + p;
        if (tok_row < T) a.coarse[(int64_t)r * T + tok_row] = valid && !isnan(s) ? s : -INFINITY;
        return true;
    };

    for (int i = 0; i < ntiles && ok; ++i) {
        const int buf = i & 1;
        const int r = (int)fdiv((uint32_t)tile_of(i), a.fd_tpr);
        // this thread's key row of tile i, two bf16 a word, dims in order
        uint32_t row[64];
        {
            // groups committed so far: ..., codes i, [page i+2 | codes i+1]; all
            // but the last (codes i+1) are complete after this wait
            cp_async_wait<1>();
            const uint4 c0 = codes_at(i)[0], c1 = codes_at(i)[1];
            const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const uint32_t cj = __byte_perm(cw[jj >> 2], 0u, 0x4440u | (uint32_t)(jj & 3));
                const uint2 e = v ? *reinterpret_cast<const uint2 *>(smem + LY::CB + (jj * 256 + cj) * 8)
                                  : make_uint2(0u, 0u);
                row[2 * jj] = e.x;
                row[2 * jj + 1] = e.y;
            }
        }
        if (buf) {
            tokB = v ? tok : -1;
            reqB = r;
        } else {
            tokA = v ? tok : -1;
            reqA = r;
        }
        // page id of tile i + 3, codes of tile i + 2 (its page id is in:
        // requested two groups ago)
        int r3 = 0, tok3 = 0;
        const bool v3 = i + 3 < ntiles && token_of(i + 3, r3, tok3);
        request_pg(i + 3, v3, r3, tok3);
        bool v2c = v2;
        request_codes(i + 2, v2c, tok2);
        // A buffer and accumulator `buf` are free once tile i - 2's product
        // is done (this thread read that accumulator in the last iteration)
        if (i >= 2 && !mbar_wait(&mma[buf], ((i - 2) >> 1) & 1, a.status, a.spin_budget)) {
            ok = false;
            break;
        }
        const int q_cur = slot ? q_req1 : q_req0;
        if (r != q_cur) {
            // a new request: its query tile goes to the other slot, whose last
            // reader (tile i - 2 at the latest) is done; this thread's part
            // of it is in place before the thread arrives below
            slot ^= 1;
            if (slot) q_req1 = r;
            else q_req0 = r;
            const uint8_t *qg = reinterpret_cast<const uint8_t *>(a.q + (int64_t)r * a.hq * 128);
            const int j = tid & 7;
            for (int task = tid >> 3; task < 2 * kPsHeads; task += kPsThreads / 8) {
                const int cc = task >> 6, g = task & (kPsHeads - 1);
                cp_async16(sbase + LY::QS + (2 * slot + cc) * LY::QCOL + atom_offset(g, j),
                           qg + (int64_t)g * 256 + cc * 128 + j * 16);
            }
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
        }
        tmem_st32(tmem + lane_base + LY::TA + 64 * buf, *reinterpret_cast<const uint32_t(*)[32]>(row));
        tmem_st32(tmem + lane_base + LY::TA + 64 * buf + 32, *reinterpret_cast<const uint32_t(*)[32]>(row + 32));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&stored[buf]);
        if (warp == 0) {
            // the tile's product, once every thread's rows are in place
            if (!mbar_wait(&stored[buf], (i >> 1) & 1, a.status, a.spin_budget)) {
                ok = false;
                break;
            }
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t bd =
                        umma_desc_sw128(sbase + LY::QS + (2 * slot + (ks >> 2)) * LY::QCOL + (ks & 3) * 32, 16, 1024);
                    umma_bf16_ta(tmem + LY::TD + 64 * buf, tmem + LY::TA + 64 * buf + 8 * ks, bd, IDESC, ks > 0);
                }
                umma_commit(&mma[buf]);
            }
            __syncwarp();
        }
        if (buf) issued1 = i;
        else issued0 = i;
        // while it runs, the previous tile's scores
        if (i >= 1 && !epilogue(i - 1)) {
            ok = false;
            break;
        }
        v = v1;
        tok = tok1;
        v1 = v2c;
        tok1 = tok2;
        v2 = v3;
        tok2 = tok3;
    }
    cp_async_wait<0>();   // nothing of this thread's ring is left in flight
    if (ok && ntiles > 0) ok = epilogue(ntiles - 1);
    if (cur >= 0) pq_flush_ext(a.row_ext, cur, kmax, kmin);
    if (!ok) {
        // a wait gave up: wait (bounded) for the products issued before the
        // tensor memory is freed
        if (issued0 >= 0) mbar_wait(&mma[0], (issued0 >> 1) & 1, nullptr, a.spin_budget);
        if (issued1 >= 0) mbar_wait(&mma[1], (issued1 >> 1) & 1, nullptr, a.spin_budget);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, LY::TCOLS);
}

// ---------------------------------------------------------------- histogram

// Bucket counts of each request's coarse scores, over kPqBins buckets of a
// linear remap between the row's smallest and largest score (the remap of
// topk_bucket.cuh, in fp32); a CTA counts kPhTok scores in shared memory and
// adds its nonzero counts to the row's.
constexpr int kPhThreads = 256;
constexpr int kPhTok = 8192;

__device__ __forceinline__ int pq_bucket(float x, float vmin, float scale)
{
    if (scale == 0.f) return 0;
    const float y = (x - vmin) * scale;
    return y >= (float)(kPqBins - 1) ? kPqBins - 1 : (int)y;
}

__device__ __forceinline__ void pq_remap(const uint32_t *row_ext, int r, float *vmin, float *scale)
{
    const uint32_t kmax = __ldcg(row_ext + 2 * r), kmin = ~__ldcg(row_ext + 2 * r + 1);
    *vmin = key_to_float(kmin);
    const float span = key_to_float(kmax) - *vmin;
    *scale = (span > 0.f && span < INFINITY) ? (float)kPqBins / span : 0.f;
}

__global__ void __launch_bounds__(kPhThreads) k_pq_hist(PqArgs a)
{
    pdl_enter();
    __shared__ uint32_t h[kPqBins];
    const int r = blockIdx.y;
    const int T = a.max_blocks * a.ic.b;
    const int t0 = blockIdx.x * kPhTok, t1 = min(t0 + kPhTok, T);
    for (int i = threadIdx.x; i < kPqBins; i += kPhThreads) h[i] = 0u;
    float vmin, scale;
    pq_remap(a.row_ext, r, &vmin, &scale);
    __syncthreads();
    // this thread's chunks of four scores, all loads in flight at once (T
    // and t0 are multiples of four: block sizes are multiples of 16)
    const float4 *row4 = reinterpret_cast<const float4 *>(a.coarse + (int64_t)r * T);
    constexpr int kPer = kPhTok / 4 / kPhThreads;
    float4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int i4 = t0 / 4 + threadIdx.x + u * kPhThreads;
        v[u] = 4 * i4 < t1 ? __ldcg(row4 + i4) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const float xs[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (xs[e] == -INFINITY || isnan(xs[e])) continue;
            atomicAdd(&h[pq_bucket(key_to_float(float_to_key(xs[e])), vmin, scale)], 1u);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kPqBins; i += kPhThreads)
        if (h[i]) atomicAdd(a.hist + (int64_t)r * kPqBins + i, h[i]);
}

// ---------------------------------------------------------------- selection

// One cluster of CS CTAs per request.  CTA c reads slice c of the request's
// coarse scores (thread-contiguous ranges, so that counts in thread order
// are counts in token order) and owns candidate positions [c * CB, (c + 1)
// * CB) of the top C; the tail tokens go to the last CTA.
struct PqSelLayout {
    static constexpr int KEYS = 0;                         // [kFtTok][128] FP8 key rows (cf_key_off)
    static constexpr int PART = KEYS + kFtTok * 128;       // [4][kFtTok] fp32 head-tile partials
    static constexpr int FS = PART + 4 * kFtTok * 4;       // [kFtTok] fp32 fine scores
    static constexpr int SC = FS + kFtTok * 4;             // [kFtTok] fp32 token scales
    static constexpr int CAND = SC + kFtTok * 4;           // [kFtTok] (int32 token, fp32 coarse score): this
                                                           // CTA's candidates, written by the cluster
    static constexpr int FTOK = CAND + kFtTok * 8;         // [kFtTok] int32 the tokens this CTA rescores
    static constexpr int FPG = FTOK + kFtTok * 4;          // [kFtTok] int32 their pages
    static constexpr int CPG = FPG + kFtTok * 4;           // [kFtTok] int32 the candidates' pages
    static constexpr int HIST = CPG + kFtTok * 4;          // [kPqBins] the row's bucket counts
    static constexpr int CKT = HIST + kPqBins * 4;         // [kBkCap] int32 this CTA's boundary tokens
    static constexpr int DX = CKT + kBkCap * 4;            // [5] fp64 exchange slots, [kFtWarps + 1] fp64 warp sums
    static constexpr int SMEM = DX + (5 + kFtWarps + 1) * 8;
};
static_assert(PqSelLayout::SMEM + sizeof(ClusterTopkScratch<kFtThreads, 8>) <= 227 * 1024, "shared memory");

// The coarse scores each CTA of a request's cluster reads: ceil(T / CS)
// rounded up to whole chunks of four tokens for every thread.
__host__ __device__ __forceinline__ int pq_slice(int T, int cs)
{
    return ((T + cs - 1) / cs + 4 * kFtThreads - 1) / (4 * kFtThreads) * (4 * kFtThreads);
}

// Sum over the CTA of every thread's fp64 value, in a fixed order (lanes,
// then warps), returned to every thread.  ws: kFtWarps + 1 doubles.  One
// thread adds the warps' sums (fp64 arithmetic is slow on this part: the
// other threads only read the result).
__device__ __forceinline__ double pq_block_dsum(double v, double *ws)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
#pragma unroll
        for (int w = 0; w < kFtWarps; ++w) s += ws[w];
        ws[kFtWarps] = s;
    }
    __syncthreads();
    const double s = ws[kFtWarps];
    __syncthreads();   // ws may be reused
    return s;
}

template <int CS>
__global__ void __launch_bounds__(kFtThreads, 1) k_pq_select(PqArgs a)
{
    using LY = PqSelLayout;
    constexpr int NT = kFtThreads;
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ ClusterTopkScratch<NT, CS> tsm;
    __shared__ uint32_t s_off[2][CS + 1];   // per-CTA prefix of winners / boundary keys (or > T / == T)
    __shared__ uint32_t s_u[8];
    const int tid = threadIdx.x;
    const uint32_t me = cluster_rank();
    const int r = blockIdx.y;
    const int b = a.ic.b;
    const int T = a.max_blocks * b;
    const int C = a.ncand, K = a.tok_k;
    const int CB = (C + CS - 1) / CS;   // candidate positions per CTA
    float *part = reinterpret_cast<float *>(smem + LY::PART);
    float *fs = reinterpret_cast<float *>(smem + LY::FS);
    float *scl = reinterpret_cast<float *>(smem + LY::SC);
    const int2 *cand = reinterpret_cast<const int2 *>(smem + LY::CAND);
    auto ctok = [&](int i) -> int { return cand[i].x; };
    auto csc = [&](int i) -> float { return __int_as_float(cand[i].y); };
    int *ftok = reinterpret_cast<int *>(smem + LY::FTOK);
    int *fpg = reinterpret_cast<int *>(smem + LY::FPG);
    int *cpg = reinterpret_cast<int *>(smem + LY::CPG);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + LY::HIST);
    int *ckt = reinterpret_cast<int *>(smem + LY::CKT);
    double *dx = reinterpret_cast<double *>(smem + LY::DX);

    // ---- prologue (before the scores are final): the query side
    WreluQ Q;
    {
        const bool big = wrelu_load_q(a.q + (int64_t)r * a.hq * 128, a.weights + (int64_t)r * a.hq, Q);
        if (big) flag_error(a.status, LSA_ERR_BOUNDS);
        if (__syncthreads_or(big ? 1 : 0)) wrelu_zero(Q);
    }
    const int L = a.lens[r];
    const bool len_ok = L >= 0 && (int64_t)L <= (int64_t)T;
    const int64_t se = len_ok ? min(a.sink, L) : 0;
    const int64_t rs = len_ok ? max((int64_t)L - a.recent, se) : 0;
    const int nfull = len_ok ? L / b : 0;
    pdl_wait();
    pdl_launch_dependents();

    // ---- A. the CTA's slice of the coarse scores into shared memory (the
    // key region, free until the rescoring): thread t's PT tokens as NCH
    // 16-byte chunks, the chunk index XORed with t mod 8 when NCH allows,
    // so that 8 threads reading their c-th chunks hit distinct banks
    {
        const int S = pq_slice(T, CS), NCH = S / NT / 4;
        const uint32_t sk = smem_addr(smem + LY::KEYS);
        const float *src = a.coarse + (int64_t)r * T + (int64_t)me * S;
        const int valid_chunks = max(0, min(S, T - (int)me * S)) / 4;
        for (int gch = tid; gch < S / 4; gch += NT) {
            const int t = gch / NCH, c = gch - t * NCH;
            const uint32_t sw = (NCH & 7) == 0 ? (uint32_t)(t & 7) : 0u;
            const uint32_t dst = sk + (uint32_t)(((size_t)t * NCH + ((uint32_t)c ^ sw)) * 16);
            if (gch < valid_chunks) cp_async16(dst, src + 4 * gch);
            else
                *reinterpret_cast<float4 *>(smem + (dst - sk) + LY::KEYS) =
                    make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        cp_async_commit();
    }
    // ---- the bucket of the C-th largest coarse score, from the row's counts
    for (int i = tid; i < kPqBins; i += NT) hist[i] = __ldcg(a.hist + (int64_t)r * kPqBins + i);
    float vmin, scale;
    pq_remap(a.row_ext, r, &vmin, &scale);
    cp_async_wait<0>();
    __syncthreads();
    constexpr int BPT = kPqBins / NT;
    const int top = kPqBins - 1 - tid * BPT;
    uint32_t cown = 0;
#pragma unroll
    for (int e = 0; e < BPT; ++e) cown += hist[top - e];
    uint32_t nvalid = 0;
    uint32_t g = bk_scan<NT>(cown, tsm.red, &nvalid);
    const int keff1 = min(C, (int)nvalid);
    if (tid == 0) {
        s_u[0] = 0xffffffffu;   // boundary bucket (none: every candidate is taken)
        s_u[1] = 0u;            // candidates above it
        s_u[2] = 0u;            // candidates in it
    }
    __syncthreads();
    if (keff1 < (int)nvalid && keff1 > 0) {
#pragma unroll
        for (int e = 0; e < BPT; ++e) {
            const uint32_t cb = hist[top - e];
            if (g < (uint32_t)keff1 && (uint32_t)keff1 <= g + cb) {
                s_u[0] = (uint32_t)(top - e);
                s_u[1] = g;
                s_u[2] = cb;
            }
            g += cb;
        }
    }
    __syncthreads();
    const int B1 = (int)s_u[0];   // -1: no boundary
    const int take1 = keff1 - (int)s_u[1];
    const int cnt1 = (int)s_u[2];
    const bool crowded = B1 >= 0 && cnt1 > kBkCap;

    // ---- B. this thread's tokens of this CTA's slice, from shared memory
    // (staged above; thread t owns PT consecutive tokens, NCH chunks of 4)
    const int S = pq_slice(T, CS);
    const int PT = S / NT, NCH = PT / 4;
    const int t_lo = min((int)me * S + tid * PT, T), t_hi = min(t_lo + PT, T);
    const uint32_t swz = (NCH & 7) == 0 ? (uint32_t)(tid & 7) : 0u;
    auto chunk_at = [&](int c) -> float4 {
        return *reinterpret_cast<const float4 *>(smem + LY::KEYS + ((size_t)tid * NCH + ((uint32_t)c ^ swz)) * 16);
    };
    auto key_of = [](float x) -> uint32_t { return (x == -INFINITY || isnan(x)) ? 0u : float_to_key(x); };
    auto bucket_of = [&](uint32_t k) -> int { return pq_bucket(key_to_float(k), vmin, scale); };
    // the bucket of a staged score straight from the float, -1 for one that
    // is not a candidate (-inf or NaN): the same as bucket_of(key_of(x))
    auto cand_bucket = [&](float x) -> int { return x > -INFINITY ? pq_bucket(x, vmin, scale) : -1; };
    const int nch = (t_hi - t_lo + 3) / 4;   // this thread's chunks inside the row

    // the candidate rule, exact in both cases: by bucket (winners above the
    // boundary bucket, the boundary bucket's keys ranked), or, with a
    // crowded boundary bucket, by the threshold key Tk (keys above it, and
    // the first ties in token order)
    uint32_t Tk = 0u;
    int take_eq = 0;
    uint32_t n_a = 0, n_b = 0;   // this thread's winners / boundary keys (or > Tk / == Tk)
    // the positions (4 * chunk + element) of this thread's first kPqList
    // winners and boundary keys, in token order, 8 bits each, so that the
    // candidates' pass below visits only them
    constexpr int kPqList = 8;
    uint64_t clist = 0;
    if (!crowded) {
        for (int c = 0; c < nch; ++c) {
            const float4 v = chunk_at(c);
            const float xs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int bk = cand_bucket(xs[e]);
                const bool w = bk >= 0 && bk > B1, bd = bk >= 0 && bk == B1;
                const uint32_t seen = n_a + n_b;
                if ((w || bd) && seen < (uint32_t)kPqList) clist |= (uint64_t)(4 * c + e) << (8 * seen);
                n_a += w;
                n_b += bd;
            }
        }
    } else {
        // the threshold by bisection over the key space, counts summed over
        // the cluster (two exchange slots alternate)
        uint64_t lo = ~__ldcg(a.row_ext + 2 * r + 1), hi = (uint64_t)__ldcg(a.row_ext + 2 * r) + 1;
        int it = 0;
        while (hi - lo > 1) {
            const uint32_t mid = (uint32_t)(lo + ((hi - lo) >> 1));
            uint32_t c = 0;
            for (int cc = 0; cc < nch; ++cc) {
                const float4 v = chunk_at(cc);
                c += (key_of(v.x) >= mid) + (key_of(v.y) >= mid) + (key_of(v.z) >= mid) + (key_of(v.w) >= mid);
            }
            const uint32_t csum = bk_sum<NT>(c, tsm.red);
            const int slot = 3 + (it & 1);
            if (tid == 0) tsm.xch[slot][0] = csum;
            cluster_sync();
            const int cs = (int)cl_gather_sum<NT, CS>(tsm, slot, 0, nullptr);
            if (cs >= keff1) lo = mid;
            else hi = mid;
            ++it;
            if (cs == keff1) break;
        }
        Tk = (uint32_t)lo;
        for (int c = 0; c < nch; ++c) {
            const float4 v = chunk_at(c);
            const float xs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint32_t k = key_of(xs[e]);
                n_a += k > Tk;
                n_b += k != 0u && k == Tk;
            }
        }
    }
    // per-CTA totals, in thread order
    uint32_t na_cta = 0, nb_cta = 0;
    const uint32_t a_base = bk_scan<NT>(n_a, tsm.red, &na_cta);
    __syncthreads();
    const uint32_t b_base = bk_scan<NT>(n_b, tsm.red, &nb_cta);
    if (!crowded && B1 >= 0 && n_b > 0) {
        // this CTA's boundary keys, in token order
        uint32_t pos = b_base;
        for (int c = 0; c < nch; ++c) {
            const float4 v = chunk_at(c);
            const float xs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (cand_bucket(xs[e]) == B1) {
                    tsm.ck[pos] = key_of(xs[e]);
                    ckt[pos] = t_lo + 4 * c + e;
                    ++pos;
                }
            }
        }
    }
    if (tid == 0) {
        tsm.xch[1][0] = na_cta;
        tsm.xch[1][1] = nb_cta;
    }
    cluster_sync();   // (S1) per-CTA totals and boundary keys are in place
    if (tid < 32) {
        const int lane = tid;
        uint32_t va = 0, vb = 0;
        if (lane < CS) {
            va = ld_cluster_u32(cluster_map(smem_addr(&tsm.xch[1][0]), (uint32_t)lane));
            vb = ld_cluster_u32(cluster_map(smem_addr(&tsm.xch[1][1]), (uint32_t)lane));
        }
        uint32_t ia = va, ib = vb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t ya = __shfl_up_sync(0xffffffffu, ia, o), yb = __shfl_up_sync(0xffffffffu, ib, o);
            if (lane >= o) {
                ia += ya;
                ib += yb;
            }
        }
        const uint32_t ta = __shfl_sync(0xffffffffu, ia, 31), tb = __shfl_sync(0xffffffffu, ib, 31);
        if (lane < CS) {
            s_off[0][lane] = ia - va;
            s_off[1][lane] = ib - vb;
        }
        if (lane == 0) {
            s_off[0][CS] = ta;
            s_off[1][CS] = tb;
        }
    }
    __syncthreads();

    // which of the boundary keys are taken: pick[i] over the cluster's list
    // (bucket rule), or the threshold's first take_eq ties
    if (crowded) {
        take_eq = keff1 - (int)s_off[0][CS];
    } else if (B1 >= 0) {
        const int cnt = (int)s_off[1][CS];   // == cnt1
        for (int gi = tid; gi < cnt; gi += NT) {
            int owner = 0;
#pragma unroll
            for (int c = 1; c < CS; ++c) owner += (uint32_t)gi >= s_off[1][c];
            tsm.ckall[gi] = ld_cluster_u32(cluster_map(smem_addr(&tsm.ck[gi - (int)s_off[1][owner]]), (uint32_t)owner));
        }
        __syncthreads();
        for (int gi = tid; gi < cnt; gi += NT) {
            const uint32_t mine = tsm.ckall[gi];
            int rank = 0;
            for (int j = 0; j < cnt; ++j) {
                const uint32_t y = tsm.ckall[j];
                rank += (y > mine) || (y == mine && j < gi);
            }
            tsm.pick[gi] = rank < take1 ? 1 : 0;
        }
        __syncthreads();
    }
    // candidates of the CTAs before this one: their winners and their taken
    // boundary keys (every CTA counts every CTA's)
    if (tid < 32) {
        const int lane = tid;
        uint32_t taken = 0;
        if (lane < CS) {
            if (crowded) {
                const int e0 = (int)s_off[1][lane], e1 = (int)s_off[1][lane + 1];
                taken = (uint32_t)max(0, min(e1, take_eq) - e0);
            } else if (B1 >= 0) {
                for (int i = (int)s_off[1][lane]; i < (int)s_off[1][lane + 1]; ++i) taken += tsm.pick[i];
            }
        }
        const uint32_t v = lane < CS ? (uint32_t)(s_off[0][lane + 1] - s_off[0][lane]) + taken : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == (int)me) s_u[3] = incl - v;
    }
    __syncthreads();
    const uint32_t cbase = s_u[3];

    // ---- C. this thread's candidates to their owners, in token order
    {
        // this thread's candidates before its own: winners, then taken
        // boundary keys, counted in thread order
        uint32_t mine = n_a;
        uint32_t bpos = s_off[1][me] + b_base;   // this thread's first boundary key in the cluster's list
        if (crowded) {
            const int e0 = (int)bpos, e1 = e0 + (int)n_b;
            mine += (uint32_t)max(0, min(e1, take_eq) - e0);
        } else if (B1 >= 0) {
            for (uint32_t i = 0; i < n_b; ++i) mine += tsm.pick[bpos + i];
        }
        uint32_t dummy = 0;
        __syncthreads();
        uint32_t pos = cbase + bk_scan<NT>(mine, tsm.red, &dummy);
        int32_t *cout = a.cand_out ? a.cand_out + (int64_t)r * C : nullptr;
        // the candidate at position q (4 * chunk + element) of this thread's
        // slice: taken or not, then to its owner (and to cand_out)
        auto emit = [&](int q, float x, bool take) {
            if (!take) return;
            const int i = t_lo + q;
            const int owner = (int)pos / CB, slot = (int)pos - owner * CB;
            // the score as its key maps it back (-0 as +0)
            const uint32_t xb = __float_as_uint(x) == 0x80000000u ? 0u : __float_as_uint(x);
            st_cluster_v2_u32(cluster_map(smem_addr(&cand[slot]), (uint32_t)owner), (uint32_t)i, xb);
            if (cout) cout[pos] = i;
            ++pos;
        };
        const bool listed = !crowded && n_a + n_b <= (uint32_t)kPqList;
        if (listed) {
            for (int n = 0; n < (int)(n_a + n_b); ++n) {
                const int q = (int)((clist >> (8 * n)) & 0xffu);
                const float x = reinterpret_cast<const float *>(smem + LY::KEYS + ((size_t)tid * NCH +
                                                                                   ((uint32_t)(q >> 2) ^ swz)) * 16)[q & 3];
                const int bk = cand_bucket(x);
                bool take = bk > B1;
                if (bk == B1) {
                    take = tsm.pick[bpos] != 0;
                    ++bpos;
                }
                emit(q, x, take);
            }
        }
        for (int c = 0; !listed && c < nch && (n_a + n_b) > 0; ++c) {
            const float4 v = chunk_at(c);
            const float xs[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x = xs[e];
                bool take;
                if (crowded) {
                    const uint32_t k = key_of(x);
                    if (k == 0u) continue;
                    if (k > Tk) take = true;
                    else if (k == Tk) {
                        take = (int)bpos < take_eq;
                        ++bpos;
                    } else take = false;
                } else {
                    const int bk = cand_bucket(x);
                    if (bk < 0) continue;   // not a candidate
                    if (bk > B1) take = true;
                    else if (bk == B1) {
                        take = tsm.pick[bpos] != 0;
                        ++bpos;
                    } else take = false;
                }
                emit(4 * c + e, x, take);
            }
        }
        if (cout && me == 0)
            for (int i = keff1 + tid; i < C; i += NT) cout[i] = -1;
    }
    cluster_sync();   // (S2) every CTA's candidates are in place

    // ---- D. the miss filter (hits kept; misses below the k-th largest
    // coarse score minus one sample standard deviation dropped)
    const int ncb = min(CB, max(0, keff1 - (int)me * CB));   // this CTA's candidates
    // pages of this CTA's candidates
    for (int i = tid; i < ncb; i += NT) {
        const int t = ctok(i);
        const int p = a.pt[(int64_t)r * a.max_blocks + t / b];
        const bool pok = p >= 0 && p < a.ic.num_pages;
        if (!pok) flag_error(a.status, LSA_ERR_BOUNDS);
        cpg[i] = pok ? p : -1;
    }
    __syncthreads();
    double tau = -INFINITY;
    if (keff1 > K) {
        // the k-th largest: the smallest key of a top-k of the candidates
        uint32_t keys[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int i = 2 * tid + e;
            keys[e] = i < ncb ? float_to_key(csc(i)) : 0u;
        }
        uint32_t kmin = 0xffffffffu;
        const int col0 = (int)me * kFtTok + 2 * tid;
        cluster_bucket_topk<NT, 2, CS>(keys, K, col0, tsm, [&](int, int col) { kmin = min(kmin, keys[col - col0]); });
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        if ((tid & 31) == 0) tsm.red[tid >> 5][0] = kmin;
        __syncthreads();
        // the sample standard deviation of the candidates' coarse scores:
        // the mean, then the sum of squared deviations, in fp64, each summed
        // in a fixed order (lanes, warps, then the cluster's CTAs in rank
        // order).  The CTA's sum of scores goes out with its smallest key of
        // the top k, in one exchange; each exchange has its own slots, so
        // none waits for the slots to be read
        double loc = 0.0;
        for (int i = tid; i < ncb; i += NT) loc += (double)csc(i);
        const double sx = pq_block_dsum(loc, dx + 5);
        if (tid == 0) {
            uint32_t m = 0xffffffffu;
            for (int w = 0; w < NT / 32; ++w) m = min(m, tsm.red[w][0]);
            tsm.xch[7][0] = ~m;
            dx[0] = sx;
        }
        cluster_sync();
        if (tid < 32) {
            uint32_t v = tid < CS ? ld_cluster_u32(cluster_map(smem_addr(&tsm.xch[7][0]), (uint32_t)tid)) : 0u;
            v = __reduce_max_sync(0xffffffffu, v);
            const double x = tid < CS ? ld_cluster_f64(cluster_map(smem_addr(&dx[0]), (uint32_t)tid)) : 0.0;
            double t = 0.0;
#pragma unroll
            for (int c = 0; c < CS; ++c) t += __shfl_sync(0xffffffffu, x, c);
            if (tid == 0) {
                s_u[4] = ~v;
                dx[1] = t / (double)keff1;   // the mean, divided once
            }
        }
        __syncthreads();
        const double sk = (double)key_to_float(s_u[4]);
        const double mean = dx[1];
        loc = 0.0;
        for (int i = tid; i < ncb; i += NT) {
            const double d = (double)csc(i) - mean;
            loc += d * d;
        }
        const double sq = pq_block_dsum(loc, dx + 5);
        if (tid == 0) dx[2] = sq;
        cluster_sync();
        if (tid < 32) {
            const double x = tid < CS ? ld_cluster_f64(cluster_map(smem_addr(&dx[2]), (uint32_t)tid)) : 0.0;
            double t = 0.0;
#pragma unroll
            for (int c = 0; c < CS; ++c) t += __shfl_sync(0xffffffffu, x, c);
            if (tid == 0) dx[3] = t;
        }
        if (tid == 0) dx[4] = sk - sqrt(dx[3] / (double)(keff1 - 1));
        __syncthreads();
        tau = dx[4];
    }

    // ---- E. the tokens this CTA rescores: its kept candidates in order,
    // then (the last CTA) the unencoded tail outside the forced ranges
    int nf = 0;
    for (int base = 0; base < ncb; base += NT) {
        const int i = base + tid;
        bool keep = false;
        if (i < ncb) {
            const int t = ctok(i), p = cpg[i];
            const bool hit = !a.hit || (p >= 0 && a.hit[(int64_t)p * b + t % b] != 0);
            keep = p >= 0 && (hit || (double)csc(i) >= tau);
        }
        uint32_t tot = 0;
        const uint32_t at = bk_scan<NT>(keep ? 1u : 0u, tsm.red, &tot);
        if (keep) {
            ftok[nf + (int)at] = ctok(i);
            fpg[nf + (int)at] = cpg[i];
        }
        nf += (int)tot;
        __syncthreads();
    }
    if (me == CS - 1) {
        const int t0 = nfull * b;
        for (int t = t0 + tid; t < L; t += NT) {
            const int j = nf + (t - t0);
            const bool in = t >= se && t < rs;
            const int p = a.pt[(int64_t)r * a.max_blocks + t / b];
            ftok[j] = in ? t : -1;
            fpg[j] = (in && p >= 0 && p < a.ic.num_pages) ? p : -1;
        }
        nf += max(0, L - t0);
    }
    __syncthreads();

    // ---- F. exact weighted-ReLU scores of those tokens
    {
        const uint32_t kbase = smem_addr(smem + LY::KEYS);
        for (int task = tid; task < nf * 8; task += NT) {
            const int j = task >> 3, u = task & 7;
            const int p = fpg[j], t = ftok[j];
            if (p >= 0 && t >= 0)
                cp_async16(kbase + cf_key_off(j, u), a.ic.k + (int64_t)p * a.ic.kps + (int64_t)(t % b) * a.ic.kts + u * 16);
            else
                *reinterpret_cast<uint4 *>(smem + LY::KEYS + cf_key_off(j, u)) = make_uint4(0u, 0u, 0u, 0u);
        }
        cp_async_commit();
        for (int j = tid; j < nf; j += NT) {
            const int p = fpg[j], t = ftok[j];
            scl[j] = (p >= 0 && t >= 0) ? a.ic.kscale[(int64_t)p * a.ic.sps + t % b] : 0.f;
        }
        cp_async_wait<0>();
        __syncthreads();
        wrelu_tile_partials(kbase, nf, Q, part);
        __syncthreads();
        for (int j = tid; j < nf; j += NT)
            fs[j] = (fpg[j] >= 0 && ftok[j] >= 0) ? scl[j] * wrelu_combine(part, j) : -INFINITY;
        __syncthreads();
    }

    // ---- G. the top k tokens over the cluster
    {
        uint32_t keys[2];
        bool nan = false;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int j = 2 * tid + e;
            const float x = j < nf ? fs[j] : -INFINITY;
            nan |= isnan(x);
            keys[e] = (isnan(x) || x == -INFINITY) ? 0u : float_to_key(x);
        }
        if (nan) flag_error(a.status, LSA_ERR_NAN);
        int32_t *orow = a.tok_idx + (int64_t)r * K;
        const int col0 = (int)me * kFtTok + 2 * tid;
        const int keff = cluster_bucket_topk<NT, 2, CS>(keys, K, col0, tsm, [&](int pos, int col) {
            orow[pos] = ftok[col - (int)me * kFtTok];
        });
        if (me == 0)
            for (int i = keff + tid; i < K; i += NT) orow[i] = -1;
    }
    // every CTA read the row's counts and extremes before the first cluster
    // barrier: reset them for the next call (here, where no cluster barrier's
    // release waits for these stores)
    if (me == 0) {
        for (int i = tid; i < kPqBins; i += NT) a.hist[(int64_t)r * kPqBins + i] = 0u;
        if (tid == 0) {
            a.row_ext[2 * r] = 0u;
            a.row_ext[2 * r + 1] = 0u;
        }
    }
}

template <int CS>
cudaError_t launch_pq_select_t(const PqArgs &a, cudaStream_t s)
{
    auto kern = k_pq_select<CS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PqSelLayout::SMEM);
    if (e != cudaSuccess) return e;
    if (CS > 8 && (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
        return e;
    e = launch_cluster_kernel(pdl_step_dependent(), CS, kern, dim3(CS, a.batch), dim3(kFtThreads),
                              (size_t)PqSelLayout::SMEM, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int pq_cluster_size()
{
    static std::mutex mu;
    static int cs[64] = {};
    static bool done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!done[dev]) {
        int c = 0;
        if (max_active_clusters(k_pq_select<16>, 16, dim3(kFtThreads), PqSelLayout::SMEM) > 0) c = 16;
        else if (max_active_clusters(k_pq_select<8>, 8, dim3(kFtThreads), PqSelLayout::SMEM) > 0) c = 8;
        cs[dev] = c;
        done[dev] = true;
    }
    return cs[dev];
}

}  // namespace

bool pq_supported(const CacheView &iv, int hq, int max_blocks, int ncand, int tok_k)
{
    if (!(iv.e4m3 && iv.dk == 128 && iv.hkv == 1 && iv.b >= 16 && iv.b <= 64 && iv.b % 16 == 0 && hq == 64))
        return false;
    if (ncand <= 0 || tok_k <= 0) return false;
    if ((iv.kts & 15) || (iv.kps & 15) || (reinterpret_cast<uintptr_t>(iv.k) & 15)) return false;
    const int cs = pq_cluster_size();
    if (cs == 0) return false;
    const int cb = (ncand + cs - 1) / cs;
    // a CTA's slice of the coarse scores fits the key region (128 KB)
    return cb + iv.b <= kFtTok && tok_k <= cs * kFtTok && iv.b % 4 == 0 &&
           (int64_t)max_blocks * iv.b <= (int64_t)cs * kFtTok * 32 &&
           pq_slice(max_blocks * iv.b, cs) * 4 <= kFtTok * 128;
}

cudaError_t launch_pq_encode(const PqArgs &a, cudaStream_t s)
{
    if (a.batch == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(k_pq_encode, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeSmem);
    if (e != cudaSuccess) return e;
    e = launch_step_kernel(k_pq_encode, dim3(min(a.max_blocks, 64), a.batch), dim3(kPeThreads), (size_t)kPeSmem, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_pq_scores(const PqArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = !(a.ic.dk == 128 && a.ic.hkv == 1 && a.hq == 64 && a.ic.b % 16 == 0);
    if (*unsupported || a.batch == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(k_pq_scores, cudaFuncAttributeMaxDynamicSharedMemorySize, PsLayout::SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles = (int64_t)a.batch * ((a.max_blocks * a.ic.b + kPsTok - 1) / kPsTok);
    const int grid = (int)std::min<int64_t>(tiles, (int64_t)kPsCtasPerSm * sms);
    PqArgs ka = a;
    ka.fd_b = make_fastdiv((uint32_t)a.ic.b);
    ka.fd_tpr = make_fastdiv((uint32_t)((a.max_blocks * a.ic.b + kPsTok - 1) / kPsTok));
    e = launch_step_kernel(k_pq_scores, dim3(grid), dim3(kPsThreads), (size_t)PsLayout::SMEM, s, ka);
    if (e != cudaSuccess) return e;
    if (!a.hist) return cudaGetLastError();   // scores only
    const int T = a.max_blocks * a.ic.b;
    e = launch_kernel_ex(pdl_step_dependent(), k_pq_hist, dim3((T + kPhTok - 1) / kPhTok, a.batch), dim3(kPhThreads),
                         0, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_pq_select(const PqArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = !pq_supported(a.ic, a.hq, a.max_blocks, a.ncand, a.tok_k);
    if (*unsupported || a.batch == 0) return cudaSuccess;
    return pq_cluster_size() == 16 ? launch_pq_select_t<16>(a, s) : launch_pq_select_t<8>(a, s);
}

}  // namespace lsa

// Sparse attention with an even split of the whole batch's work over the
// GPU (tensor cores, GQA groups of 2..8 query heads, d = 64 or 128).
//
// The attended token set of every row (request, KV head, query subgroup) is
// walked in 16-token items: forced sink tokens, the selected blocks, forced
// recent tokens (Vortex blog post, block top-k equation; ByteCross, Appendix
// A).  Every row gets the same number NS of item slots (empty slots stream
// nothing), so item i belongs to row i / NS, and the flat list of all rows'
// items is cut into equal contiguous pieces: CTA c takes the items i with
// floor(i * NC / T) == c, and its warps take equal contiguous parts of
// those.  Every SM thus streams the same number of bytes whatever the
// lengths and the selection, and a piece touches at most two rows.
//
// Each warp resolves all its items' descriptors at once (request length and
// selection in one round trip, page ids in a second), then streams K and V
// through its own ring of cp.async stages into 128-byte XOR-swizzled tiles
// for ldmatrix, and runs the group's S = Q K^T and O += P V as m16n8k16
// MMAs (the G heads in rows 0..G-1) with an online softmax.  At the end the
// CTA merges its warps' partial results per row in shared memory; a row
// that several CTAs share is merged by log-sum-exp (ByteCross, Appendix A)
// by the last of them to finish, found with a per-row counter that it
// resets for the next call.
#include <math.h>

#include "attn_items.cuh"
#include "attn_stage.cuh"
#include "lsa_device.cuh"
#include "topk_block.cuh"
#include "topk_bucket.cuh"

namespace lsa {
namespace {

constexpr int kFlWarps = 8;
constexpr int kFlCtasPerSm = 1;
constexpr int kFlMaxRowsPerCta = 2;   // the host keeps a CTA's piece within two rows
constexpr int kFlMaxItemsPerWarp = 32;
constexpr int kFlMaxSel = 512;        // blocks a CTA selects per row when it selects them itself
constexpr float kFlLn2 = 0.693147180559945309f;

template <int DK, int G>
struct FlLayout {
    static constexpr int STAGES = G <= 4 ? 3 : 2;   // one CTA of eight warps per SM
    static constexpr int SUB = kChunk * 128;      // one swizzled 16-row x 128-byte sub-tile
    static constexpr int KBYTES = (DK / 64) * SUB;
    static constexpr int STAGE = 2 * KBYTES;      // K tile then V tile
    static constexpr int WARP_RING = STAGES * STAGE;
    static constexpr int RINGS = kFlWarps * WARP_RING;
    static constexpr int SEG0 = RINGS + kFlWarps * 16;            // first-row results: [W][G][DK], m, l
    static constexpr int LAST = SEG0 + kFlWarps * G * (DK + 2) * 4;   // per-row "last CTA" flags
    static constexpr int SELBUF = LAST + 16;                          // top-k scratch, then [2][kFlMaxSel] selection
    static constexpr int SELS = SELBUF + ((int)sizeof(TopkScratch) + 15) / 16 * 16;
    static constexpr int SMEM = SELS + 2 * kFlMaxSel * 4;
    static_assert(RINGS >= kFlMaxRowsPerCta * (kFlWarps * G * (DK + 2) + G * (kFlWarps + 1)) * 4,
                  "the CTA merge reuses the rings");
    static_assert(RINGS >= (int)sizeof(BucketScratch<kFlWarps * 32>), "the selection's scratch reuses the rings");
    static_assert(SMEM * kFlCtasPerSm <= 227 * 1024, "the CTAs of one SM");
};

// Row index -> (request, KV head, query subgroup).
struct FlRow {
    int r, h, sg;
};

__device__ __forceinline__ FlRow fl_row(const AttnArgs &a, int rho)
{
    FlRow x;
    const uint32_t rh = fdiv((uint32_t)rho, a.fd_nsub);
    x.sg = rho - (int)(rh * a.fd_nsub.d);
    x.r = (int)fdiv(rh, a.fd_hkv);
    x.h = (int)rh - x.r * (int)a.fd_hkv.d;
    return x;
}

// First CTA whose piece holds item i (i * fl_ctas < 2^32: host-checked).
__device__ __forceinline__ int fl_cta_of(const AttnArgs &a, uint32_t i)
{
    return (int)fdiv(i * (uint32_t)a.fl_ctas, a.fd_total);
}

// KSEL > 0: the CTA selects its rows' blocks itself from the score rows
// (block_topk with KSEL keys per thread) instead of reading a selection.
template <int DK, int G, int KSEL>
__global__ void __launch_bounds__(kFlWarps * 32, 1) k_attn_flat(AttnArgs a)
{
    const bool early = a.pdl_early != 0;
    if (!early) pdl_wait();
    pdl_launch_dependents();
    using LY = FlLayout<DK, G>;
    static_assert(KSEL == 0 || kFlWarps * 32 == kTfThreads, "one CTA is one top-k block");
    constexpr int NT = DK / 8;
    constexpr int kFlStages = LY::STAGES;
    static_assert(G >= 2 && G <= 8, "heads of a group must fit rows 0..7 of the MMA tile");

    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Gt = a.gsize;
    const CacheView &c = a.c;
    if ((smem_addr(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) flag_error(a.status, LSA_ERR_INVALID_ARG);
        return;
    }
    // index arithmetic in 32 bits: the host keeps (T + 1) * fl_ctas < 2^32
    const uint32_t NS = (uint32_t)a.fl_ns, NC = (uint32_t)a.fl_ctas;
    const uint32_t T = (uint32_t)a.fl_total;
    const uint32_t cta = blockIdx.x;
    const uint32_t cs = fdiv(cta * T + NC - 1, a.fd_nc);   // this CTA's items [cs, ce)
    const uint32_t ce = fdiv((cta + 1) * T + NC - 1, a.fd_nc);
    const uint32_t cn = ce - cs;
    const uint32_t ws = cs + cn * warp / kFlWarps, we = cs + cn * (warp + 1) / kFlWarps;
    const int nmine = min((int)(we - ws), kFlMaxItemsPerWarp);   // the host keeps pieces within this
    const int rho_first = (int)fdiv(cs, a.fd_ns);
    const int rh_first = (int)fdiv((uint32_t)rho_first, a.fd_nsub);
    const int rh_last = cn > 0 ? (int)fdiv(fdiv(ce - 1, a.fd_ns), a.fd_nsub) : rh_first - 1;   // none when empty

    uint8_t *ring = smem + warp * LY::WARP_RING;
    const uint32_t ring_s = smem_addr(ring);
    int *stage_n = reinterpret_cast<int *>(smem + kFlWarps * LY::WARP_RING) + warp * 4;

    const int rr = lane >> 2, cc = lane & 3;

    // ---- descriptors of this warp's items, one per lane: the request
    // length and the query fragments of the warp's rows are loaded first
    // (while the CTA selects, when it does), then the selection entries
    // (read assuming the sink takes its full number of items, re-read in
    // the rare case it does not), then the page ids
    ItemDesc my{-1, 0, 0};
    int my_rho = -1, my_k = 0, my_L = 0;
    int2 my_sel = make_int2(-1, -1);
    const int nsc_full = (a.sink + kChunk - 1) / kChunk;
    if (lane < nmine) {
        const uint32_t i = ws + lane;
        my_rho = (int)fdiv(i, a.fd_ns);
        my_k = (int)(i - (uint32_t)my_rho * NS);
        my_L = a.lens[fl_row(a, my_rho).r];
    }
    const int rho_w0 = nmine > 0 ? (int)fdiv(ws, a.fd_ns) : -1;
    const int rho_w1 = nmine > 0 ? (int)fdiv(ws + nmine - 1, a.fd_ns) : -1;
    uint32_t qa0[DK / 16], qa2[DK / 16], qb0[DK / 16], qb2[DK / 16];
    auto load_q = [&](int rho, uint32_t (&q0)[DK / 16], uint32_t (&q2)[DK / 16]) {
        const FlRow x = fl_row(a, rho < 0 ? 0 : rho);
        const bool qrow = rr < G && rho >= 0;
        const uint16_t *qp = a.q + ((int64_t)x.r * a.hq + x.h * Gt + x.sg * G + (qrow ? rr : 0)) * DK;
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks) {
            q0[ks] = qrow ? *reinterpret_cast<const uint32_t *>(qp + 16 * ks + 2 * cc) : 0u;
            q2[ks] = qrow ? *reinterpret_cast<const uint32_t *>(qp + 16 * ks + 8 + 2 * cc) : 0u;
        }
    };
    load_q(rho_w0, qa0, qa2);
    load_q(rho_w1 != rho_w0 ? rho_w1 : -1, qb0, qb2);

    // the page-table rows of the piece's requests (at most two, adjacent)
    // into L1 while the CTA selects: the item descriptors read them after
    // the selection.  One prefetch per 128-byte line, at most 32 KB.
    if (KSEL > 0 && cn > 0) {
        const int rq0 = (int)fdiv((uint32_t)rh_first, a.fd_hkv), rq1 = (int)fdiv((uint32_t)rh_last, a.fd_hkv);
        const char *p0 = reinterpret_cast<const char *>(a.pt + (int64_t)rq0 * a.max_blocks);
        const int64_t bytes = (int64_t)(rq1 - rq0 + 1) * a.max_blocks * 4;
        const int lines = (bytes + 127) / 128 < 256 ? (int)((bytes + 127) / 128) : 256;
        if ((int)threadIdx.x < lines) prefetch_l1(p0 + 128 * (int64_t)threadIdx.x);
    }

    // (early launch) the score rows come from the kernel before: wait for
    // it here, then load the first row's scores
    if (early) pdl_wait();
    constexpr int KV = KSEL > 0 ? KSEL : 4;
    float sel_v[KV];
    const bool sel_aligned = (a.sel_cols & 3) == 0 && (reinterpret_cast<uintptr_t>(a.sel_scores) & 15) == 0;
    if constexpr (KSEL > 0) {
        if (rh_first <= rh_last)
            block_topk_load<KSEL>(a.sel_scores + (int64_t)rh_first * a.sel_cols, a.sel_cols, sel_aligned, sel_v);
    }

    // ---- the selection of the (request, KV head) rows of this piece (at
    // most two), when this kernel makes it: exact top-k of each score row,
    // written out by the CTA that holds the row's first item
    int32_t *s_sel = reinterpret_cast<int32_t *>(smem + LY::SELS);   // [2][kFlMaxSel]
    if constexpr (KSEL > 0) {
        TopkScratch &sm = *reinterpret_cast<TopkScratch *>(smem + LY::SELBUF);
        for (int s = 0; s < 2 && rh_first + s <= rh_last; ++s) {
            const int rh = rh_first + s;
            int32_t *dst = s_sel + s * kFlMaxSel;
            if (s > 0) block_topk_load<KSEL>(a.sel_scores + (int64_t)rh * a.sel_cols, a.sel_cols, sel_aligned, sel_v);
            int keff;
            if constexpr (KSEL == 8) {
                // rows of up to 2048 blocks: the bucketed exact top-k
                // (topk_bucket.cuh), its scratch in the K / V rings, which
                // are not in use before the selection is made
                BucketScratch<kFlWarps * 32> &bsm = *reinterpret_cast<BucketScratch<kFlWarps * 32> *>(smem);
                uint32_t keys[KSEL];
                bool nan = false;
#pragma unroll
                for (int e = 0; e < KSEL; ++e) {
                    nan |= isnan(sel_v[e]);
                    keys[e] = (isnan(sel_v[e]) || sel_v[e] == -INFINITY) ? 0u : float_to_key(sel_v[e]);
                }
                if (nan) flag_error(a.status, LSA_ERR_NAN);
                keff = block_bucket_topk<kFlWarps * 32, KSEL>(keys, a.nsel, bsm, [&](int pos, int col) { dst[pos] = col; });
            } else {
                keff = block_topk_scores<KSEL>(sel_v, a.nsel, a.status, sm, [&](int pos, int col) { dst[pos] = col; });
            }
            for (int i = keff + (int)threadIdx.x; i < a.nsel; i += blockDim.x) dst[i] = -1;
            __syncthreads();
            if (a.sel_write && fl_cta_of(a, (uint32_t)rh * a.nsub * NS) == (int)cta)
                for (int i = threadIdx.x; i < a.nsel; i += blockDim.x) a.sel_write[(int64_t)rh * a.nsel + i] = dst[i];
        }
    }
    // selection entries (entry, the one before it) of item k of this lane's
    // row under a plan whose sink takes nsc items
    auto sel_entries = [&](int rho, int r, int h, int nsc, int k) -> int2 {
        if constexpr (KSEL > 0) {
            const int kk = k - nsc, cpb = (int)a.fd_cpb.d;
            if (kk < 0 || kk >= a.nsel * cpb) return make_int2(-1, -1);
            const int ei = (int)fdiv((uint32_t)kk, a.fd_cpb);
            const int32_t *srow = s_sel + ((int)fdiv((uint32_t)rho, a.fd_nsub) - rh_first) * kFlMaxSel;
            return make_int2(srow[ei], ei > 0 ? srow[ei - 1] : -1);
        } else {
            return item_sel_entries(a, r, h, nsc, k);
        }
    };

    if (lane < nmine) {
        const FlRow x = fl_row(a, my_rho);
        my_sel = sel_entries(my_rho, x.r, x.h, nsc_full, my_k);
        const RowPlan pl = plan_of_len(a, my_L, my_k == 0 && x.h == 0 && x.sg == 0);
        if (pl.nsc != nsc_full) my_sel = sel_entries(my_rho, x.r, x.h, pl.nsc, my_k);
        my = my_k < pl.n_items ? describe_item_sel(a, pl, x.r, x.h, my_k, my_sel) : ItemDesc{-1, 0, 0};
    }

    const uint64_t pol = l2_evict_first();
    auto issue = [&](int j) {
        if (j >= nmine) {
            cp_async_commit();
            return;
        }
        const int page = __shfl_sync(0xffffffffu, my.page, j);
        const int ts = __shfl_sync(0xffffffffu, (int)my.ts, j);
        const int n = __shfl_sync(0xffffffffu, (int)my.n, j);
        const int rho = __shfl_sync(0xffffffffu, my_rho, j);
        if (lane == 0) stage_n[j % kFlStages] = n;
        if (n > 0) {
            const int h = (int)fmodu(fdiv((uint32_t)rho, a.fd_nsub), a.fd_hkv);
            const uint8_t *kb = c.k + ((int64_t)page * c.kps + (int64_t)h * c.khs + (int64_t)ts * c.kts) * 2;
            const uint8_t *vb = c.v + ((int64_t)page * c.vps + (int64_t)h * c.vhs + (int64_t)ts * c.vts) * 2;
            stage_item_kv<DK>(ring_s + (j % kFlStages) * LY::STAGE, kb, vb, c.kts, c.vts, n, pol);
        }
        cp_async_commit();
    };

    // the current row segment's state lives in registers; a segment of the
    // piece's first row that ends mid-stream is parked in shared memory
    GroupState<DK> gs;
    group_state_reset(gs);
    float *s0o = reinterpret_cast<float *>(smem + LY::SEG0) + warp * G * DK;   // [G][DK]
    float *s0m = reinterpret_cast<float *>(smem + LY::SEG0) + kFlWarps * G * DK + warp * 2 * G;   // m[G], l[G]
    if (lane < G) {
        s0m[lane] = -INFINITY;
        s0m[G + lane] = 0.f;
    }
    int cur_rho = -1;

    auto write_state = [&](float *dst_o, float *dst_ml) {
        if (rr < G) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                *reinterpret_cast<float2 *>(dst_o + rr * DK + nt * 8 + 2 * cc) = make_float2(gs.o[nt][0], gs.o[nt][1]);
            if (cc == 0) {
                dst_ml[rr] = gs.m;
                dst_ml[G + rr] = gs.l;
            }
        }
    };
    auto close_segment = [&]() {   // only the piece's first row can end mid-stream
        if (cur_rho == rho_first) write_state(s0o, s0m);
    };
    auto open_segment = [&](int rho) {
        cur_rho = rho;
        group_state_reset(gs);
        if (rho != rho_w0) {   // the warp's second row: its query fragments were loaded up front
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks) {
                qa0[ks] = qb0[ks];
                qa2[ks] = qb2[ks];
            }
        }
    };

#pragma unroll
    for (int j = 0; j < kFlStages - 1; ++j) issue(j);
    for (int j = 0; j < nmine; ++j) {
        issue(j + kFlStages - 1);
        const int rho = __shfl_sync(0xffffffffu, my_rho, j);
        if (rho != cur_rho) {
            close_segment();
            open_segment(rho);
        }
        cp_async_wait<kFlStages - 1>();
        __syncwarp();
        const int n = stage_n[j % kFlStages];
        if (n > 0)
            attend_staged_item<DK>(ring_s + (j % kFlStages) * LY::STAGE, ring + (j % kFlStages) * LY::STAGE, n, qa0,
                                   qa2, a.scale_log2, gs);
        __syncwarp();
    }
    cp_async_wait<0>();
    __syncthreads();   // rings drained: reuse them for the CTA merge

    // ---- CTA merge: per row of the piece, combine the warps' segments.
    // Merge area (in the rings): o [rows][W][G][DK], (m, l) [rows][W][2G],
    // then the warps' weights [rows][G][W] and the log2-sum-exp [rows][G].
    float *mo = reinterpret_cast<float *>(smem);
    float *mml = mo + kFlMaxRowsPerCta * kFlWarps * G * DK;
    float *mcoef = mml + kFlMaxRowsPerCta * kFlWarps * 2 * G;
    float *mlse = mcoef + kFlMaxRowsPerCta * G * kFlWarps;
    {
        // slot 0: the parked first-row segment when the warp went on to the
        // second row, else the current one; slot 1: the current one then
        const int cur_s = cur_rho < 0 ? -1 : cur_rho - rho_first;   // -1, 0 or 1 (host-guaranteed); warp-uniform
        if (cur_s == 1) {
            for (int t = lane; t < G * DK; t += 32) mo[(0 * kFlWarps + warp) * G * DK + t] = s0o[t];
            if (lane < 2 * G) mml[(0 * kFlWarps + warp) * 2 * G + lane] = s0m[lane];
        } else if (lane < 2 * G) {
            mml[(1 * kFlWarps + warp) * 2 * G + lane] = lane < G ? -INFINITY : 0.f;
            if (cur_s < 0) mml[(0 * kFlWarps + warp) * 2 * G + lane] = lane < G ? -INFINITY : 0.f;
        }
        __syncwarp();
        if (cur_s >= 0)
            write_state(mo + (cur_s * kFlWarps + warp) * G * DK, mml + (cur_s * kFlWarps + warp) * 2 * G);
    }
    __syncthreads();
    // per (row, head): the warps' weights exp2(m_w - M) / sum_w exp2(m_w - M)
    // l_w and the log2-sum-exp, once, by kFlWarps consecutive lanes each
    for (int t = threadIdx.x; t < kFlMaxRowsPerCta * G * kFlWarps; t += blockDim.x) {
        const int sl = t / (G * kFlWarps), g = (t / kFlWarps) % G, w = t % kFlWarps;
        const float mw = mml[(sl * kFlWarps + w) * 2 * G + g];
        const float lw = mml[(sl * kFlWarps + w) * 2 * G + G + g];
        float M = mw;
#pragma unroll
        for (int off = 1; off < kFlWarps; off <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float f = mw == -INFINITY ? 0.f : fast_ex2(mw - M);
        float wsum = f * lw;
#pragma unroll
        for (int off = 1; off < kFlWarps; off <<= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
        const bool empty_set = !(wsum > 0.f);
        mcoef[(sl * G + g) * kFlWarps + w] = empty_set ? 0.f : f / wsum;
        if (w == 0) mlse[sl * G + g] = empty_set ? -INFINITY : M + fast_lg2(wsum);
    }
    __syncthreads();

    const int rho_last = cn > 0 ? (int)fdiv(ce - 1, a.fd_ns) : rho_first - 1;
    int *s_last = reinterpret_cast<int *>(smem + LY::LAST);
    for (int s = 0; s < kFlMaxRowsPerCta && rho_first + s <= rho_last; ++s) {
        const int rho = rho_first + s;
        const FlRow x = fl_row(a, rho);
        const int fc = fl_cta_of(a, (uint32_t)rho * NS);
        const int lc = fl_cta_of(a, (uint32_t)(rho + 1) * NS - 1);
        const int parts = lc - fc + 1;
        for (int t = threadIdx.x; t < G * DK / 2; t += blockDim.x) {
            const int g = t / (DK / 2), d = (t % (DK / 2)) * 2;
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kFlWarps; ++w) {
                // a warp with nothing in this row has weight 0 and an unwritten slot
                const float cw = mcoef[(s * G + g) * kFlWarps + w];
                const float2 v = *reinterpret_cast<const float2 *>(mo + ((s * kFlWarps + w) * G + g) * DK + d);
                acc.x = cw != 0.f ? fmaf(cw, v.x, acc.x) : acc.x;
                acc.y = cw != 0.f ? fmaf(cw, v.y, acc.y) : acc.y;
            }
            const float lse2 = mlse[s * G + g];
            const int64_t orow = (int64_t)x.r * a.hq + x.h * Gt + x.sg * G + g;
            if (parts == 1) {
                *reinterpret_cast<uint32_t *>(a.out + orow * DK + d) = pack_bf16x2(acc.x, acc.y);
                if (a.lse && d == 0) a.lse[orow] = lse2 == -INFINITY ? -INFINITY : lse2 * kFlLn2;
            } else {
                const int part = cta - fc;
                *reinterpret_cast<float2 *>(a.o_part + (orow * a.fl_parts + part) * DK + d) = acc;
                if (d == 0) a.lse_part[orow * a.fl_parts + part] = lse2;
            }
        }
        if (parts == 1) continue;
        // the last CTA of the row to finish merges its parts
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t prev = atomicAdd(&a.row_done[rho], 1u);
            s_last[s] = prev == (uint32_t)parts - 1;
        }
        __syncthreads();
        if (!s_last[s]) continue;
        __threadfence();
        for (int t = threadIdx.x; t < G * DK / 4; t += blockDim.x) {
            const int g = t / (DK / 4), d = (t % (DK / 4)) * 4;
            const int64_t orow = (int64_t)x.r * a.hq + x.h * Gt + x.sg * G + g;
            const float *lp = a.lse_part + orow * a.fl_parts;
            float M = -INFINITY;
            for (int p = 0; p < parts; ++p) M = fmaxf(M, __ldcg(lp + p));
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            float wsum = 0.f;
            if (M != -INFINITY) {
                for (int p = 0; p < parts; ++p) {
                    const float ls = __ldcg(lp + p);
                    if (ls == -INFINITY) continue;
                    const float f = fast_ex2(ls - M);
                    wsum += f;
                    const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.o_part + (orow * a.fl_parts + p) * DK + d));
                    acc.x += f * v.x;
                    acc.y += f * v.y;
                    acc.z += f * v.z;
                    acc.w += f * v.w;
                }
            }
            const bool empty_set = !(wsum > 0.f);
            const float inv = empty_set ? 0.f : 1.f / wsum;
            uint2 pk;
            pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
            pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2 *>(a.out + orow * DK + d) = pk;
            if (a.lse && d == 0) a.lse[orow] = empty_set ? -INFINITY : (M + fast_lg2(wsum)) * kFlLn2;
        }
        if (threadIdx.x == 0) a.row_done[rho] = 0u;   // ready for the next call
    }
}

template <int DK, int G, int KSEL>
cudaError_t launch_flat_t(const AttnArgs &a, cudaStream_t s)
{
    using LY = FlLayout<DK, G>;
    auto kern = k_attn_flat<DK, G, KSEL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM);
    if (e != cudaSuccess) return e;
    e = launch_kernel_ex(a.pdl_early != 0 || pdl_enabled(), kern, dim3(a.fl_ctas), dim3(kFlWarps * 32), LY::SMEM, s,
                         a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int attention_flat_ctas_per_sm() { return kFlCtasPerSm; }
int attention_flat_warps() { return kFlWarps; }
int attention_flat_max_items_per_warp() { return kFlMaxItemsPerWarp; }
bool attention_flat_can_select(int cols, int k) { return cols <= kTfThreads * 32 && k > 0 && k <= kFlMaxSel; }

cudaError_t launch_attention_flat(const AttnArgs &a, int gs, cudaStream_t s, bool *unsupported)
{
    *unsupported = false;
    if (a.batch == 0 || a.fl_total == 0) return cudaSuccess;
    const int ksel = !a.sel_scores ? 0 : (a.sel_cols <= kTfThreads * 8 ? 8 : 32);
    if (a.sel_scores && (a.sel_cols > kTfThreads * 32 || a.nsel > kFlMaxSel || a.nsel <= 0)) {
        *unsupported = true;
        return cudaSuccess;
    }
#define LSA_FL_CASE(D, G_)                                                    \
    if (a.c.dk == D && gs == G_) {                                            \
        if (ksel == 8) return launch_flat_t<D, G_, 8>(a, s);                  \
        if (ksel == 32) return launch_flat_t<D, G_, 32>(a, s);                \
        return launch_flat_t<D, G_, 0>(a, s);                                 \
    }
    LSA_FL_CASE(64, 2) LSA_FL_CASE(64, 4) LSA_FL_CASE(64, 8)
    LSA_FL_CASE(128, 2) LSA_FL_CASE(128, 4) LSA_FL_CASE(128, 8)
#undef LSA_FL_CASE
    *unsupported = true;
    return cudaSuccess;
}

}  // namespace lsa

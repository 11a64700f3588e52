// Sparse attention for GQA groups of 64 query heads on the fifth-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// The 64 heads of a group share one KV head: the coarse-to-fine workload
// (64 query heads over one KV head, d = 128) and the MLA-shaped latent cache
// (64 heads over one latent head, 576-dim keys whose first 512 dims are the
// values).  A decode step has one query per head, so over a tile of 128
// attended tokens the two products of attention, S = Q K^T and O = P V
// (Vortex blog post, block top-k equation), are dense [64 x dk x 128] and
// [64 x 128 x dv] contractions -- the case the post's own MLA kernel serves
// ("Designing for a new architecture").  They run transposed, so that the
// tile's tokens (and then the value dims) are the MMA's M = 128 rows, one
// TMEM lane each:
//   S^T [128 tokens x 64 heads] = K_tile [128 x dk]  . Q^T [dk x 64]
//   O^T [128 dims   x 64 heads] = V_tile^T [128 x 128] . P^T [128 x 64]
// (one O^T product per 128 value dims).
//
// One CTA of four warps per (request, KV head, tile of 128 tokens).  The
// tile's token rows (forced sink tokens, the selected blocks or tokens, the
// forced recent tokens, walked in 16-token items as by the other attention
// kernels) are gathered with 16-byte cp.async copies into shared memory in
// the 128-byte swizzled atom layout the MMA descriptors describe; the
// latent cache's values are read as V^T straight from the key tile.  Warp
// w reads TMEM lane quadrant w: a thread owns one token, and reads its 64
// scores from TMEM 32 heads at a time; the softmax's per-head maximum and
// sum are reduced across the tile (a reduce-scatter within each warp, then
// across the four warps in shared memory), and the bf16 weights P^T go back
// to shared memory, over the query atoms, as the B operand of the second
// product.  Every tile writes
// its normalised output and log-sum-exp; the tiles of a row are merged by
// log-sum-exp (ByteCross, Appendix A) in the merge kernel.
#include <cuda.h>   // CUtensorMap (the encoder is taken from the driver at run time)
#include <math.h>

#include "attn_items.cuh"
#include "lsa_device.cuh"

namespace lsa {
namespace {

constexpr int kUmThreads = 128;                 // four warps: warp w reads TMEM lane quadrant w
constexpr int kUmTok = 128;                     // tokens per tile (the MMA's M)
constexpr int kUmHeads = 64;                    // query heads of the group (the MMA's N)
constexpr int kUmItems = kUmTok / kChunk;       // 16-token items per tile
constexpr float kUmLn2 = 0.693147180559945309f;

template <int DK, int DV, bool ALIAS>
struct UmLayout {
    static constexpr int KC = DK / 64;                   // 64-dim atom columns of a key row
    static constexpr int VC = DV / 64;
    static constexpr int COL = (kUmTok / 8) * 1024;      // one atom column of a tile: 16 atoms of 8 rows
    static constexpr int QCOL = (kUmHeads / 8) * 1024;   // one atom column of the query tile
    // values in a region of their own when it fits; otherwise (and for the
    // latent cache) the value rows are the key region's first DV / 64 atom
    // columns: aliased, or reloaded there once S^T is done
    static constexpr bool VSEP = !ALIAS && (KC + VC) * COL + KC * QCOL <= 200 * 1024;
    static constexpr int KS = 0;
    static constexpr int VS = VSEP ? KC * COL : 0;
    static constexpr int QS = (KC + (VSEP ? VC : 0)) * COL;
    static constexpr int PS = QS;                        // P^T reuses the query atoms once S^T is done
    static constexpr int ROWS = QS + KC * QCOL;          // int2 (page, slot) per token row
    static constexpr int ROFF = ROWS + kUmTok * 8;       // int64 byte offset of each K / V row (-1: none)
    static constexpr int RED = ROFF + 2 * kUmTok * 8;    // [4 quadrants][64] per-head partials
    static constexpr int STAT = RED + 4 * kUmHeads * 4;  // per-head max, 1 / sum
    static constexpr int BAR = STAT + 2 * kUmHeads * 4;  // mbarrier, TMEM base address, merge flag, query mbarrier
    static constexpr int SMEM = BAR + 24;
    static constexpr int TCOLS_USED = kUmHeads + kUmHeads * (DV / 128);   // S^T, then O^T per 128 dims
    static constexpr int TCOLS = TCOLS_USED <= 128 ? 128 : (TCOLS_USED <= 256 ? 256 : 512);
    static_assert(DK % 64 == 0 && DV % 128 == 0, "tile shapes");
    static_assert(ALIAS ? DV <= DK : true, "latent values are a prefix of the key");
    static_assert(KC * QCOL >= (kUmTok / 8) * 1024, "P^T fits over the query atoms");
    static_assert(VSEP || VC <= KC, "values fit in the key region");
    static_assert(TCOLS_USED <= 512, "tensor memory has 512 columns");
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

// Reduces 32 per-thread values over the warp's 32 lanes column by column
// (a reduce-scatter: each step hands half of the columns to the partner
// lane); lane L ends with column L.
template <class Op>
__device__ __forceinline__ float warp_col_reduce32(const float (&v)[32], Op op)
{
    const int lane = threadIdx.x & 31;
    float b[16], c[8], d[4], e[2];
    bool up = (lane & 16) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float send = up ? v[i] : v[16 + i];
        b[i] = op(up ? v[16 + i] : v[i], __shfl_xor_sync(0xffffffffu, send, 16));
    }
    up = (lane & 8) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float send = up ? b[i] : b[8 + i];
        c[i] = op(up ? b[8 + i] : b[i], __shfl_xor_sync(0xffffffffu, send, 8));
    }
    up = (lane & 4) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = up ? c[i] : c[4 + i];
        d[i] = op(up ? c[4 + i] : c[i], __shfl_xor_sync(0xffffffffu, send, 4));
    }
    up = (lane & 2) != 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = up ? d[i] : d[2 + i];
        e[i] = op(up ? d[2 + i] : d[i], __shfl_xor_sync(0xffffffffu, send, 2));
    }
    up = (lane & 1) != 0;
    const float send = up ? e[0] : e[1];
    return op(up ? e[1] : e[0], __shfl_xor_sync(0xffffffffu, send, 1));
}

struct OpMax {
    __device__ float operator()(float x, float y) const { return fmaxf(x, y); }
};
struct OpAdd {
    __device__ float operator()(float x, float y) const { return x + y; }
};

// Gathers the tile's rows of a paged cache into NC atom columns (128 bytes
// of every row each): a task is one (atom column, row) pair, copied by 8
// lanes with 16-byte cp.async, so one warp instruction moves 4 whole
// 128-byte lines.  roff[t]: the row's byte offset from `base`, or -1 for a
// row with nothing to attend, which is zero-filled instead (it carries
// weight 0, and must not hold NaNs that 0 * NaN would spread).
template <int NC>
__device__ __forceinline__ void gather_rows(uint32_t dst, uint8_t *dst_generic, const uint8_t *base,
                                            const int64_t *roff, int col_bytes, uint64_t pol)
{
    const int lane = threadIdx.x & 31, j = lane & 7;
    for (int task = (threadIdx.x >> 3); task < NC * kUmTok; task += kUmThreads / 8) {
        const int cc = task >> 7, t = task & (kUmTok - 1);
        const int64_t o = roff[t];
        const uint32_t off = (uint32_t)(cc * col_bytes) + atom_offset(t, j);
        if (o >= 0)
            cp_async16_policy(dst + off, base + o + cc * 128 + j * 16, pol);
        else
            *reinterpret_cast<uint4 *>(dst_generic + off) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// tmq: a 2-D tensor map of the queries [B * Hq rows, DK] (bf16, 64 x 64
// boxes, 128-byte swizzle): the group's 64 x DK query tile comes in with one
// tensor copy per 64-dim atom column, already in the MMA's atom layout.
template <int DK, int DV, bool ALIAS>
__global__ void __launch_bounds__(kUmThreads, 1) k_sparse_attn_umma(AttnArgs a, const __grid_constant__ CUtensorMap tmq)
{
    pdl_enter();
    using LY = UmLayout<DK, DV, ALIAS>;
    constexpr uint32_t IDESC_S = umma_idesc_bf16(kUmTok, kUmHeads, false, false);
    constexpr uint32_t IDESC_O = umma_idesc_bf16(128, kUmHeads, true, true);
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_addr(smem) & 1023u) != 0) {   // the swizzled atoms must be 1024-byte aligned
        if (tid == 0) flag_error(a.status, LSA_ERR_INVALID_ARG);
        return;
    }
    const CacheView &c = a.c;
    const int split = blockIdx.x;
    const int rh = blockIdx.y;
    const int r = (int)fdiv((uint32_t)rh, a.fd_hkv), h = rh - r * c.hkv;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + LY::BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + LY::BAR + 8);
    uint64_t *qbar = reinterpret_cast<uint64_t *>(smem + LY::BAR + 16);
    int2 *rows = reinterpret_cast<int2 *>(smem + LY::ROWS);
    int64_t *koff = reinterpret_cast<int64_t *>(smem + LY::ROFF);   // [128] K rows, then [128] V rows
    int64_t *voff = koff + kUmTok;
    float *red = reinterpret_cast<float *>(smem + LY::RED);
    float *st_m = reinterpret_cast<float *>(smem + LY::STAT);
    float *st_il = st_m + kUmHeads;
    const uint32_t sbase = smem_addr(smem);
    // the TMEM lane quadrant this warp reads
    const int quad = warp;

    if (warp == 0) {
        tmem_alloc(tslot, LY::TCOLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(qbar, 1);
        fence_barrier_init();
    }

    // ---- the tile's token rows: (page, slot), page -1 where nothing is
    // attended, and their byte offsets in K and V
    const RowPlan pl = make_plan(a, r, tid == 0 && split == 0 && h == 0);
    if (tid < kUmTok) {
        const int it = split * kUmItems + tid / kChunk, u = tid % kChunk;
        ItemDesc d{-1, 0, 0};
        if ((lane & 15) == 0 && it < pl.n_items) d = describe_item(a, pl, r, h, it);
        const int src = lane & 16;
        d.page = __shfl_sync(0xffffffffu, d.page, src);
        const int ts = __shfl_sync(0xffffffffu, (int)d.ts, src);
        const int n = __shfl_sync(0xffffffffu, (int)d.n, src);
        int2 rw = make_int2(-1, 0);
        if (n == -1)
            rw = describe_token(a, pl, r, h, it, u);
        else if (u < n)
            rw = make_int2(d.page, ts + u);
        rows[tid] = rw;
        koff[tid] = rw.x >= 0 ? ((int64_t)rw.x * c.kps + (int64_t)h * c.khs + (int64_t)rw.y * c.kts) * 2 : -1;
        voff[tid] = rw.x >= 0 && c.v ? ((int64_t)rw.x * c.vps + (int64_t)h * c.vhs + (int64_t)rw.y * c.vts) * 2 : -1;
    }
    tc_fence_before();
    __syncthreads();   // rows, the barrier and the TMEM address are visible
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;

    // ---- gather K (and V when it has its own region) and the group's queries
    const uint64_t pol = l2_evict_first();
    gather_rows<LY::KC>(sbase + LY::KS, smem + LY::KS, c.k, koff, LY::COL, pol);
    if constexpr (LY::VSEP) gather_rows<LY::VC>(sbase + LY::VS, smem + LY::VS, c.v, voff, LY::COL, pol);
    if (tid == 0) {
        // the group's queries: one tensor copy per 64-dim atom column
        mbar_arrive_expect_tx(qbar, (uint32_t)(LY::KC * kUmHeads * 128));
#pragma unroll 1
        for (int cc = 0; cc < LY::KC; ++cc)
            tma_load_2d(sbase + LY::QS + cc * LY::QCOL, &tmq, cc * 64, r * a.hq + h * a.gsize, qbar);
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- S^T = K_tile Q^T: one 64-dim atom column (four K = 16 steps) at a
    // time, once the queries have landed (a wait that gives up issues
    // nothing; the product's wait below then gives up too)
    bool q_ok = true;
    if (tid == 0) q_ok = mbar_wait(qbar, 0, a.status, a.spin_budget);
    q_ok = __syncthreads_and(q_ok) != 0;
    if (tid == 0 && q_ok) {
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < LY::KC; ++cc) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint64_t ad = umma_desc_sw128(sbase + LY::KS + cc * LY::COL + s * 32, 16, 1024);
                const uint64_t bd = umma_desc_sw128(sbase + LY::QS + cc * LY::QCOL + s * 32, 16, 1024);
                umma_bf16(tmem, ad, bd, IDESC_S, cc > 0 || s > 0);
            }
        }
        umma_commit(bar);
    }
    // a wait that gives up records LSA_ERR_TIMEOUT; the products it waited
    // for are then waited for once more (bounded) before the tensor memory
    // they write is freed
    uint32_t phase = 0;
    bool ok = q_ok && mbar_wait(bar, phase, a.status, a.spin_budget);
    ok = __syncthreads_and(ok) != 0;
    if (ok) {
        tc_fence_after();
        // the values of a cache without its own value region go over the key
        // atoms, which the first product has finished reading
        if constexpr (!ALIAS && !LY::VSEP) {
            gather_rows<LY::VC>(sbase + LY::KS, smem + LY::KS, c.v, voff, LY::COL, pol);
            cp_async_commit();
        }

        // ---- softmax over the tile's tokens, per head (log2 domain): this
        // thread holds token 32 * quad + lane, the 64 heads as two halves of
        // 32 columns
        const int tok = 32 * quad + lane;
        float z[2][32];
        {
            const bool valid = rows[tok].x >= 0;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float sv[32];
                tmem_ld32(tmem + lane_base + 32 * half, sv);
#pragma unroll
                for (int i = 0; i < 32; ++i) z[half][i] = valid ? sv[i] * a.scale_log2 : -INFINITY;
            }
        }
#pragma unroll
        for (int half = 0; half < 2; ++half)
            red[quad * kUmHeads + 32 * half + lane] = warp_col_reduce32(z[half], OpMax());
        __syncthreads();
        if (tid < kUmHeads)
            st_m[tid] = fmaxf(fmaxf(red[tid], red[kUmHeads + tid]), fmaxf(red[2 * kUmHeads + tid], red[3 * kUmHeads + tid]));
        __syncthreads();
        // weights rounded to bf16 once: the MMA multiplies V by these and the
        // denominator sums the same rounded values
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float pr[32];
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float m0 = st_m[32 * half + 2 * i], m1 = st_m[32 * half + 2 * i + 1];
                const float p0 = z[half][2 * i] == -INFINITY ? 0.f : fast_ex2(z[half][2 * i] - m0);
                const float p1 = z[half][2 * i + 1] == -INFINITY ? 0.f : fast_ex2(z[half][2 * i + 1] - m1);
                pk[i] = pack_bf16x2(p0, p1);
                const float2 f = bf2_to_f2(pk[i]);
                pr[2 * i] = f.x;
                pr[2 * i + 1] = f.y;
            }
            // P^T row `tok`, heads 32 * half .. + 31: 4 chunks of 16 bytes
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                *reinterpret_cast<uint4 *>(smem + LY::PS + atom_offset(tok, 4 * half + jj)) =
                    make_uint4(pk[4 * jj], pk[4 * jj + 1], pk[4 * jj + 2], pk[4 * jj + 3]);
            // the column maxima of `red` were read before the last barrier
            red[quad * kUmHeads + 32 * half + lane] = warp_col_reduce32(pr, OpAdd());
        }
        if constexpr (!ALIAS && !LY::VSEP) cp_async_wait<0>();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- O^T = V_tile^T P^T, 128 value dims per product, 16 tokens per step
        if (tid == 0) {
            tc_fence_after();
#pragma unroll 1
            for (int d = 0; d < DV / 128; ++d) {
#pragma unroll
                for (int s = 0; s < kUmTok / 16; ++s) {
                    const uint64_t ad = umma_desc_sw128(sbase + LY::VS + 2 * d * LY::COL + 2 * s * 1024, LY::COL, 1024);
                    // P^T is one atom wide along N (64 heads): its leading
                    // offset is never stepped, and is set equal to the
                    // 8-token stride so that the descriptor stays inside
                    // the P^T atoms under either reading of the two fields
                    const uint64_t bd = umma_desc_sw128(sbase + LY::PS + 2 * s * 1024, 1024, 1024);
                    umma_bf16(tmem + kUmHeads + kUmHeads * d, ad, bd, IDESC_O, s > 0);
                }
            }
            umma_commit(bar);
        }
        if (tid < kUmHeads) {
            const float l = red[tid] + red[kUmHeads + tid] + red[2 * kUmHeads + tid] + red[3 * kUmHeads + tid];
            const float m = st_m[tid];
            const bool empty_set = !(l > 0.f);
            st_il[tid] = empty_set ? 0.f : 1.f / l;
            const float lse2 = empty_set ? -INFINITY : m + fast_lg2(l);
            const int64_t orow = (int64_t)r * a.hq + (int64_t)h * a.gsize + tid;
            if (a.splits == 1) {
                if (a.lse) a.lse[orow] = empty_set ? -INFINITY : lse2 * kUmLn2;
            } else {
                a.lse_part[orow * a.splits + split] = lse2;
            }
        }
        phase = 1;
        ok = mbar_wait(bar, phase, a.status, a.spin_budget);
        ok = __syncthreads_and(ok) != 0;   // also makes st_il visible
        if (ok) {
            tc_fence_after();
            // ---- epilogue: this thread holds value dim d * 128 + 32 * quad +
            // lane of all 64 heads, read 32 heads at a time
#pragma unroll 1
            for (int d = 0; d < DV / 128; ++d) {
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float o[32];
                    tmem_ld32(tmem + lane_base + kUmHeads + kUmHeads * d + 32 * half, o);
                    const int64_t hrow0 = (int64_t)r * a.hq + (int64_t)h * a.gsize + 32 * half;
                    const int dim = d * 128 + 32 * quad + lane;
                    const float *il = st_il + 32 * half;
                    if (a.splits == 1) {
                        uint16_t *dst = a.out + hrow0 * DV + dim;
#pragma unroll
                        for (int g = 0; g < 32; ++g) {
                            const __nv_bfloat16 bv = __float2bfloat16_rn(o[g] * il[g]);
                            dst[(int64_t)g * DV] = *reinterpret_cast<const uint16_t *>(&bv);
                        }
                    } else {
                        float *dst = a.o_part + (hrow0 * a.splits + split) * DV + dim;
                        const int64_t stride = (int64_t)a.splits * DV;
#pragma unroll
                        for (int g = 0; g < 32; ++g) dst[g * stride] = o[g] * il[g];
                    }
                }
            }
        }
    }
    if (!ok) {
        if (q_ok) mbar_wait(bar, phase, nullptr, a.spin_budget);   // products in flight
        else if (tid == 0) mbar_wait(qbar, 0, nullptr, a.spin_budget);   // query copies in flight
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, LY::TCOLS);

    // ---- the row's tiles merged inside the kernel (the planner launches
    // this only when every CTA of the grid is resident at once): when all
    // tiles of the row have written their parts, tile `split` merges a
    // slice of the row's 64 x DV outputs by log-sum-exp (ByteCross,
    // Appendix A)
    if (a.merge_in_kernel && a.splits > 1) {
        uint32_t *s_ok = reinterpret_cast<uint32_t *>(smem + LY::BAR + 12);
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            atomicAdd(a.mrg_arrive + rh, 1u);
            *s_ok = wait_counter_eq(a.mrg_arrive + rh, (uint32_t)a.splits, a.status, a.spin_budget) ? 1u : 0u;
        }
        __syncthreads();
        if (*s_ok) {
            constexpr int kB = 8;
            const int total4 = kUmHeads * DV / 4;
            const int per = (total4 + a.splits - 1) / a.splits;
            const int q1 = min(total4, (split + 1) * per);
            const int64_t orow0 = (int64_t)r * a.hq + (int64_t)h * a.gsize;
            for (int q = split * per + tid; q < q1; q += kUmThreads) {
                const int g = q / (DV / 4), d = (q % (DV / 4)) * 4;
                const int64_t orow = orow0 + g;
                const float *lp = a.lse_part + orow * a.splits;
                float M = -INFINITY;
                for (int s0 = 0; s0 < a.splits; s0 += kB) {
                    float l8[kB];
#pragma unroll
                    for (int e = 0; e < kB; ++e) l8[e] = s0 + e < a.splits ? __ldcg(lp + s0 + e) : -INFINITY;
#pragma unroll
                    for (int e = 0; e < kB; ++e) M = fmaxf(M, l8[e]);
                }
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float wsum = 0.f;
                if (M != -INFINITY) {
                    for (int s0 = 0; s0 < a.splits; s0 += kB) {
                        float l8[kB];
                        float4 v8[kB];
#pragma unroll
                        for (int e = 0; e < kB; ++e) {
                            const int sp = s0 + e;
                            l8[e] = sp < a.splits ? __ldcg(lp + sp) : -INFINITY;
                            v8[e] = sp < a.splits ? __ldcg(reinterpret_cast<const float4 *>(a.o_part + (orow * a.splits + sp) * DV + d))
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int e = 0; e < kB; ++e) {
                            if (l8[e] == -INFINITY) continue;
                            const float f = fast_ex2(l8[e] - M);
                            wsum += f;
                            acc.x += f * v8[e].x;
                            acc.y += f * v8[e].y;
                            acc.z += f * v8[e].z;
                            acc.w += f * v8[e].w;
                        }
                    }
                }
                const bool empty_set = !(wsum > 0.f);
                const float inv = empty_set ? 0.f : 1.f / wsum;
                uint2 pk;
                pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
                pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
                *reinterpret_cast<uint2 *>(a.out + orow * DV + d) = pk;
                if (a.lse && d == 0) a.lse[orow] = empty_set ? -INFINITY : (M + fast_lg2(wsum)) * kUmLn2;
            }
        }
        __syncthreads();
        if (tid == 0) {   // the row's last CTA out resets its counters for the next call
            const uint32_t prev = atomicAdd(a.mrg_done + rh, 1u);
            if (prev == (uint32_t)a.splits - 1) {
                a.mrg_arrive[rh] = 0u;
                a.mrg_done[rh] = 0u;
            }
        }
    }
}

// cuTensorMapEncodeTiled from the driver (the runtime is linked statically;
// the driver library is not linked).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled()
{
    static const EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiledFn) nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The queries [rows, dk] bf16 (rows = batch * Hq, row stride dk) as 64 x 64
// boxes with the 128-byte swizzle.
bool encode_query_map(CUtensorMap *m, const void *q, int64_t rows, int dk)
{
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t gdim[2] = {(cuuint64_t)dk, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)dk * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estride[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DK, int DV, bool ALIAS>
cudaError_t launch_umma_t(const AttnArgs &a, cudaStream_t s)
{
    using LY = UmLayout<DK, DV, ALIAS>;
    auto kern = k_sparse_attn_umma<DK, DV, ALIAS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM);
    if (e != cudaSuccess) return e;
    CUtensorMap tmq;
    if (!encode_query_map(&tmq, a.q, (int64_t)a.batch * a.hq, DK)) return cudaErrorNotSupported;
    e = launch_step_kernel(kern, dim3(a.splits, a.batch * a.c.hkv), dim3(kUmThreads), LY::SMEM, s, a, tmq);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool attention_umma_supported(int dk, int dv, int group, bool alias)
{
    if (group != kUmHeads) return false;
    if (dk == 128 && dv == 128 && !alias) return true;
    if (dk == 576 && dv == 512) return true;
    return false;
}

int attention_umma_items_per_tile() { return kUmItems; }

// CTAs of the kernel for these shapes that one SM holds at once (0 when the
// shape has no instance).
int attention_umma_ctas_per_sm(int dk, int dv, bool alias)
{
    int n = 0;
    auto occ = [&](auto kern, int smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kUmThreads, smem) != cudaSuccess) return 0;
        return b;
    };
    if (dk == 128 && dv == 128 && !alias) n = occ(k_sparse_attn_umma<128, 128, false>, UmLayout<128, 128, false>::SMEM);
    else if (dk == 576 && dv == 512 && alias) n = occ(k_sparse_attn_umma<576, 512, true>, UmLayout<576, 512, true>::SMEM);
    else if (dk == 576 && dv == 512 && !alias) n = occ(k_sparse_attn_umma<576, 512, false>, UmLayout<576, 512, false>::SMEM);
    return n;
}

cudaError_t launch_attention_umma(const AttnArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = false;
    if (a.batch == 0) return cudaSuccess;
    const bool alias = a.c.v_alias != 0;
    if (a.c.dk == 128 && a.c.dv == 128 && !alias) return launch_umma_t<128, 128, false>(a, s);
    if (a.c.dk == 576 && a.c.dv == 512 && alias) return launch_umma_t<576, 512, true>(a, s);
    if (a.c.dk == 576 && a.c.dv == 512 && !alias) return launch_umma_t<576, 512, false>(a, s);
    *unsupported = true;
    return cudaSuccess;
}

}  // namespace lsa

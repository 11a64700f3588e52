// Exact attention over the attended token set T = F U selected, split-K,
// with a log-sum-exp merge of the parts.
//
//   o = softmax(q K_T^T * scale) V_T      (Vortex blog post, block top-k
//                                           equation)
//   parts over a partition of T are merged by log-sum-exp (ByteCross,
//   Appendix A: the sink call and the window call are merged by
//   log-sum-exp; Section 4.4 / Appendix D: split-K decode attention).
//
// One CTA per (request, KV head, query-head subgroup, split).  The split's
// token rows are staged into shared memory by the bulk-copy (TMA) engine in
// items of 16 tokens, one item per slot of a ring: a producer warp issues
// cp.async.bulk for the key and value rows of each item (one copy per
// contiguous run of rows within a page) and arms the slot's mbarrier; four
// consumer warps take items round-robin and run an online softmax.  Inside
// a consumer warp, four groups of eight lanes each own every fourth token of
// the item; a lane holds 8-dim chunks of the queries and of the output
// accumulator, so q . K_t is 16-byte shared loads, packed f32x2 FMAs and a
// three-step shuffle reduction, and P V needs no reduction at all.  The
// lane groups, then the warps, are merged by log-sum-exp at the end.
#include <math.h>

#include "attn_items.cuh"
#include "lsa_device.cuh"

namespace lsa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
constexpr float kLn2 = 0.693147180559945309f;
constexpr int kAttnMaxSmem = 200 * 1024;

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int DK, int DV, bool ALIAS>
struct Layout {
    static constexpr int KROW = DK * 2;
    static constexpr int VROW = DV * 2;
    static constexpr int VOFF = ALIAS ? 0 : kChunk * KROW;        // V rows within a slot
    static constexpr int VSTRIDE = ALIAS ? KROW : VROW;            // bytes between V rows
    static constexpr int ROWB = KROW + (ALIAS ? 0 : VROW);         // bytes staged per token
    static constexpr int SLOT = kChunk * ROWB;
    static constexpr int NSLOT = SLOT <= 8192 ? 8 : 4;
    static constexpr int BAR_OFF = NSLOT * SLOT;
    static constexpr int DESC_OFF = BAR_OFF + NSLOT * 16 + NSLOT * 4 + 16;   // 16-byte aligned
    static int smem_bytes(int ips, int token_mode)
    {
        return DESC_OFF + ips * (int)sizeof(ItemDesc) + (token_mode ? ips * kChunk * (int)sizeof(int2) : 0);
    }
};

// Producer: issue the bulk copies of one described item into a slot;
// returns the rows staged.  `nslot` is written before the barrier is armed.
template <int DK, int DV, bool ALIAS>
__device__ int issue_item(const AttnArgs &a, int h, const ItemDesc &d, const int2 *rows, uint8_t *dst,
                          uint64_t *bar, int *nslot)
{
    using LY = Layout<DK, DV, ALIAS>;
    const CacheView &c = a.c;
    if (d.n > 0) {
        const int n = d.n;
        *nslot = n;   // visible to the consumer through the arrive's release
        mbar_arrive_expect_tx(bar, n * LY::ROWB);
        const uint8_t *ks = c.k + ((int64_t)d.page * c.kps + (int64_t)h * c.khs + (int64_t)d.ts * c.kts) * 2;
        if (c.kts == DK) {
            bulk_g2s(dst, ks, n * LY::KROW, bar);
        } else {
            for (int u = 0; u < n; ++u) bulk_g2s(dst + u * LY::KROW, ks + (int64_t)u * c.kts * 2, LY::KROW, bar);
        }
        if constexpr (!ALIAS) {
            const uint8_t *vs = c.v + ((int64_t)d.page * c.vps + (int64_t)h * c.vhs + (int64_t)d.ts * c.vts) * 2;
            if (c.vts == DV) {
                bulk_g2s(dst + LY::VOFF, vs, n * LY::VROW, bar);
            } else {
                for (int u = 0; u < n; ++u)
                    bulk_g2s(dst + LY::VOFF + u * LY::VROW, vs + (int64_t)u * c.vts * 2, LY::VROW, bar);
            }
        }
        return n;
    }
    if (d.n == 0) return 0;
    int n = 0;
    for (int u = 0; u < kChunk; ++u) n += rows[u].x >= 0;
    if (n == 0) return 0;
    *nslot = n;
    mbar_arrive_expect_tx(bar, n * LY::ROWB);
    int m = 0;
    for (int u = 0; u < kChunk; ++u) {
        const int2 rw = rows[u];
        if (rw.x < 0) continue;
        const uint8_t *ks = c.k + ((int64_t)rw.x * c.kps + (int64_t)h * c.khs + (int64_t)rw.y * c.kts) * 2;
        bulk_g2s(dst + m * LY::KROW, ks, LY::KROW, bar);
        if constexpr (!ALIAS) {
            const uint8_t *vs = c.v + ((int64_t)rw.x * c.vps + (int64_t)h * c.vhs + (int64_t)rw.y * c.vts) * 2;
            bulk_g2s(dst + LY::VOFF + m * LY::VROW, vs, LY::VROW, bar);
        }
        ++m;
    }
    return n;
}

template <int DK, int DV, int GS, bool ALIAS>
__global__ void __launch_bounds__(kAttnThreads, 2) k_sparse_attn(AttnArgs a)
{
    pdl_enter();
    using LY = Layout<DK, DV, ALIAS>;
    constexpr int NCK = DK / 64;   // 8-dim key chunks per lane
    constexpr int NCV = DV / 64;   // 8-dim value chunks per lane
    constexpr int NSLOT = LY::NSLOT;
    static_assert(DK % 64 == 0 && DV % 64 == 0, "head dims must be multiples of 64");

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + LY::BAR_OFF);
    uint64_t *empty = full + NSLOT;
    int *item_n = reinterpret_cast<int *>(empty + NSLOT);
    ItemDesc *descs = reinterpret_cast<ItemDesc *>(smem + LY::DESC_OFF);
    int2 *rows = reinterpret_cast<int2 *>(descs + a.items_per_split);

    const int split = blockIdx.x;
    const int h = blockIdx.y / a.nsub, sg = blockIdx.y % a.nsub;
    const int r = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.hq / a.c.hkv;

    const RowPlan pl = make_plan(a, r, threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0);
    const int i_begin = split * a.items_per_split;
    const int nloc = max(0, min(pl.n_items, i_begin + a.items_per_split) - i_begin);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        fence_barrier_init();
    }
    // resolve every item of this split (selection entries, page ids) in
    // parallel, so the producer streams without dependent global loads
    for (int it = threadIdx.x; it < nloc; it += blockDim.x) descs[it] = describe_item(a, pl, r, h, i_begin + it);
    if (a.token_mode) {
        for (int u = threadIdx.x; u < nloc * kChunk; u += blockDim.x) {
            const int i = i_begin + u / kChunk;
            int2 rw = make_int2(-1, 0);
            if (i >= pl.nsc && i < pl.nsc + pl.nsel_items) rw = describe_token(a, pl, r, h, i, u % kChunk);
            rows[u] = rw;
        }
    }
    __syncthreads();

    float m[GS], l[GS];
    float2 o[GS][NCV][4];
    const int grp = lane >> 3, sub = lane & 7;

    if (warp == kConsumerWarps) {
        // ---------------- producer
        if (lane == 0) {
            for (int k = 0; k < nloc; ++k) {
                const int slot = k % NSLOT;
                if (k >= NSLOT && !mbar_wait(&empty[slot], ((k / NSLOT) - 1) & 1, a.status, a.spin_budget)) break;
                const int n = issue_item<DK, DV, ALIAS>(a, h, descs[k], rows + k * kChunk, smem + slot * LY::SLOT,
                                                        &full[slot], &item_n[slot]);
                if (n == 0) {
                    item_n[slot] = 0;
                    mbar_arrive(&full[slot]);
                }
            }
        }
    } else {
        // ---------------- consumers
        float2 qf[GS][NCK][4];
#pragma unroll
        for (int g = 0; g < GS; ++g) {
            const int hq = h * G + sg * GS + g;
            const uint16_t *qrow = a.q + ((int64_t)r * a.hq + hq) * DK;
#pragma unroll
            for (int kk = 0; kk < NCK; ++kk) {
                const uint4 v = *reinterpret_cast<const uint4 *>(qrow + (sub + 8 * kk) * 8);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 f = bf2_to_f2(w[e]);
                    qf[g][kk][e] = make_float2(f.x * a.scale_log2, f.y * a.scale_log2);
                }
            }
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int kk = 0; kk < NCV; ++kk)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[g][kk][e] = make_float2(0.f, 0.f);
        }

        for (int k = warp; k < nloc; k += kConsumerWarps) {
            const int slot = k % NSLOT;
            if (!mbar_wait(&full[slot], (k / NSLOT) & 1, a.status, a.spin_budget)) break;
            const int n = item_n[slot];
            const uint8_t *Ks = smem + slot * LY::SLOT;
            const uint8_t *Vs = Ks + LY::VOFF;
            if (n > 0) {
                float z[4][GS];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = grp + 4 * j;
                    const uint8_t *krow = Ks + t * LY::KROW;
                    float2 acc[GS];
#pragma unroll
                    for (int g = 0; g < GS; ++g) acc[g] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int kk = 0; kk < NCK; ++kk) {
                        const uint4 kv = *reinterpret_cast<const uint4 *>(krow + (sub + 8 * kk) * 16);
                        const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 kf = bf2_to_f2(w[e]);
#pragma unroll
                            for (int g = 0; g < GS; ++g) acc[g] = __ffma2_rn(qf[g][kk][e], kf, acc[g]);
                        }
                    }
#pragma unroll
                    for (int g = 0; g < GS; ++g) {
                        float zz = acc[g].x + acc[g].y;
                        zz += __shfl_xor_sync(0xffffffffu, zz, 4);
                        zz += __shfl_xor_sync(0xffffffffu, zz, 2);
                        zz += __shfl_xor_sync(0xffffffffu, zz, 1);
                        z[j][g] = t < n ? zz : -INFINITY;
                    }
                }
                float p[4][GS];
#pragma unroll
                for (int g = 0; g < GS; ++g) {
                    const float mx = fmaxf(fmaxf(z[0][g], z[1][g]), fmaxf(z[2][g], z[3][g]));
                    const float mn = fmaxf(m[g], mx);
                    if (mn == -INFINITY) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) p[j][g] = 0.f;
                        continue;
                    }
                    const float alpha = ex2(m[g] - mn);
                    float ps = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        p[j][g] = ex2(z[j][g] - mn);
                        ps += p[j][g];
                    }
                    l[g] = l[g] * alpha + ps;
                    m[g] = mn;
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int kk = 0; kk < NCV; ++kk)
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[g][kk][e] = __fmul2_rn(o[g][kk][e], a2);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = grp + 4 * j;
                    if (t < n) {
                        const uint8_t *vrow = Vs + t * LY::VSTRIDE;
#pragma unroll
                        for (int kk = 0; kk < NCV; ++kk) {
                            const uint4 vv = *reinterpret_cast<const uint4 *>(vrow + (sub + 8 * kk) * 16);
                            const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 vf = bf2_to_f2(w[e]);
#pragma unroll
                                for (int g = 0; g < GS; ++g)
                                    o[g][kk][e] = __ffma2_rn(make_float2(p[j][g], p[j][g]), vf, o[g][kk][e]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        // merge the four lane groups of this warp (xor 8, 16)
#pragma unroll
        for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
            for (int g = 0; g < GS; ++g) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m[g], off);
                const float l2 = __shfl_xor_sync(0xffffffffu, l[g], off);
                const float mn = fmaxf(m[g], m2);
                const float a1 = m[g] == -INFINITY ? 0.f : ex2(m[g] - mn);
                const float b1 = m2 == -INFINITY ? 0.f : ex2(m2 - mn);
                l[g] = l[g] * a1 + l2 * b1;
                m[g] = mn;
#pragma unroll
                for (int kk = 0; kk < NCV; ++kk)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 ov;
                        ov.x = __shfl_xor_sync(0xffffffffu, o[g][kk][e].x, off);
                        ov.y = __shfl_xor_sync(0xffffffffu, o[g][kk][e].y, off);
                        o[g][kk][e] = make_float2(o[g][kk][e].x * a1 + ov.x * b1, o[g][kk][e].y * a1 + ov.y * b1);
                    }
            }
        }
    }
    __syncthreads();   // every slot consumed: the ring is reused for the merge

    // merge the consumer warps through shared memory
    float *mo = reinterpret_cast<float *>(smem);                    // [NW][GS][DV]
    float *mm = mo + kConsumerWarps * GS * DV;                      // [NW][GS]
    float *ml = mm + kConsumerWarps * GS;                           // [NW][GS]
    if (warp < kConsumerWarps && grp == 0) {
#pragma unroll
        for (int g = 0; g < GS; ++g) {
#pragma unroll
            for (int kk = 0; kk < NCV; ++kk) {
                float *dst = mo + (warp * GS + g) * DV + (sub + 8 * kk) * 8;
                reinterpret_cast<float4 *>(dst)[0] = make_float4(o[g][kk][0].x, o[g][kk][0].y, o[g][kk][1].x, o[g][kk][1].y);
                reinterpret_cast<float4 *>(dst)[1] = make_float4(o[g][kk][2].x, o[g][kk][2].y, o[g][kk][3].x, o[g][kk][3].y);
            }
            if (sub == 0) {
                mm[warp * GS + g] = m[g];
                ml[warp * GS + g] = l[g];
            }
        }
    }
    __syncthreads();

    for (int t = threadIdx.x; t < GS * DV / 4; t += blockDim.x) {
        const int g = t / (DV / 4), d = (t % (DV / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * GS + g]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float mw = mm[w * GS + g];
                if (mw == -INFINITY) continue;
                const float f = ex2(mw - M);
                wsum += f * ml[w * GS + g];
                const float4 v = *reinterpret_cast<const float4 *>(mo + (w * GS + g) * DV + d);
                acc.x += f * v.x;
                acc.y += f * v.y;
                acc.z += f * v.z;
                acc.w += f * v.w;
            }
        }
        const bool empty_set = !(wsum > 0.f);
        const float inv = empty_set ? 0.f : 1.f / wsum;
        acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        const float lse2 = empty_set ? -INFINITY : M + lg2(wsum);
        const int hq = h * G + sg * GS + g;
        const int64_t orow = (int64_t)r * a.hq + hq;
        if (a.splits == 1) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 packed;
            packed.x = *reinterpret_cast<uint32_t *>(&lo);
            packed.y = *reinterpret_cast<uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(a.out + orow * DV + d) = packed;
            if (a.lse && d == 0) a.lse[orow] = empty_set ? -INFINITY : lse2 * kLn2;
        } else {
            *reinterpret_cast<float4 *>(a.o_part + (orow * a.splits + split) * DV + d) = acc;
            if (d == 0) a.lse_part[orow * a.splits + split] = lse2;
        }
    }
}

// Log-sum-exp merge of the split partials: weights exp2(lse_s - max).  The
// partials of eight splits are loaded at once (one round trip per eight
// splits instead of one per split).
__global__ void k_merge(MergeArgs a)
{
    pdl_enter();
    constexpr int kB = 8;
    const int row = blockIdx.x;
    const int d = threadIdx.x * 4;
    if (d >= a.dv) return;
    const float *lp = a.lse_part + (int64_t)row * a.splits;
    float M = -INFINITY;
    for (int s0 = 0; s0 < a.splits; s0 += kB) {
        float l8[kB];
#pragma unroll
        for (int e = 0; e < kB; ++e) l8[e] = s0 + e < a.splits ? lp[s0 + e] : -INFINITY;
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
                l8[e] = sp < a.splits ? lp[sp] : -INFINITY;
                v8[e] = sp < a.splits ? *reinterpret_cast<const float4 *>(a.o_part + ((int64_t)row * a.splits + sp) * a.dv + d)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int e = 0; e < kB; ++e) {
                if (l8[e] == -INFINITY) continue;   // an empty part adds nothing (its output is not read)
                const float f = ex2(l8[e] - M);
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
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t *>(&lo);
    packed.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(a.out + (int64_t)row * a.dv + d) = packed;
    if (a.lse && d == 0) a.lse[row] = empty_set ? -INFINITY : (M + lg2(wsum)) * kLn2;
}

template <int DK, int DV, int GS, bool ALIAS>
cudaError_t launch_attn_t(const AttnArgs &a, cudaStream_t s)
{
    using LY = Layout<DK, DV, ALIAS>;
    static_assert(LY::NSLOT * LY::SLOT >= kConsumerWarps * GS * DV * 4 + 2 * kConsumerWarps * GS * 4,
                  "merge buffers must fit in the slot ring");
    auto kern = k_sparse_attn<DK, DV, GS, ALIAS>;
    const int smem = LY::smem_bytes(a.items_per_split, a.token_mode);
    if (smem > kAttnMaxSmem) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnMaxSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.splits, a.c.hkv * a.nsub, a.batch);
    cudaError_t le = launch_step_kernel(kern, grid, dim3(kAttnThreads), smem, s, a);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

}  // namespace

bool attention_supported(int dk, int dv, int group, bool alias, int *sub_group)
{
    int gs = 0;
    if (dk == 64 && dv == 64 && !alias) gs = group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1);
    else if (dk == 128 && dv == 128 && !alias) gs = group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1);
    else if (dk == 576 && dv == 512) gs = 1;
    if (sub_group) *sub_group = gs;
    return gs > 0;
}

int attention_max_items_per_split(int dk, int dv, bool alias, int token_mode)
{
    const int rowb = dk * 2 + (alias ? 0 : dv * 2);
    const int slot = kChunk * rowb;
    const int nslot = slot <= 8192 ? 8 : 4;
    const int fixed = nslot * slot + nslot * 20 + 16;
    const int per = (int)sizeof(ItemDesc) + (token_mode ? kChunk * (int)sizeof(int2) : 0);
    return (kAttnMaxSmem - fixed) / per;
}

int attention_items_max(int sink, int recent, int b, int nsel, int token_mode)
{
    const int sel_items = token_mode ? (nsel + kChunk - 1) / kChunk : nsel * (b / kChunk);
    return (sink + kChunk - 1) / kChunk + sel_items + (recent + kChunk - 1) / kChunk + 1;
}

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s, bool *unsupported)
{
    *unsupported = false;
    if (a.batch == 0) return cudaSuccess;
    const int G = a.hq / a.c.hkv;
    const int gs = G / a.nsub;
    const bool alias = a.c.v_alias != 0;
#define LSA_ATTN_CASE(DK_, DV_, GS_, AL_) \
    if (a.c.dk == DK_ && a.c.dv == DV_ && gs == GS_ && alias == AL_) return launch_attn_t<DK_, DV_, GS_, AL_>(a, s);
    LSA_ATTN_CASE(64, 64, 4, false) LSA_ATTN_CASE(64, 64, 2, false) LSA_ATTN_CASE(64, 64, 1, false)
    LSA_ATTN_CASE(128, 128, 4, false) LSA_ATTN_CASE(128, 128, 2, false) LSA_ATTN_CASE(128, 128, 1, false)
    LSA_ATTN_CASE(576, 512, 1, true) LSA_ATTN_CASE(576, 512, 1, false)
#undef LSA_ATTN_CASE
    *unsupported = true;
    return cudaSuccess;
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s)
{
    if (a.rows == 0) return cudaSuccess;
    cudaError_t le = launch_step_kernel(k_merge, dim3(a.rows), dim3((a.dv + 3) / 4), 0, s, a);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

}  // namespace lsa

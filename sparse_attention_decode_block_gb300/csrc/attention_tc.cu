// Split-K sparse attention for GQA groups of 2..8 query heads on the
// tensor cores (mma.sync m16n8k16, bf16 inputs, fp32 accumulation).
//
// Same contract as the CUDA-core kernel in attention.cu: one CTA per
// (request, KV head, split) walks the split's 16-token items (forced sink
// tokens, selected blocks, forced recent tokens), runs an online softmax and
// writes the split's normalised output and log-sum-exp for the log-sum-exp
// merge (ByteCross, Appendix A; Vortex blog post, block top-k equation).
//
// What differs is the inner product engine.  A decode step has one query
// per head, so a KV head's group forms a small dense tile: S = Q K^T is
// [G heads x 16 tokens x d] and O += P V is [G x 16 x d].  Both run as
// m16n8k16 MMAs with the G heads in the M dimension (rows G..15 are zero),
// which needs ~130 issued instructions per 16-token item where the CUDA-core
// kernel needs ~1000.
//
// Staging: every warp streams its own items.  A bulk (TMA) copy engine
// serves the copies of one issuing warp one after another (about one copy
// per DRAM round trip, measured), so a single producer warp caps a CTA at a
// few GB/s; instead each warp issues 16-byte cp.async copies for its next
// items into its own ring of stages (no producer, no mbarriers: commit
// groups), writing K and V rows in a 128-byte XOR-swizzled layout so that
// the ldmatrix fragment loads (8 token rows at one column) hit 8 different
// bank groups.
#include <math.h>

#include "attn_items.cuh"
#include "lsa_device.cuh"

namespace lsa {
namespace {

constexpr int kTcWarps = 4;     // each warp streams and computes its own items
constexpr int kTcStages = 3;    // ring stages per warp
constexpr float kTcLn2 = 0.693147180559945309f;

template <int DK>
struct TcLayout {
    static constexpr int CPR = DK / 8;            // 16-byte chunks per token row
    static constexpr int SUB = kChunk * 128;      // one swizzled 16-row x 128-byte sub-tile
    static constexpr int KBYTES = (DK / 64) * SUB;
    static constexpr int STAGE = 2 * KBYTES;      // K tile then V tile
    static constexpr int WARP_RING = kTcStages * STAGE;
    static constexpr int SMEM = kTcWarps * WARP_RING + kTcWarps * 16;   // + rows staged per stage
};

template <int DK, int G>
__global__ void __launch_bounds__(kTcWarps * 32) k_sparse_attn_tc(AttnArgs a)
{
    pdl_enter();
    using LY = TcLayout<DK>;
    constexpr int NT = DK / 8;        // n-tiles of the output (DV = DK)
    constexpr int CPL = kChunk * LY::CPR / 32;   // 16-byte chunks per lane per tile
    static_assert(G >= 2 && G <= 8, "heads of a group must fit rows 0..7 of the MMA tile");

    extern __shared__ __align__(1024) uint8_t smem[];
    const int split = blockIdx.x;
    const int h = blockIdx.y / a.nsub, sg = blockIdx.y % a.nsub;
    const int r = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Gt = a.hq / a.c.hkv;
    const CacheView &c = a.c;

    if ((smem_addr(smem) & 1023u) != 0) {       // the swizzle assumes 1 KB aligned tiles
        if (threadIdx.x == 0) flag_error(a.status, LSA_ERR_INVALID_ARG);
        return;
    }
    const RowPlan pl = make_plan(a, r, threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0);
    const int i_begin = split * a.items_per_split;
    const int nloc = max(0, min(pl.n_items, i_begin + a.items_per_split) - i_begin);
    // this warp's items: k = warp, warp + W, ...; item j of the warp is k = warp + j*W
    const int nmine = nloc > warp ? (nloc - warp + kTcWarps - 1) / kTcWarps : 0;

    uint8_t *ring = smem + warp * LY::WARP_RING;
    const uint32_t ring_s = smem_addr(ring);
    int *stage_n = reinterpret_cast<int *>(smem + kTcWarps * LY::WARP_RING) + warp * 4;

    // lane-parallel item descriptors, 32 items at a time
    ItemDesc my{-1, 0, 0};
    int my_base = -32;
    auto describe = [&](int j0) {
        my_base = j0;
        const int j = j0 + lane;
        my = j < nmine ? describe_item(a, pl, r, h, i_begin + warp + j * kTcWarps) : ItemDesc{-1, 0, 0};
    };
    auto issue = [&](int j) {
        if (j >= nmine) {
            cp_async_commit();
            return;
        }
        if (j >= my_base + 32) describe(j - (j % 32));
        const int src_lane = j - my_base;
        const int page = __shfl_sync(0xffffffffu, my.page, src_lane);
        const int ts = __shfl_sync(0xffffffffu, (int)my.ts, src_lane);
        const int n = __shfl_sync(0xffffffffu, (int)my.n, src_lane);
        if (lane == 0) stage_n[j % kTcStages] = n;
        if (n > 0) {
            const uint32_t st = ring_s + (j % kTcStages) * LY::STAGE;
            const uint8_t *kb = c.k + ((int64_t)page * c.kps + (int64_t)h * c.khs + (int64_t)ts * c.kts) * 2;
            const uint8_t *vb = c.v + ((int64_t)page * c.vps + (int64_t)h * c.vhs + (int64_t)ts * c.vts) * 2;
#pragma unroll
            for (int u = 0; u < CPL; ++u) {
                const int q = lane + 32 * u;
                const int t = q / LY::CPR, ch = q % LY::CPR;
                if (t < n) {
                    cp_async16(st + swizzle_offset(t, ch), kb + (int64_t)t * c.kts * 2 + ch * 16);
                    cp_async16(st + LY::KBYTES + swizzle_offset(t, ch), vb + (int64_t)t * c.vts * 2 + ch * 16);
                }
            }
        }
        cp_async_commit();
    };

    // query fragments (rows >= G stay zero)
    const int rr = lane >> 2, cc = lane & 3;
    uint32_t qa0[DK / 16], qa2[DK / 16];
    {
        const bool qrow = rr < G;
        const uint16_t *qp = a.q + ((int64_t)r * a.hq + h * Gt + sg * G + (qrow ? rr : 0)) * DK;
#pragma unroll
        for (int ks = 0; ks < DK / 16; ++ks) {
            qa0[ks] = qrow ? *reinterpret_cast<const uint32_t *>(qp + 16 * ks + 2 * cc) : 0u;
            qa2[ks] = qrow ? *reinterpret_cast<const uint32_t *>(qp + 16 * ks + 8 + 2 * cc) : 0u;
        }
    }
    float m = -INFINITY, l = 0.f;
    float o[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    const int mi = lane >> 3, r8 = lane & 7;
    const int tk = (mi >> 1) * 8 + r8, ck = mi & 1;   // K: tokens 0-7/8-15 x dims lo/hi 8
    const int tv = (mi & 1) * 8 + r8, cv = mi >> 1;   // V (transposed)

    describe(0);
#pragma unroll
    for (int j = 0; j < kTcStages - 1; ++j) issue(j);
    for (int j = 0; j < nmine; ++j) {
        issue(j + kTcStages - 1);
        cp_async_wait<kTcStages - 1>();
        __syncwarp();
        const int n = stage_n[j % kTcStages];
        if (n > 0) {
            const uint32_t kbase = ring_s + (j % kTcStages) * LY::STAGE;
            const uint32_t vbase = kbase + LY::KBYTES;
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks) {
                uint32_t b[4];
                ldsm_x4(b, kbase + swizzle_offset(tk, 2 * ks + ck));
                mma_bf16_rows8(s0, qa0[ks], qa2[ks], b[0], b[1]);
                mma_bf16_rows8(s1, qa0[ks], qa2[ks], b[2], b[3]);
            }
            // online softmax on row rr (tokens 2cc, 2cc+1, 8+2cc, 9+2cc); rows
            // of tokens >= n hold stale data and are masked
            const int t0 = 2 * cc;
            const float z0 = t0 < n ? s0[0] * a.scale_log2 : -INFINITY;
            const float z1 = t0 + 1 < n ? s0[1] * a.scale_log2 : -INFINITY;
            const float z2 = t0 + 8 < n ? s1[0] * a.scale_log2 : -INFINITY;
            const float z3 = t0 + 9 < n ? s1[1] * a.scale_log2 : -INFINITY;
            float mx = fmaxf(fmaxf(z0, z1), fmaxf(z2, z3));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m, mx);
            float alpha = 1.f;
            uint32_t pa0 = 0u, pa2 = 0u;
            if (mn != -INFINITY) {
                alpha = fast_ex2(m - mn);
                pa0 = pack_bf16x2(fast_ex2(z0 - mn), fast_ex2(z1 - mn));
                pa2 = pack_bf16x2(fast_ex2(z2 - mn), fast_ex2(z3 - mn));
                m = mn;
            }
            // the denominator sums the same bf16-rounded weights the MMA uses
            const float2 p01 = bf2_to_f2(pa0), p23 = bf2_to_f2(pa2);
            float ps = (p01.x + p01.y) + (p23.x + p23.y);
            ps += __shfl_xor_sync(0xffffffffu, ps, 1);
            ps += __shfl_xor_sync(0xffffffffu, ps, 2);
            l = l * alpha + ps;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                o[nt][0] *= alpha;
                o[nt][1] *= alpha;
            }
            // stale V rows (tokens >= n) meet zero weights, but 0 * NaN is NaN:
            // zero them first
            if (n < kChunk) {
                for (int q = lane; q < (kChunk - n) * LY::CPR; q += 32) {
                    const int t = n + q / LY::CPR, ch = q % LY::CPR;
                    *reinterpret_cast<uint4 *>(ring + (j % kTcStages) * LY::STAGE + LY::KBYTES + swizzle_offset(t, ch)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
#pragma unroll
            for (int dt = 0; dt < DK / 16; ++dt) {
                uint32_t b[4];
                ldsm_x4_t(b, vbase + swizzle_offset(tv, 2 * dt + cv));
                mma_bf16_rows8(o[2 * dt], pa0, pa2, b[0], b[1]);
                mma_bf16_rows8(o[2 * dt + 1], pa0, pa2, b[2], b[3]);
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
    __syncthreads();   // rings drained: reuse them for the merge of the warps

    float *mo = reinterpret_cast<float *>(smem);                // [W][G][DK]
    float *mm = mo + kTcWarps * G * DK;                         // [W][G]
    float *ml = mm + kTcWarps * G;                              // [W][G]
    if (rr < G) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            *reinterpret_cast<float2 *>(mo + (warp * G + rr) * DK + nt * 8 + 2 * cc) = make_float2(o[nt][0], o[nt][1]);
        if (cc == 0) {
            mm[warp * G + rr] = m;
            ml[warp * G + rr] = l;
        }
    }
    __syncthreads();

    for (int t = threadIdx.x; t < G * DK / 4; t += blockDim.x) {
        const int g = t / (DK / 4), d = (t % (DK / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kTcWarps; ++w) M = fmaxf(M, mm[w * G + g]);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kTcWarps; ++w) {
                const float mw = mm[w * G + g];
                if (mw == -INFINITY) continue;
                const float f = fast_ex2(mw - M);
                wsum += f * ml[w * G + g];
                const float4 v = *reinterpret_cast<const float4 *>(mo + (w * G + g) * DK + d);
                acc.x += f * v.x;
                acc.y += f * v.y;
                acc.z += f * v.z;
                acc.w += f * v.w;
            }
        }
        const bool empty_set = !(wsum > 0.f);
        const float inv = empty_set ? 0.f : 1.f / wsum;
        acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        const float lse2 = empty_set ? -INFINITY : M + fast_lg2(wsum);
        const int64_t orow = (int64_t)r * a.hq + h * Gt + sg * G + g;
        if (a.splits == 1) {
            uint2 pk;
            pk.x = pack_bf16x2(acc.x, acc.y);
            pk.y = pack_bf16x2(acc.z, acc.w);
            *reinterpret_cast<uint2 *>(a.out + orow * DK + d) = pk;
            if (a.lse && d == 0) a.lse[orow] = empty_set ? -INFINITY : lse2 * kTcLn2;
        } else {
            *reinterpret_cast<float4 *>(a.o_part + (orow * a.splits + split) * DK + d) = acc;
            if (d == 0) a.lse_part[orow * a.splits + split] = lse2;
        }
    }
}

template <int DK, int G>
cudaError_t launch_tc_t(const AttnArgs &a, cudaStream_t s)
{
    using LY = TcLayout<DK>;
    static_assert(LY::SMEM >= kTcWarps * G * DK * 4 + 2 * kTcWarps * G * 4, "merge buffers must fit in the rings");
    auto kern = k_sparse_attn_tc<DK, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(a.splits, a.c.hkv * a.nsub, a.batch);
    e = launch_step_kernel(kern, grid, dim3(kTcWarps * 32), LY::SMEM, s, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int attention_tc_group(int dk, int dv, int group, bool alias, bool token_mode, const CacheView &v)
{
    if (alias || token_mode || dk != dv || (dk != 64 && dk != 128)) return 0;
    if (group % 8 == 0) return 8;
    if (group % 4 == 0) return 4;
    if (group % 2 == 0) return 2;
    return 0;
}

int attention_tc_max_items_per_split(int)
{
    return 1 << 20;   // descriptors are resolved per warp, 32 at a time
}

cudaError_t launch_attention_tc(const AttnArgs &a, int gs, cudaStream_t s, bool *unsupported)
{
    *unsupported = false;
    if (a.batch == 0) return cudaSuccess;
#define LSA_TC_CASE(D, G_) \
    if (a.c.dk == D && gs == G_) return launch_tc_t<D, G_>(a, s);
    LSA_TC_CASE(64, 2) LSA_TC_CASE(64, 4) LSA_TC_CASE(64, 8)
    LSA_TC_CASE(128, 2) LSA_TC_CASE(128, 4) LSA_TC_CASE(128, 8)
#undef LSA_TC_CASE
    *unsupported = true;
    return cudaSuccess;
}

}  // namespace lsa

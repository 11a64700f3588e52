// The fused decode step: block scores, top-k and split-K attention in one
// persistent kernel (Vortex blog post, "Making it fast": every length is
// known at step start, work is balanced across thread blocks, and operators
// are fused so block scores never make a round trip through a separate
// launch).  The attention phase alone also serves the split-K sparse decode.
//
// Every warp is an independent worker.  It takes tickets from a global
// counter in a fixed order and streams the bytes of its work through its own
// ring of shared-memory stages filled by 16-byte cp.async copies (the
// bulk-copy engine serves one issuing warp's copies one at a time, so it
// cannot feed many small random reads).  The ring stays full across unit
// boundaries: the next unit is described while the previous one's stages
// are still in flight.
//   1. score units     (request, 32 blocks): candidate blocks' summary rows
//                      are dotted with the sum of the group's queries;
//   2. top-k units     (request, KV head): once every score unit of the
//                      request is done, exact radix select of the row held in
//                      registers (ties to the lower block index, ascending
//                      output) with the selected blocks' page ids;
//   3. attention units (request, KV head, part): once the row's selection is
//                      done, 16-token chunks of K and V are streamed through
//                      the ring and run through the tensor cores (m16n8k16,
//                      the group's query heads in the M dimension); each part's
//                      normalised output and log-sum-exp go to the workspace
//                      and the last part of a row to finish merges them by
//                      log-sum-exp (ByteCross, Appendix A).
// A worker only waits for units with smaller tickets, which running workers
// hold and finish without waiting on larger ones, so every wait ends; the
// waits are bounded anyway (LSA_ERR_TIMEOUT) and the launch is cooperative
// (every CTA resident).  The control counters live in the caller's
// workspace; the last worker to leave resets them.
#include <math.h>

#include "attn_items.cuh"
#include "lsa_device.cuh"

namespace lsa {
namespace {

constexpr int kWarps = 8;              // workers per CTA
constexpr int kStages = 3;             // ring stages per worker
constexpr int kStageBytes = 8192;
constexpr int kScoreBlocks = 16;       // blocks per score unit (<= 32: one per lane)
constexpr int kMaxKpl = 64;            // top-k keys per lane (rows of up to 2048 blocks)
constexpr int kPartChunks = 8;         // attention chunks per part (64 KB of K/V at d = 128)
constexpr float kLn2 = 0.693147180559945309f;
constexpr int kCtr = 64;               // words between control counters (256 bytes: one L2 line each)

// Per-stage bookkeeping written by a worker's issuing side and read by its
// computing side.
struct StageMeta {
    int n;          // rows staged (-1: end of the stream)
    int unit;       // score: request; attention: row * parts + part
    int flags;      // bit 0: first stage of the unit, bit 1: last stage
    int pad;
    int j[4];       // score: block index of each staged row
};

constexpr int kMetaBytes = kStages * (int)sizeof(StageMeta);
constexpr int kWarpBytes = kStages * kStageBytes;

#ifdef LSA_FUSED_TRACE
__device__ __forceinline__ uint64_t gtimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
#define LSA_TRACE(a, unit, field)                                                         \
    do {                                                                                  \
        if ((a).trace && (threadIdx.x & 31) == 0) (a).trace[4 * (int64_t)(unit) + (field)] = gtimer(); \
    } while (0)
#else
#define LSA_TRACE(a, unit, field) \
    do {                          \
    } while (0)
#endif

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait of a whole warp until *p >= target (acquire); backs off so
// that many waiting warps do not flood one L2 slice.
__device__ __forceinline__ bool wait_counter(const uint32_t *p, uint32_t target, uint32_t *status, long long budget)
{
    uint32_t ok = 1;
    if ((threadIdx.x & 31) == 0 && ld_acquire(p) < target) {
        const long long t0 = clock64();
        unsigned ns = 64;
        while (ld_acquire(p) < target) {
            if (clock64() - t0 > budget) {
                flag_error(status, LSA_ERR_TIMEOUT);
                ok = 0;
                break;
            }
            __nanosleep(ns);
            if (ns < 1024) ns <<= 1;
        }
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Tickets are unsigned and compared against the unit counts before any
// use, so a counter that was not zero at launch (a workspace that broke the
// zero-fill contract) can only skip work, never index out of range.
__device__ __forceinline__ uint32_t fetch_ticket(uint32_t *ctr)
{
    uint32_t t = 0;
    if ((threadIdx.x & 31) == 0) t = atomicAdd(ctr, 1u);
    return __shfl_sync(0xffffffffu, t, 0);
}

// Every lane fences its own writes before lane 0 publishes them.
__device__ __forceinline__ void publish(uint32_t *ctr)
{
    __threadfence();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) atomicAdd(ctr, 1u);
}

// Ticket order: score units of request 0, then of request 1, then the top-k
// units of request 0, score units of request 2, top-k of request 1, ...;
// then every attention unit.  A request's top-k comes one request's worth of
// score units after its own score units, so it rarely waits, and the
// selection of early requests overlaps the scoring of later ones.
enum UnitKind { kScoreUnit = 0, kTopkUnit = 1, kAttnUnit = 2 };

__device__ __forceinline__ int unit_kind(const FusedArgs &a, uint32_t t, int *id)
{
    const uint32_t SP = (uint32_t)a.score_chunks, H = (uint32_t)a.c.hkv, B = (uint32_t)a.batch;
    if (t >= (uint32_t)a.attn_base) {
        *id = (int)(t - (uint32_t)a.attn_base);
        return kAttnUnit;
    }
    if (t < SP) {
        *id = (int)t;
        return kScoreUnit;
    }
    t -= SP;
    if (t < (B - 1) * (SP + H)) {
        const uint32_t blk = t / (SP + H) + 1, wi = t % (SP + H);
        if (wi < SP) {
            *id = (int)(blk * SP + wi);
            return kScoreUnit;
        }
        *id = (int)((blk - 1) * H + (wi - SP));
        return kTopkUnit;
    }
    *id = (int)((B - 1) * H + (t - (B - 1) * (SP + H)));
    return kTopkUnit;
}

struct Worker {
    uint8_t *ring;          // kStages stages of kStageBytes
    uint32_t ring_s;        // shared-window address of the ring
    StageMeta *meta;
    int issued, computed;   // stage counters
};

// ================================================================== scores

template <int DK, int HKV>
struct ScoreStream {
    static constexpr int ROWB = HKV * DK * 2;                 // one page's summaries
    static constexpr int BPS = kStageBytes / ROWB > 4 ? 4 : kStageBytes / ROWB;   // rows per stage
    static constexpr int NCH = HKV * DK / 8;                  // 16-byte chunks per row
    static constexpr int NI = (NCH + 31) / 32;
    static constexpr int CPH = DK / 8;
    static_assert(BPS >= 1, "summary row larger than a stage");
    static_assert((CPH <= 32 && 32 % CPH == 0) || HKV == 1, "head rows must tile the warp");

    int u_r, u_j0, u_ncand, u_nst, u_k;   // current unit; lane l describes block u_j0 + l
    uint32_t u_mask;
    int u_page;
    bool have, ended;
    uint32_t t_next;                      // next ticket (already taken)
    float qs[NI][8];                      // sum of the group's queries, this lane's chunks
    int qs_r;
};

template <int DK, int HKV>
__device__ void score_describe(const FusedArgs &a, ScoreStream<DK, HKV> &S, int unit)
{
    const int lane = threadIdx.x & 31;
    const int r = unit / a.score_chunks, c = unit % a.score_chunks;
    const int j0 = c * a.score_blocks, j = j0 + lane;
    const bool mine = lane < a.score_blocks && j < a.max_blocks;
    int L = a.lens[r];
    const int p_raw = mine ? a.pt[(int64_t)r * a.max_blocks + j] : -1;   // in parallel with L
    const bool len_ok = L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * a.c.b;
    if (!len_ok) {
        if (lane == 0 && c == 0) flag_error(a.status, LSA_ERR_BOUNDS);
        L = 0;
    }
    const int se = min(a.sink, L);
    const int rs = max(L - a.recent, se);
    bool cand = mine && (int64_t)j * a.c.b >= se && (int64_t)(j + 1) * a.c.b <= rs;
    int p = cand ? p_raw : -1;
    if (cand && (p < 0 || p >= a.c.num_pages)) {
        flag_error(a.status, LSA_ERR_BOUNDS);
        cand = false;
    }
    if (!cand && mine) {
#pragma unroll
        for (int h = 0; h < HKV; ++h) a.scores[((int64_t)r * HKV + h) * a.max_blocks + j] = -INFINITY;
    }
    S.u_mask = __ballot_sync(0xffffffffu, cand);
    S.u_ncand = __popc(S.u_mask);
    S.u_nst = (S.u_ncand + S.BPS - 1) / S.BPS;
    S.u_k = 0;
    S.u_r = r;
    S.u_j0 = j0;
    S.u_page = p;
    S.have = true;
}

// Issue the next stage of the score stream (an empty group at its end).
template <int DK, int HKV>
__device__ void score_issue(const FusedArgs &a, ScoreStream<DK, HKV> &S, Worker &w)
{
    using SS = ScoreStream<DK, HKV>;
    const int lane = threadIdx.x & 31;
    const int slot = w.issued % kStages;
    while (true) {
        if (!S.have) {
            int unit = 0;
            if (S.ended || unit_kind(a, S.t_next, &unit) != kScoreUnit) {
                S.ended = true;
                if (lane == 0) w.meta[slot].n = -1;
                cp_async_commit();
                ++w.issued;
                return;
            }
            LSA_TRACE(a, S.t_next, 0);
            score_describe<DK, HKV>(a, S, unit);
            S.t_next = fetch_ticket(a.ctrl);
            if (S.u_ncand == 0) {
                publish(&a.score_done[S.u_r * kCtr]);   // nothing to stream: the unit is done
                S.have = false;
                continue;
            }
        }
        const int lo = S.u_k * SS::BPS, n = min(SS::BPS, S.u_ncand - lo);
        const uint32_t st = w.ring_s + slot * kStageBytes;
        const bool cand = (S.u_mask >> lane) & 1u;
        const int pos = __popc(S.u_mask & ((1u << lane) - 1u));
        for (int i = 0; i < n; ++i) {
            const int src = __ffs(__ballot_sync(0xffffffffu, cand && pos == lo + i)) - 1;
            const int p = __shfl_sync(0xffffffffu, S.u_page, src);
            const uint8_t *row = reinterpret_cast<const uint8_t *>(a.summ) + (int64_t)p * SS::ROWB;
#pragma unroll
            for (int u = 0; u < SS::NI; ++u) {
                const int ch = lane + 32 * u;
                if (ch < SS::NCH) cp_async16(st + i * SS::ROWB + ch * 16, row + ch * 16);
            }
            if (lane == 0) w.meta[slot].j[i] = S.u_j0 + src;
        }
        if (lane == 0) {
            w.meta[slot].n = n;
            w.meta[slot].unit = S.u_r;
            w.meta[slot].flags = (S.u_k + 1 == S.u_nst) ? 2 : 0;
        }
        cp_async_commit();
        ++w.issued;
        if (++S.u_k == S.u_nst) S.have = false;
        return;
    }
}

template <int DK, int HKV>
__device__ bool score_compute(const FusedArgs &a, ScoreStream<DK, HKV> &S, Worker &w)
{
    using SS = ScoreStream<DK, HKV>;
    const int lane = threadIdx.x & 31;
    const int slot = w.computed % kStages;
    const StageMeta md = w.meta[slot];
    if (md.n < 0) return false;
    ++w.computed;
    const int r = md.unit;
    if (S.qs_r != r) {
        S.qs_r = r;
        const int Gt = a.hq / HKV;
#pragma unroll
        for (int i = 0; i < SS::NI; ++i) {
            const int ch = lane + 32 * i;
#pragma unroll
            for (int e = 0; e < 8; ++e) S.qs[i][e] = 0.f;
            if (ch < SS::NCH) {
                const int h = ch / SS::CPH, d0 = (ch % SS::CPH) * 8;
                for (int g = 0; g < Gt; ++g) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(a.q + ((int64_t)r * a.hq + h * Gt + g) * DK + d0);
                    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = bf2_to_f2(wd[e]);
                        S.qs[i][2 * e] += f.x;
                        S.qs[i][2 * e + 1] += f.y;
                    }
                }
            }
        }
    }
    const uint8_t *st = w.ring + slot * kStageBytes;
    for (int i = 0; i < md.n; ++i) {
        const int j = md.j[i];
        float part[SS::NI];
#pragma unroll
        for (int u = 0; u < SS::NI; ++u) {
            const int ch = lane + 32 * u;
            part[u] = 0.f;
            if (ch < SS::NCH) {
                const uint4 v = *reinterpret_cast<const uint4 *>(st + i * SS::ROWB + ch * 16);
                const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc = __ffma2_rn(make_float2(S.qs[u][2 * e], S.qs[u][2 * e + 1]), bf2_to_f2(wd[e]), acc);
                part[u] = acc.x + acc.y;
            }
        }
        if constexpr (SS::CPH <= 32 && 32 % SS::CPH == 0) {
#pragma unroll
            for (int u = 0; u < SS::NI; ++u) {
#pragma unroll
                for (int off = SS::CPH / 2; off > 0; off >>= 1) part[u] += __shfl_xor_sync(0xffffffffu, part[u], off);
                const int ch = lane + 32 * u;
                if (ch < SS::NCH && (lane % SS::CPH) == 0)
                    a.scores[((int64_t)r * HKV + ch / SS::CPH) * a.max_blocks + j] = part[u];
            }
        } else {
            float tot = 0.f;
#pragma unroll
            for (int u = 0; u < SS::NI; ++u) tot += part[u];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
            if (lane == 0) a.scores[(int64_t)r * a.max_blocks + j] = tot;
        }
    }
    if (md.flags & 2) {
        publish(&a.score_done[r * kCtr]);
#ifdef LSA_FUSED_TRACE
        const int c = md.j[md.n - 1] / a.score_blocks;
        LSA_TRACE(a, r == 0 ? c : a.score_chunks + (r - 1) * (a.score_chunks + a.c.hkv) + c, 1);
#endif
    }
    return true;
}

// Streams score units from ticket t on; returns the first ticket past the
// score units that it took.
template <int DK, int HKV>
__device__ uint32_t score_phase(const FusedArgs &a, uint32_t t, Worker &w)
{
    ScoreStream<DK, HKV> S;
    S.have = false;
    S.ended = false;
    S.t_next = t;
    S.qs_r = -1;
    w.issued = w.computed = 0;
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) score_issue<DK, HKV>(a, S, w);
    while (true) {
        score_issue<DK, HKV>(a, S, w);
        cp_async_wait<kStages - 1>();
        __syncwarp();
        if (!score_compute<DK, HKV>(a, S, w)) break;
        __syncwarp();
    }
    cp_async_wait<0>();
    __syncwarp();
    return S.t_next;
}

// ================================================================== top-k

// Exact top-k of one row by one warp.  Lane l owns the contiguous columns
// [l*KPL, (l+1)*KPL) as order-preserving 32-bit keys in registers.  The k-th
// largest key is found by bisection on the key value; each step counts the
// keys at or above the midpoint with independent compares (four accumulator
// chains) and one warp reduction -- no per-key warp collectives, no atomics.
// Ties go to the lower column: the selection is every key above the
// threshold plus the first keys equal to it; each lane emits its own
// columns in order at offsets given by two warp scans (ascending output,
// -1 padded).
// Bisection on the key value over the keys a warp holds (KPL per lane, 0 =
// not a candidate).  On entry count(key >= lo) >= keff > count(key >= hi);
// returns the largest such lo, or an earlier one with count(key >= lo) ==
// keff exactly (either way the selection is every key > lo plus the first
// keff - count(key > lo) keys == lo).
template <int KPL>
__device__ __forceinline__ uint32_t bisect_keys(const uint32_t (&keys)[KPL], uint64_t lo, uint64_t hi, int keff)
{
    while (hi - lo > 1) {
        const uint32_t mid = (uint32_t)(lo + ((hi - lo) >> 1));
        int c4[4] = {0, 0, 0, 0};
#pragma unroll
        for (int e = 0; e < KPL; ++e) c4[e & 3] += keys[e] >= mid;
        const int c = (int)__reduce_add_sync(0xffffffffu, (uint32_t)((c4[0] + c4[1]) + (c4[2] + c4[3])));
        if (c >= keff) lo = mid;
        else hi = mid;
        if (c == keff) break;
    }
    return (uint32_t)lo;
}

// Writes the selected columns of the keys a warp holds in column order (lane
// l's keys precede lane l+1's, col(e) gives key e's column): every key >
// thresh and the first take_eq keys == thresh.  Position of a taken key =
// taken keys before it = (keys > thresh before it) + min(ties before it,
// take_eq).
template <int KPL, class Col>
__device__ __forceinline__ void emit_selection(const uint32_t (&keys)[KPL], uint32_t thresh, int take_eq,
                                               int32_t *sel, Col col)
{
    const int lane = threadIdx.x & 31;
    uint32_t cnt = 0;   // keys > thresh in the low half, ties in the high half
#pragma unroll
    for (int e = 0; e < KPL; ++e)
        cnt += (keys[e] > thresh ? 1u : 0u) + (keys[e] != 0 && keys[e] == thresh ? 0x10000u : 0u);
    uint32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const uint32_t excl = incl - cnt;
    int g = (int)(excl & 0xffffu), q = (int)(excl >> 16);
    if (cnt == 0) return;
#pragma unroll
    for (int e = 0; e < KPL; ++e) {
        const uint32_t key = keys[e];
        const bool gt = key > thresh, eq = key != 0 && key == thresh;
        if (gt || (eq && q < take_eq)) sel[g + min(q, take_eq)] = col(e);
        g += gt;
        q += eq;
    }
}

constexpr int kCompactKeys = 512;   // candidates kept for the narrow bisection (16 per lane)
static_assert(2 * kCompactKeys * 4 <= kStages * kStageBytes, "top-k scratch lives in the worker's ring");

// Top-k of one score row by one warp, ties to the lower block index, output
// ascending and padded with -1.  The row's keys stay in registers (KPL per
// lane).  A lower bound on the threshold comes from the lanes' own top-2:
// a lane holds at least j keys >= its j-th largest, so the smallest j-th
// largest over n_j lanes has >= j n_j keys at or above it.  When at
// most kCompactKeys keys reach the bound they are compacted (in column
// order) into `scratch` (2 * kCompactKeys words of shared memory) and the
// bisection runs over 8 keys per lane; otherwise over all of them.
template <int KPL>
__device__ void warp_topk(const FusedArgs &a, int row, uint32_t *scratch)
{
    static_assert(KPL % 4 == 0, "keys per lane come in fours");
    const int lane = threadIdx.x & 31;
    const int n = a.max_blocks, k = a.k_blocks;
    const float *srow = a.scores + (int64_t)row * n;
    const int c0 = lane * KPL;
    // Lane l owns columns [l*KPL, (l+1)*KPL).  All loads are issued before
    // any key is inspected: 16-byte loads when the row starts on a 16-byte
    // boundary (max_blocks % 4 == 0) and the lane's range is complete,
    // scalar loads otherwise.
    float v[KPL];
    if (c0 + KPL <= n && (n & 3) == 0) {
#pragma unroll
        for (int e = 0; e < KPL; e += 4) {
            const float4 f = __ldcg(reinterpret_cast<const float4 *>(srow + c0 + e));
            v[e] = f.x;
            v[e + 1] = f.y;
            v[e + 2] = f.z;
            v[e + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < KPL; ++e) v[e] = c0 + e < n ? __ldcg(srow + c0 + e) : -INFINITY;
    }
    uint32_t keys[KPL];
    bool nan = false;
#pragma unroll
    for (int e = 0; e < KPL; ++e) {
        nan |= isnan(v[e]);
        keys[e] = (isnan(v[e]) || v[e] == -INFINITY) ? 0u : float_to_key(v[e]);
    }
    if (nan) flag_error(a.status, LSA_ERR_NAN);
    // valid count, smallest valid key, and the lane's two largest keys
    // (two interleaved chains, merged)
    int nv2[2] = {0, 0};
    uint32_t kmin2[2] = {~0u, ~0u}, t1[2] = {0u, 0u}, t2[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < KPL; ++e) {
        const uint32_t key = keys[e];
        nv2[e & 1] += key != 0;
        kmin2[e & 1] = min(kmin2[e & 1], key ? key : ~0u);
        t2[e & 1] = max(t2[e & 1], min(t1[e & 1], key));
        t1[e & 1] = max(t1[e & 1], key);
    }
    const uint32_t m1 = max(t1[0], t1[1]);
    const uint32_t m2 = max(min(t1[0], t1[1]), max(t2[0], t2[1]));
    const int nv = (int)__reduce_add_sync(0xffffffffu, (uint32_t)(nv2[0] + nv2[1]));
    const uint32_t kmin = __reduce_min_sync(0xffffffffu, min(kmin2[0], kmin2[1]));
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, m1);
    const int keff = min(k, nv);
    int32_t *sel = a.sel + (int64_t)row * k;
    uint32_t thresh = 0;   // with keff == nv every valid key is taken (key > 0)
    int take_eq = 0;
    bool done = false;
    if (keff > 0 && keff < nv) {
        // bound from the lanes holding >= j valid keys (j = 1, 2): their
        // smallest j-th largest key has >= j * (such lanes) keys above it
        uint32_t lo0 = kmin;
        const int l1 = (int)__reduce_add_sync(0xffffffffu, m1 != 0 ? 1u : 0u);
        const int l2 = (int)__reduce_add_sync(0xffffffffu, m2 != 0 ? 1u : 0u);
        if (l1 >= keff) lo0 = max(lo0, __reduce_min_sync(0xffffffffu, m1 != 0 ? m1 : ~0u));
        if (2 * l2 >= keff) lo0 = max(lo0, __reduce_min_sync(0xffffffffu, m2 != 0 ? m2 : ~0u));
        int cl = 0;
#pragma unroll
        for (int e = 0; e < KPL; ++e) cl += keys[e] >= lo0;
        int incl = cl;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const int C = __shfl_sync(0xffffffffu, incl, 31);
        if (C <= kCompactKeys) {
            int pos = incl - cl;
#pragma unroll
            for (int e = 0; e < KPL; ++e) {
                if (keys[e] >= lo0) {
                    scratch[pos] = keys[e];
                    scratch[kCompactKeys + pos] = (uint32_t)(c0 + e);
                    ++pos;
                }
            }
            __syncwarp();
            constexpr int PL = kCompactKeys / 32;
            uint32_t ck[PL];
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                const int idx = lane * PL + i;
                ck[i] = idx < C ? scratch[idx] : 0u;
            }
            const uint32_t th = bisect_keys<PL>(ck, lo0, (uint64_t)kmax + 1, keff);
            int g = 0;
#pragma unroll
            for (int i = 0; i < PL; ++i) g += ck[i] > th;
            const int teq = keff - (int)__reduce_add_sync(0xffffffffu, (uint32_t)g);
            emit_selection<PL>(ck, th, teq, sel,
                               [&](int i) { return (int32_t)scratch[kCompactKeys + lane * PL + i]; });
            __syncwarp();   // scratch is free again
            done = true;
        } else {
            thresh = bisect_keys<KPL>(keys, lo0, (uint64_t)kmax + 1, keff);
            int g4[4] = {0, 0, 0, 0};
#pragma unroll
            for (int e = 0; e < KPL; ++e) g4[e & 3] += keys[e] > thresh;
            take_eq = keff - (int)__reduce_add_sync(0xffffffffu, (uint32_t)((g4[0] + g4[1]) + (g4[2] + g4[3])));
        }
    }
    if (keff > 0 && !done) emit_selection<KPL>(keys, thresh, take_eq, sel, [&](int e) { return c0 + e; });
    for (int i = keff + lane; i < k; i += 32) sel[i] = -1;
}

// ================================================================== attention

struct ChunkDescV {
    int page, ts, n;
};

// Chunk c of row (request r, KV head row % hkv): forced sink tokens, the
// selected blocks in 16-token chunks, forced recent tokens.
__device__ ChunkDescV chunk_desc_v(const FusedArgs &a, int r, int rowi, int L, int se, int rs, int nsc, int nsel_ch,
                                   int c)
{
    const int b = a.c.b;
    ChunkDescV d{-1, 0, 0};
    int t0 = 0, n = 0;
    if (c < nsc) {
        t0 = c * kChunk;
        n = min(kChunk, se - t0);
    } else if (c < nsc + nsel_ch) {
        const int cpb = b / kChunk;
        const int k = c - nsc, ei = k / cpb;
        const int32_t *srow = a.sel + (int64_t)rowi * a.k_blocks;
        const int e = srow[ei];
        const int prev = ei > 0 ? srow[ei - 1] : -1;
        if (e < 0) return d;
        const bool valid = e < a.max_blocks && (int64_t)e * b >= se && (int64_t)(e + 1) * b <= rs && prev < e;
        if (!valid) {
            if (k % cpb == 0) flag_error(a.status, LSA_ERR_BOUNDS);
            return d;
        }
        t0 = e * b + (k % cpb) * kChunk;
        n = kChunk;
    } else {
        const int blk16 = rs / kChunk + (c - nsc - nsel_ch);
        t0 = max(rs, blk16 * kChunk);
        n = min(L, blk16 * kChunk + kChunk) - t0;
    }
    if (n <= 0) return d;
    const int p = a.pt[(int64_t)r * a.max_blocks + t0 / b];
    if (p < 0 || p >= a.c.num_pages) {
        flag_error(a.status, LSA_ERR_BOUNDS);
        return d;
    }
    d.page = p;
    d.ts = t0 % b;
    d.n = n;
    return d;
}

template <int DK>
struct AttnStream {
    static constexpr int KBYTES = (DK / 64) * 16 * 128;   // one swizzled 16-row K (or V) tile
    static constexpr int NT = DK / 8;                       // output n-tiles (DV = DK)
    static constexpr int CPR = DK / 8;                      // 16-byte chunks per token row
    static_assert(2 * KBYTES <= kStageBytes, "K and V tiles must fit a stage");
    int u_row, u_part, u_nck, u_k;
    ChunkDescV my;          // lane i: chunk i of the current unit
    bool have, ended;
    uint32_t t_next;
};

template <int DK>
__device__ void attn_describe(const FusedArgs &a, AttnStream<DK> &S, int unit)
{
    const int lane = threadIdx.x & 31;
    const int rowi = unit / a.units_per_row, part = unit % a.units_per_row;
    const int r = rowi / a.c.hkv;
    if (a.wait_ready) wait_counter(&a.ready[rowi * kCtr], 1u, a.status, a.spin_budget);
    int L = a.lens[r];
    if (L < 0 || (int64_t)L > (int64_t)a.max_blocks * a.c.b) {
        if (lane == 0 && part == 0 && rowi % a.c.hkv == 0) flag_error(a.status, LSA_ERR_BOUNDS);
        L = 0;
    }
    const int se = min(a.sink, L);
    const int rs = max(L - a.recent, se);
    const int nsc = (se + kChunk - 1) / kChunk;
    const int nsel_ch = a.k_blocks * (a.c.b / kChunk);
    const int nrc = L > rs ? (L + kChunk - 1) / kChunk - rs / kChunk : 0;
    const int nck = nsc + nsel_ch + nrc;
    const int c0 = part * a.chunks_per_unit;
    S.u_nck = max(0, min(nck, c0 + a.chunks_per_unit) - c0);
    S.u_row = rowi;
    S.u_part = part;
    S.u_k = 0;
    S.my = lane < S.u_nck ? chunk_desc_v(a, r, rowi, L, se, rs, nsc, nsel_ch, c0 + lane) : ChunkDescV{-1, 0, 0};
    S.have = true;
}

template <int DK>
__device__ void attn_issue(const FusedArgs &a, AttnStream<DK> &S, Worker &w)
{
    using AS = AttnStream<DK>;
    const int lane = threadIdx.x & 31;
    const int slot = w.issued % kStages;
    if (!S.have) {
        if (S.ended || S.t_next >= (uint32_t)a.total_units) {
            S.ended = true;
            if (lane == 0) w.meta[slot].n = -1;
            cp_async_commit();
            ++w.issued;
            return;
        }
        LSA_TRACE(a, S.t_next, 0);
        attn_describe<DK>(a, S, (int)(S.t_next - (uint32_t)a.attn_base));
        LSA_TRACE(a, S.t_next, 2);
        S.t_next = fetch_ticket(a.ctrl);
    }
    const int k = S.u_k;
    int flags = k == 0 ? 1 : 0;
    int n = 0;
    if (S.u_nck > 0) {
        const int page = __shfl_sync(0xffffffffu, S.my.page, k);
        const int ts = __shfl_sync(0xffffffffu, S.my.ts, k);
        n = __shfl_sync(0xffffffffu, S.my.n, k);
        if (n > 0) {
            const CacheView &c = a.c;
            const int h = S.u_row % c.hkv;
            const uint32_t st = w.ring_s + slot * kStageBytes;
            const uint8_t *kb = c.k + ((int64_t)page * c.kps + (int64_t)h * c.khs + (int64_t)ts * c.kts) * 2;
            const uint8_t *vb = c.v + ((int64_t)page * c.vps + (int64_t)h * c.vhs + (int64_t)ts * c.vts) * 2;
#pragma unroll
            for (int u = 0; u < 16 * AS::CPR / 32; ++u) {
                const int q = lane + 32 * u;
                const int t = q / AS::CPR, ch = q % AS::CPR;
                if (t < n) {
                    cp_async16(st + swizzle_offset(t, ch), kb + (int64_t)t * c.kts * 2 + ch * 16);
                    cp_async16(st + AS::KBYTES + swizzle_offset(t, ch), vb + (int64_t)t * c.vts * 2 + ch * 16);
                }
            }
        }
    }
    const bool last = S.u_nck == 0 || k + 1 == S.u_nck;
    if (last) flags |= 2;
    if (lane == 0) {
        w.meta[slot].n = n;
        w.meta[slot].unit = S.u_row * a.units_per_row + S.u_part;
        w.meta[slot].flags = flags;
    }
    cp_async_commit();
    ++w.issued;
    if (last) S.have = false;
    else ++S.u_k;
}

// The parts of a row are merged by the last one to finish.
template <int DK, int G>
__device__ void attn_merge_row(const FusedArgs &a, int rowi)
{
    const int lane = threadIdx.x & 31;
    const int r = rowi / a.c.hkv, h = rowi % a.c.hkv;
    const int Gt = a.hq / a.c.hkv;
    const int P = a.units_per_row;
    for (int t = lane; t < G * DK / 4; t += 32) {
        const int g = t / (DK / 4), d = (t % (DK / 4)) * 4;
        const int64_t orow = (int64_t)r * a.hq + h * Gt + g;
        const float *lp = a.lse_part + orow * P;
        float M = -INFINITY;
        for (int s = 0; s < P; ++s) M = fmaxf(M, __ldcg(lp + s));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < P; ++s) {
                const float ls = __ldcg(lp + s);
                if (ls == -INFINITY) continue;
                const float f = fast_ex2(ls - M);
                wsum += f;
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.o_part + (orow * P + s) * DK + d));
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
        if (a.lse && d == 0) a.lse[orow] = empty_set ? -INFINITY : (M + fast_lg2(wsum)) * kLn2;
    }
}

template <int DK, int G>
__device__ void attn_phase(const FusedArgs &a, uint32_t t, Worker &w)
{
    using AS = AttnStream<DK>;
    const int lane = threadIdx.x & 31;
    const int rr = lane >> 2, cc = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;
    const int tk = (mi >> 1) * 8 + r8, ck = mi & 1;   // K fragment rows: tokens 0-7/8-15 x dims lo/hi
    const int tv = (mi & 1) * 8 + r8, cv = mi >> 1;   // V (transposed)
    const int Gt = a.hq / a.c.hkv;

    AS S;
    S.have = false;
    S.ended = false;
    S.t_next = t;
    w.issued = w.computed = 0;

    uint32_t qa0[DK / 16], qa2[DK / 16];
    int q_row = -1;
    float m = -INFINITY, l = 0.f;
    float o[AS::NT][4];
#pragma unroll
    for (int nt = 0; nt < AS::NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) attn_issue<DK>(a, S, w);
    while (true) {
        attn_issue<DK>(a, S, w);
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const int slot = w.computed % kStages;
        const StageMeta md = w.meta[slot];
        if (md.n < 0) break;
        ++w.computed;
        const int rowi = md.unit / a.units_per_row, part = md.unit % a.units_per_row;
        const int r = rowi / a.c.hkv, h = rowi % a.c.hkv;
        if (md.flags & 1) {
            if (q_row != rowi) {
                q_row = rowi;
                const bool qok = rr < G;
                const uint16_t *qp = a.q + ((int64_t)r * a.hq + h * Gt + (qok ? rr : 0)) * DK;
#pragma unroll
                for (int ks = 0; ks < DK / 16; ++ks) {
                    qa0[ks] = qok ? *reinterpret_cast<const uint32_t *>(qp + 16 * ks + 2 * cc) : 0u;
                    qa2[ks] = qok ? *reinterpret_cast<const uint32_t *>(qp + 16 * ks + 8 + 2 * cc) : 0u;
                }
            }
            m = -INFINITY;
            l = 0.f;
#pragma unroll
            for (int nt = 0; nt < AS::NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        }
        const int n = md.n;
        if (n > 0) {
            const uint32_t kbase = w.ring_s + slot * kStageBytes;
            const uint32_t vbase = kbase + AS::KBYTES;
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < DK / 16; ++ks) {
                uint32_t b[4];
                ldsm_x4(b, kbase + swizzle_offset(tk, 2 * ks + ck));
                mma_bf16_rows8(s0, qa0[ks], qa2[ks], b[0], b[1]);
                mma_bf16_rows8(s1, qa0[ks], qa2[ks], b[2], b[3]);
            }
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
            for (int nt = 0; nt < AS::NT; ++nt) {
                o[nt][0] *= alpha;
                o[nt][1] *= alpha;
            }
            if (n < kChunk) {   // stale V rows meet zero weights; 0 * NaN must not happen
                for (int q = lane; q < (kChunk - n) * AS::CPR; q += 32) {
                    const int tt = n + q / AS::CPR, ch = q % AS::CPR;
                    *reinterpret_cast<uint4 *>(w.ring + slot * kStageBytes + AS::KBYTES + swizzle_offset(tt, ch)) =
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
        if (md.flags & 2) {
            LSA_TRACE(a, a.attn_base + md.unit, 1);
            // the part is complete: write it (or the row's output when unsplit)
            const int P = a.units_per_row;
            if (rr < G) {
                const int64_t orow = (int64_t)r * a.hq + h * Gt + rr;
                const bool empty_set = !(l > 0.f);
                const float inv = empty_set ? 0.f : 1.f / l;
                if (P == 1) {
#pragma unroll
                    for (int nt = 0; nt < AS::NT; ++nt)
                        *reinterpret_cast<uint32_t *>(a.out + orow * DK + nt * 8 + 2 * cc) =
                            pack_bf16x2(o[nt][0] * inv, o[nt][1] * inv);
                    if (a.lse && cc == 0) a.lse[orow] = empty_set ? -INFINITY : (m + fast_lg2(l)) * kLn2;
                } else {
                    float *dst = a.o_part + (orow * P + part) * DK;
#pragma unroll
                    for (int nt = 0; nt < AS::NT; ++nt)
                        *reinterpret_cast<float2 *>(dst + nt * 8 + 2 * cc) = make_float2(o[nt][0] * inv, o[nt][1] * inv);
                    if (cc == 0) a.lse_part[orow * P + part] = empty_set ? -INFINITY : m + fast_lg2(l);
                }
            }
            if (P > 1) {
                __threadfence();
                __syncwarp();
                uint32_t prev = 0;
                if (lane == 0) prev = atomicAdd(&a.split_done[rowi * kCtr], 1u);
                prev = __shfl_sync(0xffffffffu, prev, 0);
                if (prev == (uint32_t)P - 1) {
                    __threadfence();
                    attn_merge_row<DK, G>(a, rowi);
                    if (lane == 0) a.split_done[rowi * kCtr] = 0;
                }
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
    __syncwarp();
}

// ================================================================== kernel

template <int DK, int HKV, int G>
__global__ void __launch_bounds__(kWarps * 32, 1) k_decode_fused(FusedArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((smem_addr(smem) & 1023u) != 0) {       // the K/V swizzle assumes 1 KB aligned stages
        if (threadIdx.x == 0) flag_error(a.status, LSA_ERR_INVALID_ARG);
        return;
    }
    Worker w;
    w.ring = smem + warp * kWarpBytes;
    w.ring_s = smem_addr(w.ring);
    w.meta = reinterpret_cast<StageMeta *>(smem + kWarps * kWarpBytes + warp * kMetaBytes);

    const uint32_t total = (uint32_t)a.total_units;
    uint32_t t = fetch_ticket(a.ctrl);
    if (t >= total + (uint32_t)a.total_warps && lane == 0) flag_error(a.status, LSA_ERR_INVALID_ARG);
    while (t < total) {
        int id = 0;
        const int kind = unit_kind(a, t, &id);
        if (kind == kScoreUnit) {
            t = score_phase<DK, HKV>(a, t, w);   // returns the first ticket that is not a score unit
        } else if (kind == kTopkUnit) {
            const int row = id, r = row / HKV;
            LSA_TRACE(a, t, 0);
            if (wait_counter(&a.score_done[r * kCtr], (uint32_t)a.score_chunks, a.status, a.spin_budget)) {
                LSA_TRACE(a, t, 2);
                uint32_t *scratch = reinterpret_cast<uint32_t *>(w.ring);   // idle between streams
                if (a.max_blocks <= 32 * 4) warp_topk<4>(a, row, scratch);
                else if (a.max_blocks <= 32 * 16) warp_topk<16>(a, row, scratch);
                else warp_topk<kMaxKpl>(a, row, scratch);
                __syncwarp();
                LSA_TRACE(a, t, 3);
            }
            publish(&a.ready[row * kCtr]);
            LSA_TRACE(a, t, 1);
            t = fetch_ticket(a.ctrl);
        } else {
            attn_phase<DK, G>(a, t, w);            // attention units are the last tickets
            break;
        }
    }

    // the last worker out resets the control counters for the next call
    // (all its lanes; plain stores: nothing else of this launch reads them)
    __threadfence();
    __syncwarp();
    uint32_t done = 0;
    if (lane == 0) done = atomicAdd(&a.ctrl[kCtr], 1u);
    done = __shfl_sync(0xffffffffu, done, 0);
    if (done == (uint32_t)a.total_warps - 1) {
        __threadfence();
        for (int i = lane; i < a.batch; i += 32) a.score_done[i * kCtr] = 0u;
        for (int i = lane; i < a.batch * a.c.hkv; i += 32) {
            a.ready[i * kCtr] = 0u;
            a.split_done[i * kCtr] = 0u;
        }
        if (lane == 0) {
            a.ctrl[0] = 0u;
            a.ctrl[kCtr] = 0u;
        }
    }
}

template <int DK, int HKV, int G>
cudaError_t launch_fused_t(const FusedArgs &a, cudaStream_t s, int sms)
{
    auto kern = k_decode_fused<DK, HKV, G>;
    const int smem = fused_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    FusedArgs b = a;
    const int grid = per_sm * sms;
    b.total_warps = grid * kWarps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, b);
}

}  // namespace

int fused_smem_bytes() { return kWarps * (kWarpBytes + kMetaBytes); }

// Instantiated (head dim, KV heads, group size) combinations.
static bool fused_instance(int dk, int hkv, int g)
{
    if (dk != 64 && dk != 128) return false;
    if (hkv == 1 || hkv == 8) return g == 2 || g == 4 || g == 8;
    return (hkv == 2 || hkv == 4) && g == 4;
}

bool fused_supported(int dk, int dv, int hkv, int group, bool alias, int b, int max_blocks, int k_blocks)
{
    if (alias || dk != dv || b % kChunk != 0 || max_blocks > 32 * kMaxKpl || k_blocks > 32 * kMaxKpl) return false;
    return fused_instance(dk, hkv, group);
}

void fused_plan(int sink, int recent, int b, int k_blocks, int batch, int hkv, int max_blocks, bool scoring,
                FusedPlan *pl)
{
    const int nck = attention_items_max(sink, recent, b, k_blocks, 0);
    pl->units_per_row = (nck + kPartChunks - 1) / kPartChunks;
    pl->chunks_per_unit = (nck + pl->units_per_row - 1) / pl->units_per_row;
    pl->score_blocks = kScoreBlocks;
    pl->score_chunks = scoring ? (max_blocks + kScoreBlocks - 1) / kScoreBlocks : 0;
    pl->score_units = batch * pl->score_chunks;
    pl->attn_base = pl->score_units + (scoring ? batch * hkv : 0);
    pl->total_units = pl->attn_base + batch * hkv * pl->units_per_row;
}

cudaError_t launch_fused(const FusedArgs &a, cudaStream_t s, int sms, bool *unsupported)
{
    *unsupported = false;
    if (a.batch == 0) return cudaSuccess;
    const int G = a.hq / a.c.hkv;
#define LSA_FUSED_CASE(D, H, G_) \
    if (a.c.dk == D && a.c.hkv == H && G == G_) return launch_fused_t<D, H, G_>(a, s, sms);
    LSA_FUSED_CASE(64, 1, 2) LSA_FUSED_CASE(64, 1, 4) LSA_FUSED_CASE(64, 1, 8)
    LSA_FUSED_CASE(64, 2, 4) LSA_FUSED_CASE(64, 4, 4)
    LSA_FUSED_CASE(64, 8, 2) LSA_FUSED_CASE(64, 8, 4) LSA_FUSED_CASE(64, 8, 8)
    LSA_FUSED_CASE(128, 1, 2) LSA_FUSED_CASE(128, 1, 4) LSA_FUSED_CASE(128, 1, 8)
    LSA_FUSED_CASE(128, 2, 4) LSA_FUSED_CASE(128, 4, 4)
    LSA_FUSED_CASE(128, 8, 2) LSA_FUSED_CASE(128, 8, 4) LSA_FUSED_CASE(128, 8, 8)
#undef LSA_FUSED_CASE
    *unsupported = true;
    return cudaSuccess;
}

}  // namespace lsa

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
constexpr int kScoreBlocks = 4;        // blocks per score unit (<= 32: one per lane): one stage
constexpr int kMaxKpl = 64;            // top-k keys per lane (rows of up to 2048 blocks)
constexpr int kPartChunks = 8;         // attention chunks per part (64 KB of K/V at d = 128)
constexpr float kLn2 = 0.693147180559945309f;
constexpr int kCtr = 64;               // words between control counters (256 bytes: one L2 line each)

// Block scores travel from the score units to the top-k warps as
// order-preserving 32-bit keys (larger score, larger key) in a buffer that
// is zero between calls: a key of 0 has not been written yet, so the top-k
// warp needs no counter or fence, it polls its row until no zero is left
// (every key is one 32-bit store).  Blocks that are not candidates get
// kKeyNotCand, the key of -inf; a NaN score gets kKeyNaN (flagged).  Both
// are below every key of a finite score.
constexpr uint32_t kKeyNotCand = 0x007fffffu;   // the key of -inf
constexpr uint32_t kKeyNaN = 1u;

// Per-stage bookkeeping written by a worker's issuing side and read by its
// computing side.
struct StageMeta {
    int n;          // rows staged (-1: end of the stream)
    int unit;       // score: request; attention: row * parts + part
    int flags;      // bit 0: first stage of the unit, bit 1: last stage
    int slot;       // score: the unit's slot in the worker's key buffer
    int j[4];       // score: block index of each staged row
};

constexpr int kMetaBytes = kStages * (int)sizeof(StageMeta);
constexpr int kWarpBytes = kStages * kStageBytes;
constexpr int kScorePageSlots = 512;    // blocks of a CTA's share of the score units
constexpr int kQsReq = 2;               // requests whose query sum a CTA keeps in shared memory
constexpr int kQsFloats = kQsReq * 8 * 128;
constexpr int kPgOffset = kWarps * (kWarpBytes + kMetaBytes);
constexpr int kQsOffset = kPgOffset + kScorePageSlots * 4;
// Block-score keys wait in shared memory until the worker's copies are
// drained: a global store issued while the worker's cp.async copies are in
// flight waits for them, which would empty the ring at every stage.
constexpr int kKeyBufUnits = 20;        // score units whose keys a worker holds: its whole share
constexpr int kKeyOffset = kQsOffset + kQsFloats * 4;
constexpr int kKeyWarpBytes = kKeyBufUnits * (32 * 4 + 8);   // keys, then (unit, mask) per slot
constexpr int kSmemBytes = kKeyOffset + kWarps * kKeyWarpBytes;
static_assert(kScoreBlocks * 8 <= 32, "a unit's keys (blocks x KV heads <= 8) fill one warp-wide row");
static_assert(kKeyBufUnits * (kWarps - 1) >= kScorePageSlots / kScoreBlocks,
              "a streaming warp's whole share of score units fits its key buffer");
static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");

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

// Relaxed (unordered) increment with no reply: a hint for pollers, never
// a guarantee that the data it counts is visible.
__device__ __forceinline__ void red_relaxed_add(uint32_t *p, uint32_t v)
{
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

struct Worker {
    uint8_t *ring;          // kStages stages of kStageBytes
    uint32_t ring_s;        // shared-window address of the ring
    StageMeta *meta;
    int issued, computed;   // stage counters
    uint32_t *tk_ctr;       // the phase's ticket counter
    uint32_t tk_next;       // the next ticket (known)
    uint32_t tk_pend;       // lane 0: the one after it (atomic in flight)
};

// Tickets are taken one ahead: the counter's reply for ticket i+2 is read
// only when ticket i+1 is taken, a whole unit later, so no worker waits on
// the atomic's round trip.  Tickets are unsigned and compared against the
// unit counts before any use, so a counter that was not zero at launch (a
// workspace that broke the zero-fill contract) can only skip work, never
// index out of range.
__device__ __forceinline__ void tickets_init(Worker &w, uint32_t *ctr)
{
    w.tk_ctr = ctr;
    uint32_t t = 0;
    if ((threadIdx.x & 31) == 0) t = atomicAdd(ctr, 1u);
    w.tk_next = __shfl_sync(0xffffffffu, t, 0);
    w.tk_pend = 0;
    if ((threadIdx.x & 31) == 0) w.tk_pend = atomicAdd(ctr, 1u);
}

__device__ __forceinline__ uint32_t take_ticket(Worker &w)
{
    const uint32_t t = w.tk_next;
    w.tk_next = __shfl_sync(0xffffffffu, w.tk_pend, 0);
    if ((threadIdx.x & 31) == 0) w.tk_pend = atomicAdd(w.tk_ctr, 1u);
    return t;
}

// Reads the reply to the outstanding request, so it is complete before the
// worker moves to another counter or leaves.
__device__ __forceinline__ void tickets_done(Worker &w)
{
    const uint32_t last_reply = __shfl_sync(0xffffffffu, w.tk_pend, 0);
    asm volatile("" ::"r"(last_reply));
}

// ================================================================== scores

__device__ __forceinline__ int score_swz(int ch) { return (ch & ~7) | ((ch ^ (ch >> 3)) & 7); }

template <int DK, int HKV>
struct ScoreStream {
    static constexpr int ROWB = HKV * DK * 2;                 // one page's summaries
    static constexpr int NCH = HKV * DK / 8;                  // 16-byte chunks per row
    static constexpr int NI = (NCH + 31) / 32;                // chunks per lane, contiguous
    static constexpr int CPH = DK / 8;                        // chunks per head
    static constexpr int LPH = CPH / NI;                      // lanes per head
    static_assert(kScoreBlocks * ROWB <= kStageBytes, "a unit's summary rows fill one stage");
    static_assert(NCH <= 32 || NCH % 32 == 0, "chunks tile the warp");
    static_assert(CPH % NI == 0 && 32 % LPH == 0, "a lane's chunks lie in one head");

    int u_r, u_j0, u_ncand, u_nst, u_k;   // current unit; lane l describes block u_j0 + l
    uint32_t u_mask;
    int u_page;
    bool have, ended;
    int next, stride, end, u0;            // this worker's units: next, next + stride, ... below end
    int u_slot;                           // the current unit's slot in the key buffer
    const int *s_pg;                      // the CTA's page ids of its units' blocks (-1: not a candidate)
    const float *s_qs;                    // query sums of requests r_first, r_first + 1
    int r_first;
    uint32_t *keys;                       // the worker's key buffer: kKeyBufUnits x 32 keys
    int2 *slots;                          // (unit, candidate mask) of each buffered unit
    int nslots;
    float qs[NI][8];                      // sum of the group's queries, this lane's chunks
    int qs_r;
};

// Writes the buffered keys of the worker's units to the score rows, then
// counts the units in the requests' hint words.
template <int DK, int HKV>
__device__ void score_flush(const FusedArgs &a, ScoreStream<DK, HKV> &S)
{
    const int lane = threadIdx.x & 31;
    __syncwarp();
    const int blk = lane / 8, h = lane % 8;
    for (int k = 0; k < S.nslots; ++k) {
        const int2 um = S.slots[k];
        const int r = um.x / a.score_chunks, j = (um.x % a.score_chunks) * a.score_blocks + blk;
        if (h < HKV && blk < a.score_blocks && ((um.y >> blk) & 1))
            a.scores[((int64_t)r * HKV + h) * a.max_blocks + j] = S.keys[k * 32 + lane];
    }
    __syncwarp();
    for (int k = 0; k < S.nslots; ++k)
        if (lane == 0) red_relaxed_add(&a.score_hint[(S.slots[k].x / a.score_chunks) * kCtr], 1u);
    S.nslots = 0;
    __syncwarp();
}

__device__ __forceinline__ uint32_t score_key(const FusedArgs &a, float s)
{
    if (isnan(s)) {
        flag_error(a.status, LSA_ERR_NAN);
        return kKeyNaN;
    }
    return s == -INFINITY ? kKeyNotCand : float_to_key(s);
}

// Make the worker's next unit the current one: its candidate blocks' page
// ids come from the CTA's table in shared memory.
template <int DK, int HKV>
__device__ void score_finish(const FusedArgs &a, ScoreStream<DK, HKV> &S)
{
    const int lane = threadIdx.x & 31;
    const int unit = S.next;
    S.next += S.stride;
    const int r = unit / a.score_chunks, c = unit % a.score_chunks;
    const int p = lane < a.score_blocks ? S.s_pg[(unit - S.u0) * a.score_blocks + lane] : -1;
    S.u_mask = __ballot_sync(0xffffffffu, p >= 0);
    S.u_ncand = __popc(S.u_mask);
    S.u_nst = S.u_ncand > 0 ? 1 : 0;
    S.u_k = 0;
    S.u_r = r;
    S.u_j0 = c * a.score_blocks;
    S.u_page = p;
    S.have = true;
    // the host admits only shapes whose shares fit (fused_supported); a
    // unit past the buffer is flagged and not scored
    if (S.nslots == kKeyBufUnits) {
        if (lane == 0) flag_error(a.status, LSA_ERR_INVALID_ARG);
        S.u_mask = 0u;
        S.u_ncand = 0;
        S.u_nst = 0;
        S.u_slot = kKeyBufUnits - 1;
        return;
    }
    if (lane == 0) S.slots[S.nslots] = make_int2(unit, (int)S.u_mask);
    S.u_slot = S.nslots++;
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
            if (S.ended || S.next >= S.end) {
                S.ended = true;
                if (lane == 0) w.meta[slot].n = -1;
                cp_async_commit();
                ++w.issued;
                return;
            }
            LSA_TRACE(a, S.next, 0);
            score_finish<DK, HKV>(a, S);
            if (S.u_ncand == 0) {   // nothing to stream
                S.have = false;
                continue;
            }
        }
        // row i of the stage holds block u_j0 + i (non-candidates are not
        // copied); chunk ch of a row goes to 16-byte slot ch ^ ((ch >> 3) & 7)
        // within its 128-byte group, so that the compute's reads (lane l:
        // chunks l * NI ...) hit distinct banks
        const uint32_t st = w.ring_s + slot * kStageBytes;
#pragma unroll
        for (int i = 0; i < kScoreBlocks; ++i) {
            const int p = __shfl_sync(0xffffffffu, S.u_page, i);
            if (p >= 0) {
                const uint8_t *row = reinterpret_cast<const uint8_t *>(a.summ) + (int64_t)p * SS::ROWB;
#pragma unroll
                for (int u = 0; u < SS::NI; ++u) {
                    const int ch = lane + 32 * u;
                    if (ch < SS::NCH) cp_async16(st + i * SS::ROWB + score_swz(ch) * 16, row + ch * 16);
                }
            }
        }
        if (lane == 0) {
            w.meta[slot].n = kScoreBlocks;
            w.meta[slot].unit = S.u_r;
            w.meta[slot].flags = 2 | (int)(S.u_mask << 8);
            w.meta[slot].slot = S.u_slot;
            w.meta[slot].j[0] = S.u_j0;
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
    if (S.qs_r != r && r - S.r_first < kQsReq) {
        S.qs_r = r;
        const float *src = S.s_qs + (r - S.r_first) * HKV * DK;
#pragma unroll
        for (int i = 0; i < SS::NI; ++i) {
            const int ch = lane * SS::NI + i;
#pragma unroll
            for (int e = 0; e < 8; ++e) S.qs[i][e] = ch < SS::NCH ? src[(ch / SS::CPH) * DK + (ch % SS::CPH) * 8 + e] : 0.f;
        }
    }
    if (S.qs_r != r) {   // a request past the CTA's table: sum the queries here
        S.qs_r = r;
        const int Gt = a.hq / HKV;
#pragma unroll
        for (int i = 0; i < SS::NI; ++i) {
            const int ch = lane * SS::NI + i;
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
    const uint32_t mask = (uint32_t)md.flags >> 8;
#pragma unroll
    for (int i = 0; i < kScoreBlocks; ++i) {
        if (!((mask >> i) & 1u)) continue;   // warp-uniform
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < SS::NI; ++c) {
            const int ch = lane * SS::NI + c;
            if (ch < SS::NCH) {
                const uint4 v = *reinterpret_cast<const uint4 *>(st + i * SS::ROWB + score_swz(ch) * 16);
                const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc = __ffma2_rn(make_float2(S.qs[c][2 * e], S.qs[c][2 * e + 1]), bf2_to_f2(wd[e]), acc);
            }
        }
        float part = acc.x + acc.y;
#pragma unroll
        for (int off = SS::LPH / 2; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane % SS::LPH == 0 && lane * SS::NI < SS::NCH)
            S.keys[md.slot * 32 + i * 8 + (lane * SS::NI) / SS::CPH] = score_key(a, part);
    }
#ifdef LSA_FUSED_TRACE
    LSA_TRACE(a, r * a.score_chunks + md.j[0] / a.score_blocks, 1);
#endif
    return true;
}

// CTA prologue of the score phase, one memory round trip for all threads:
// the page id of every block of the CTA's units [u0, u1) after the
// candidate test (-1 otherwise; non-candidates get their key right away),
// and the group query sums of the first kQsReq requests of the share.
template <int DK, int HKV>
__device__ void score_prologue(const FusedArgs &a, int u0, int u1, int *s_pg, float *s_qs)
{
    constexpr int PER = kScorePageSlots / (kWarps * 32);
    constexpr int CPH = DK / 8;
    const int SB = a.score_blocks;
    const int nb = (u1 - u0) * SB;
    const int r_first = u0 / a.score_chunks;
    const int G = a.hq / HKV;
    // loads first
    int pr[PER], lr[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int i = threadIdx.x + k * kWarps * 32;
        pr[k] = -1;
        lr[k] = 0;
        if (i < nb) {
            const int u = u0 + i / SB, r = u / a.score_chunks, j = (u % a.score_chunks) * SB + i % SB;
            lr[k] = a.lens[r];
            if (j < a.max_blocks) pr[k] = a.pt[(int64_t)r * a.max_blocks + j];
        }
    }
    const int qi = threadIdx.x;   // one (request, head, 8 dims) slice per thread
    const int qk = qi / (HKV * CPH), qh = (qi / CPH) % HKV, qd = (qi % CPH) * 8;
    const int qr = r_first + qk;
    const bool qthread = qk < kQsReq && qr < a.batch && qr * a.score_chunks < u1;
    if (qthread) {
        float qacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint16_t *qp = a.q + ((int64_t)qr * a.hq + qh * G) * DK + qd;
        for (int g = 0; g < G; ++g) {
            const uint4 v = *reinterpret_cast<const uint4 *>(qp + (int64_t)g * DK);
            const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = bf2_to_f2(wd[e]);
                qacc[2 * e] += f.x;
                qacc[2 * e + 1] += f.y;
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) s_qs[(qk * HKV + qh) * DK + qd + e] = qacc[e];
    }
    // then the candidate test and the keys of the blocks that are not candidates
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int i = threadIdx.x + k * kWarps * 32;
        if (i >= nb) continue;
        const int u = u0 + i / SB, r = u / a.score_chunks, j = (u % a.score_chunks) * SB + i % SB;
        int L = lr[k];
        const bool len_ok = L >= 0 && (int64_t)L <= (int64_t)a.max_blocks * a.c.b;
        if (!len_ok) {
            if (j == 0) flag_error(a.status, LSA_ERR_BOUNDS);
            L = 0;
        }
        const int se = min(a.sink, L);
        const int rs = max(L - a.recent, se);
        bool cand = j < a.max_blocks && (int64_t)j * a.c.b >= se && (int64_t)(j + 1) * a.c.b <= rs;
        int p = cand ? pr[k] : -1;
        if (cand && (p < 0 || p >= a.c.num_pages)) {
            flag_error(a.status, LSA_ERR_BOUNDS);
            cand = false;
            p = -1;
        }
        s_pg[i] = p;
        if (!cand && j < a.max_blocks) {
#pragma unroll
            for (int h = 0; h < HKV; ++h) a.scores[((int64_t)r * HKV + h) * a.max_blocks + j] = kKeyNotCand;
        }
    }
}

// Streams the score units first, first + stride, ... below end, described
// by the CTA's tables in shared memory (no global loads but the summaries).
template <int DK, int HKV>
__device__ void score_phase(const FusedArgs &a, int first, int stride, int u0, int end, const int *s_pg,
                            const float *s_qs, uint32_t *keys, Worker &w)
{
    ScoreStream<DK, HKV> S;
    S.have = false;
    S.ended = false;
    S.qs_r = -1;
    S.next = first;
    S.stride = stride;
    S.end = end;
    S.u0 = u0;
    S.s_pg = s_pg;
    S.s_qs = s_qs;
    S.r_first = u0 / a.score_chunks;
    S.keys = keys;
    S.slots = reinterpret_cast<int2 *>(keys + kKeyBufUnits * 32);
    S.nslots = 0;
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
    score_flush<DK, HKV>(a, S);
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
                                               int32_t *sel, int32_t *sel_s, Col col)
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
        if (gt || (eq && q < take_eq)) {
            const int32_t cidx = col(e);
            sel[g + min(q, take_eq)] = cidx;
            sel_s[g + min(q, take_eq)] = cidx;
        }
        g += gt;
        q += eq;
    }
}

constexpr int kCompactKeys = 512;   // candidates kept for the narrow bisection (16 per lane)
static_assert(2 * kCompactKeys * 4 + 4 * 32 * kMaxKpl <= kStages * kStageBytes,
              "top-k scratch and the selection live in the worker's ring");

// Top-k of one score row by one warp, ties to the lower block index, output
// ascending and padded with -1.  The row's keys stay in registers (KPL per
// lane).  A lower bound on the threshold comes from the lanes' own top-2:
// a lane holds at least j keys >= its j-th largest, so the smallest j-th
// largest over n_j lanes has >= j n_j keys at or above it.  When at
// most kCompactKeys keys reach the bound they are compacted (in column
// order) into `scratch` (2 * kCompactKeys words of shared memory) and the
// bisection runs over 8 keys per lane; otherwise over all of them.
template <int KPL>
__device__ void warp_topk(const FusedArgs &a, int row, uint32_t *scratch, int32_t *sel_s)
{
    static_assert(KPL % 4 == 0, "keys per lane come in fours");
    const int lane = threadIdx.x & 31;
    const int n = a.max_blocks, k = a.k_blocks;
    uint32_t *srow = a.scores + (int64_t)row * n;
    const int c0 = lane * KPL;
    // Lane l owns columns [l*KPL, (l+1)*KPL).  The row is read (16-byte
    // loads when it starts on a 16-byte boundary, max_blocks % 4 == 0, and
    // the lane's range is complete; scalar loads otherwise) until every key
    // has been written; columns past the row count as written.
    const bool vec = c0 + KPL <= n && (n & 3) == 0;
    uint32_t keys[KPL];
    const long long t0 = clock64();
    unsigned ns = 32;
    // the request's score units count themselves in a hint word: wait for
    // the full count with one-word polls before reading the row
    {
        const uint32_t *hint = &a.score_hint[(row / a.c.hkv) * kCtr];
        uint32_t ok = 1;
        if (lane == 0) {
            unsigned hns = 64;
            while (ld_relaxed(hint) < (uint32_t)a.score_chunks) {
                if (clock64() - t0 > a.spin_budget) {
                    ok = 0;
                    break;
                }
                __nanosleep(hns);
                if (hns < 512) hns <<= 1;
            }
        }
        (void)__shfl_sync(0xffffffffu, ok, 0);
    }
    while (true) {
        if (vec) {
#pragma unroll
            for (int e = 0; e < KPL; e += 4) {
                const uint4 f = __ldcg(reinterpret_cast<const uint4 *>(srow + c0 + e));
                keys[e] = f.x;
                keys[e + 1] = f.y;
                keys[e + 2] = f.z;
                keys[e + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < KPL; ++e) keys[e] = c0 + e < n ? __ldcg(srow + c0 + e) : kKeyNotCand;
        }
        bool missing = false;
#pragma unroll
        for (int e = 0; e < KPL; ++e) missing |= keys[e] == 0u;
        if (!__any_sync(0xffffffffu, missing)) break;
        if (clock64() - t0 > a.spin_budget) {
            if (lane == 0) flag_error(a.status, LSA_ERR_TIMEOUT);
            break;
        }
        __nanosleep(ns);
        if (ns < 512) ns <<= 1;
    }
    // the row is consumed: zero it for the next call
    if (vec) {
#pragma unroll
        for (int e = 0; e < KPL; e += 4) *reinterpret_cast<uint4 *>(srow + c0 + e) = make_uint4(0u, 0u, 0u, 0u);
    } else {
#pragma unroll
        for (int e = 0; e < KPL; ++e)
            if (c0 + e < n) srow[c0 + e] = 0u;
    }
    // keys at or below the key of -inf (not a candidate, NaN, never
    // written) are not candidates: 0
#pragma unroll
    for (int e = 0; e < KPL; ++e) keys[e] = keys[e] > kKeyNotCand ? keys[e] : 0u;
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
            emit_selection<PL>(ck, th, teq, sel, sel_s,
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
    if (keff > 0 && !done) emit_selection<KPL>(keys, thresh, take_eq, sel, sel_s, [&](int e) { return c0 + e; });
    for (int i = keff + lane; i < k; i += 32) {
        sel[i] = -1;
        sel_s[i] = -1;
    }
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

// Chunk-table entries (one per 16-token chunk of a row, written by the
// row's top-k unit): page id in the low word; token offset in the page,
// token count << 16 and the "written" bit 31 in the high word.  An entry of
// 0 has not been written in this call; the attention unit that reads an
// entry sets it back to 0, so the table is all zero between calls.
constexpr uint32_t kTabWritten = 1u << 31;

__device__ __forceinline__ uint64_t tab_pack(int page, int ts, int n)
{
    return (uint64_t)(uint32_t)page | ((uint64_t)(kTabWritten | (uint32_t)ts | ((uint32_t)n << 16)) << 32);
}

__device__ __forceinline__ uint64_t ld_cg_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(v) : "l"(p));
    return v;
}

// Lane-parallel description of every chunk of row `rowi` (request r) from
// its selection sel_s (shared memory, ascending, -1 padded): forced sink
// tokens, the selected blocks in 16-token chunks, forced recent tokens.
__device__ void write_chunk_table(const FusedArgs &a, int r, int rowi, int L, const int32_t *sel_s)
{
    const int lane = threadIdx.x & 31;
    const int b = a.c.b, cpb = b / kChunk;
    if (L < 0 || (int64_t)L > (int64_t)a.max_blocks * b) L = 0;   // flagged by the score units
    const int se = min(a.sink, L);
    const int rs = max(L - a.recent, se);
    const int nsc = (se + kChunk - 1) / kChunk;
    const int nsel_ch = a.k_blocks * cpb;
    const int nrc = L > rs ? (L + kChunk - 1) / kChunk - rs / kChunk : 0;
    const int ncpr = a.units_per_row * a.chunks_per_unit;
    uint64_t *tab = a.ctab + (int64_t)rowi * ncpr;
    for (int c = lane; c < ncpr; c += 32) {
        int t0 = 0, n = 0;
        if (c < nsc) {
            t0 = c * kChunk;
            n = min(kChunk, se - t0);
        } else if (c < nsc + nsel_ch) {
            const int k = c - nsc, e = sel_s[k / cpb];
            if (e >= 0) {
                t0 = e * b + (k % cpb) * kChunk;
                n = kChunk;
            }
        } else if (c < nsc + nsel_ch + nrc) {
            const int blk16 = rs / kChunk + (c - nsc - nsel_ch);
            t0 = max(rs, blk16 * kChunk);
            n = min(L, blk16 * kChunk + kChunk) - t0;
        }
        int p = -1;
        if (n > 0) {
            p = a.pt[(int64_t)r * a.max_blocks + t0 / b];
            if (p < 0 || p >= a.c.num_pages) {
                flag_error(a.status, LSA_ERR_BOUNDS);
                n = 0;
                p = -1;
            }
        }
        tab[c] = tab_pack(p, n > 0 ? t0 % b : 0, max(n, 0));
    }
}

template <int DK>
struct AttnStream {
    static constexpr int KBYTES = (DK / 64) * 16 * 128;   // one swizzled 16-row K (or V) tile
    static constexpr int NT = DK / 8;                       // output n-tiles (DV = DK)
    static constexpr int CPR = DK / 8;                      // 16-byte chunks per token row
    static_assert(2 * KBYTES <= kStageBytes, "K and V tiles must fit a stage");
    int u_row, u_part, u_nck, u_k;
    uint32_t u_mask;        // lanes whose chunk is streamed (non-empty)
    ChunkDescV my;          // lane i: chunk i of the current unit
    bool have, ended;
    int nx_unit;            // next unit (-1: none); with a chunk table its entries are in flight
    uint64_t nx_tab;
};

// Start describing attention unit `unit`: with a chunk table, issue the
// loads of its entries now (they are read one unit later).
template <int DK>
__device__ __forceinline__ void attn_prefetch(const FusedArgs &a, AttnStream<DK> &S, int unit)
{
    const int lane = threadIdx.x & 31;
    S.nx_unit = unit;
    S.nx_tab = 0;
    if (a.ctab && lane < a.chunks_per_unit) {
        const int rowi = unit / a.units_per_row, part = unit % a.units_per_row;
        S.nx_tab = ld_cg_u64(a.ctab + ((int64_t)rowi * a.units_per_row + part) * a.chunks_per_unit + lane);
    }
}

// Make the prefetched unit current.  With a chunk table: if some entry was
// not yet written when it was loaded, wait for the row's top-k and load it
// again; then clear the entries.  Without one (attention over the caller's
// selection): describe the chunks from the selection and the page table.
template <int DK>
__device__ void attn_finish(const FusedArgs &a, AttnStream<DK> &S)
{
    const int lane = threadIdx.x & 31;
    const int unit = S.nx_unit;
    const int rowi = unit / a.units_per_row, part = unit % a.units_per_row;
    S.u_row = rowi;
    S.u_part = part;
    S.u_k = 0;
    ChunkDescV d{-1, 0, 0};
    if (a.ctab) {
        const bool mine = lane < a.chunks_per_unit;
        uint64_t *ent = a.ctab + ((int64_t)rowi * a.units_per_row + part) * a.chunks_per_unit + lane;
        uint64_t e = S.nx_tab;
        // entries not yet written when they were prefetched: poll them
        const long long t0 = clock64();
        unsigned ns = 64;
        while (__any_sync(0xffffffffu, mine && !((uint32_t)(e >> 32) & kTabWritten))) {
            if (clock64() - t0 > a.spin_budget) {
                if (lane == 0) flag_error(a.status, LSA_ERR_TIMEOUT);
                break;
            }
            __nanosleep(ns);
            if (ns < 1024) ns <<= 1;
            if (mine) e = ld_cg_u64(ent);
        }
        if (mine) {
            const uint32_t hi = (uint32_t)(e >> 32);
            if (hi & kTabWritten) {
                d.page = (int)(uint32_t)e;
                d.ts = (int)(hi & 0xffffu);
                d.n = (int)((hi >> 16) & 0x7fffu);
            }
            *ent = 0ull;   // consumed: the table is zero again for the next call
        }
    } else {
        const int r = rowi / a.c.hkv;
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
        const int cnt = max(0, min(nck, c0 + a.chunks_per_unit) - c0);
        if (lane < cnt) d = chunk_desc_v(a, r, rowi, L, se, rs, nsc, nsel_ch, c0 + lane);
    }
    const bool valid = d.n > 0;
    S.u_mask = __ballot_sync(0xffffffffu, valid);
    S.u_nck = __popc(S.u_mask);
    S.my = d;
    S.have = true;
    S.nx_unit = -1;
}

template <int DK>
__device__ void attn_issue(const FusedArgs &a, AttnStream<DK> &S, Worker &w)
{
    using AS = AttnStream<DK>;
    const int lane = threadIdx.x & 31;
    const int slot = w.issued % kStages;
    if (!S.have) {
        if (S.ended || S.nx_unit < 0) {
            S.ended = true;
            if (lane == 0) w.meta[slot].n = -1;
            cp_async_commit();
            ++w.issued;
            return;
        }
        attn_finish<DK>(a, S);
        LSA_TRACE(a, a.attn_base + S.u_row * a.units_per_row + S.u_part, 2);
        const uint32_t t = take_ticket(w);
        if (t < (uint32_t)(a.total_units - a.attn_base)) {
            LSA_TRACE(a, a.attn_base + t, 0);
            attn_prefetch<DK>(a, S, (int)t);
        }
    }
    const int k = S.u_k;
    int flags = k == 0 ? 1 : 0;
    int n = 0;
    if (S.u_nck > 0) {
        const bool v = (S.u_mask >> lane) & 1u;
        const int pos = __popc(S.u_mask & ((1u << lane) - 1u));
        const int src = __ffs(__ballot_sync(0xffffffffu, v && pos == k)) - 1;
        const int page = __shfl_sync(0xffffffffu, S.my.page, src);
        const int ts = __shfl_sync(0xffffffffu, S.my.ts, src);
        n = __shfl_sync(0xffffffffu, S.my.n, src);
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
    w.issued = w.computed = 0;
    LSA_TRACE(a, a.attn_base + t, 0);
    attn_prefetch<DK>(a, S, (int)t);

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

    // The last warp of every CTA selects: it takes the rows blockIdx.x,
    // blockIdx.x + gridDim.x, ... and for each polls the row's score keys
    // until the score units have written them all, runs the top-k and
    // writes the row's chunk table.  The other warps stream the score units.
    // Then every warp streams attention units (tickets taken
    // one ahead); an attention unit polls its chunk-table entries.  Score
    // units never wait, and a selecting warp holds no other unit, so every
    // wait ends.
    uint32_t *attn_ctr = a.ctrl + 2 * kCtr;
    const uint32_t rows = (uint32_t)(a.batch * a.c.hkv);
    const uint32_t attn_units = (uint32_t)(a.total_units - a.attn_base);
    if (a.score_units > 0) {
        // the CTA's contiguous share [u0, u1) of the (request-major) score
        // units, dealt round-robin to its streaming warps
        const int u0 = (int)((int64_t)a.score_units * blockIdx.x / gridDim.x);
        const int u1 = (int)((int64_t)a.score_units * (blockIdx.x + 1) / gridDim.x);
        int *s_pg = reinterpret_cast<int *>(smem + kPgOffset);
        float *s_qs = reinterpret_cast<float *>(smem + kQsOffset);
        score_prologue<DK, HKV>(a, u0, u1, s_pg, s_qs);
        __syncthreads();
        if (warp < kWarps - 1) {
            uint32_t *keys = reinterpret_cast<uint32_t *>(smem + kKeyOffset + warp * kKeyWarpBytes);
            score_phase<DK, HKV>(a, u0 + warp, kWarps - 1, u0, u1, s_pg, s_qs, keys, w);
        } else {
            for (uint32_t row = blockIdx.x; row < rows; row += gridDim.x) {
                const int r = (int)row / HKV;
                LSA_TRACE(a, a.score_units + row, 0);
                const int L = a.lens[r];
                // the worker's ring is idle: compaction scratch, then the
                // selection for the chunk table
                uint32_t *scratch = reinterpret_cast<uint32_t *>(w.ring);
                int32_t *sel_s = reinterpret_cast<int32_t *>(scratch + 2 * kCompactKeys);
                if (a.max_blocks <= 32 * 4) warp_topk<4>(a, (int)row, scratch, sel_s);
                else if (a.max_blocks <= 32 * 16) warp_topk<16>(a, (int)row, scratch, sel_s);
                else warp_topk<kMaxKpl>(a, (int)row, scratch, sel_s);
                __syncwarp();
                LSA_TRACE(a, a.score_units + row, 3);
                write_chunk_table(a, r, (int)row, L, sel_s);
                __syncwarp();
                LSA_TRACE(a, a.score_units + row, 1);
            }
        }
    }
    tickets_init(w, attn_ctr);
    {
        const uint32_t t = take_ticket(w);
        // a worker requests at most three tickets past the last unit (two
        // at init, one with its first take): a larger first ticket means the
        // counters did not start at zero
        if (t >= attn_units + 3u * (uint32_t)a.total_warps && lane == 0) flag_error(a.status, LSA_ERR_INVALID_ARG);
        if (t < attn_units) attn_phase<DK, G>(a, t, w);
    }
    tickets_done(w);

    // the last worker out resets the control counters for the next call
    // (all its lanes; plain stores: nothing else of this launch reads them).
    // The reply to the worker's last ticket request is read first, so that
    // request is complete before the worker leaves.
    __threadfence();
    __syncwarp();
    uint32_t done = 0;
    if (lane == 0) done = atomicAdd(&a.ctrl[kCtr], 1u);
    done = __shfl_sync(0xffffffffu, done, 0);
    if (done == (uint32_t)a.total_warps - 1) {
        __threadfence();
        for (int i = lane; i < a.batch * a.c.hkv; i += 32) a.split_done[i * kCtr] = 0u;
        for (int i = lane; i < a.batch; i += 32) a.score_hint[i * kCtr] = 0u;
        if (lane < 3) a.ctrl[lane * kCtr] = 0u;   // score tickets, leave counter, attention tickets
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

int fused_smem_bytes() { return kSmemBytes; }

// Instantiated (head dim, KV heads, group size) combinations.
static bool fused_instance(int dk, int hkv, int g)
{
    if (dk != 64 && dk != 128) return false;
    if (hkv == 1 || hkv == 8) return g == 2 || g == 4 || g == 8;
    return (hkv == 2 || hkv == 4) && g == 4;
}

bool fused_supported(int dk, int dv, int hkv, int group, bool alias, int b, int max_blocks, int k_blocks, int batch,
                     int sms)
{
    if (alias || dk != dv || b % kChunk != 0 || max_blocks > 32 * kMaxKpl || k_blocks > 32 * kMaxKpl) return false;
    // a CTA's share of the score units must fit its page-id table (the grid
    // has at least one CTA per SM)
    const int64_t units = (int64_t)batch * ((max_blocks + kScoreBlocks - 1) / kScoreBlocks);
    if (sms <= 0 || (units + sms - 1) / sms * kScoreBlocks > kScorePageSlots) return false;
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

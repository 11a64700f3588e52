// Internal declarations shared by the translation units of liblsa.so:
// kernel argument blocks and the launchers each .cu file provides to the
// C-ABI layer (api.cu).  Not installed; the public interface is lsa.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/lsa.h"

namespace lsa {

// Tokens per staged item of the attention kernels.  Block sizes must be
// multiples of it, so an item never crosses a page.
constexpr int kChunk = 16;

// Default budget of a bounded wait, in SM clock cycles (about 1 s).
constexpr long long kSpinBudget = 2000000000LL;

// A paged cache as the kernels see it: byte pointers, element strides.
// x / d for 0 <= x < 2^31 as one multiply-high and a shift (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994).
// With l = ceil(log2 d) and m = ceil(2^(31+l) / d): m < 2^32, and
// x m / 2^(31+l) = x / d + x e / (d 2^(31+l)) with 0 <= e < d, where the
// second term is below 2^-l <= 1/d, too small to carry floor(x / d) over
// the next integer; so floor(x / d) = floor(x m / 2^(31+l)).  d = 1: s = -1.
struct FastDiv {
    uint32_t d, m;
    int32_t s;   // l - 1
};

inline FastDiv make_fastdiv(uint32_t d)
{
    FastDiv f;
    f.d = d < 1 ? 1 : d;
    int l = 0;
    while ((1ull << l) < f.d) ++l;
    if (f.d == 1) {
        f.m = 0;
        f.s = -1;
    } else {
        f.m = (uint32_t)(((1ull << (31 + l)) + f.d - 1) / f.d);
        f.s = l - 1;
    }
    return f;
}

__host__ __device__ __forceinline__ uint32_t fdiv(uint32_t x, const FastDiv &f)
{
#ifdef __CUDA_ARCH__
    return f.s < 0 ? x : __umulhi(x, f.m) >> f.s;
#else
    return f.s < 0 ? x : (uint32_t)(((uint64_t)x * f.m) >> 32) >> f.s;
#endif
}

__host__ __device__ __forceinline__ uint32_t fmodu(uint32_t x, const FastDiv &f) { return x - fdiv(x, f) * f.d; }

// LSA_PDL=1: every kernel is launched as a programmatic dependent (off by
// default: with the wait at the top of every kernel it saved nothing on the
// B=16 x 32K step, 38.4 vs 38.4 us, and with some kernel mixes cost time,
// 59.7 vs 38.7 us, as early-launched CTAs held SMs the running kernel could
// use).  LSA_PDL=0: no kernel is, not even the decode step's attention
// kernel, which by default is (it sets up before its wait).
inline int pdl_mode()
{
    static const int m = [] {
        const char *e = getenv("LSA_PDL");
        if (!e) return 1;
        if (strcmp(e, "0") == 0) return 0;
        return strcmp(e, "1") == 0 ? 2 : 1;
    }();
    return m;
}
inline bool pdl_enabled() { return pdl_mode() == 2; }
inline bool pdl_step_dependent() { return pdl_mode() >= 1; }

struct CacheView {
    const uint8_t *k;
    const uint8_t *v;
    int64_t kps, khs, kts;      // key strides (elements)
    int64_t vps, vhs, vts;      // value strides (elements)
    int32_t num_pages, b, hkv, dk, dv;
    int32_t e4m3;               // keys are e4m3 bytes with per-token scales
    const float *kscale;
    int64_t sps, shs;           // scale strides (elements); token stride 1
    int32_t v_alias;            // V = K[..., :dv]
};

struct SummaryArgs {
    CacheView c;
    const int32_t *pt;
    int32_t *lens;              // read-only for build; incremented by append
    int32_t batch, max_blocks;
    uint16_t *summ;             // [num_pages, hkv, dk] bf16
    const uint16_t *k_new;      // append only: [batch, hkv, dk]
    const uint16_t *v_new;      // append only: [batch, hkv, dv]
    uint32_t *status;
};

struct ScoreArgs {
    const uint16_t *q;          // [B, Hq, dk]
    const uint16_t *summ;       // [num_pages, hkv, dk]
    const int32_t *pt;
    const int32_t *lens;
    int32_t batch, hq, hkv, dk, b, num_pages, max_blocks;
    int32_t sink, recent;
    int32_t chunk;              // blocks per CTA (score_chunk)
    float *scores;              // [B, hkv, max_blocks]
    uint32_t *status;
};

struct TopkArgs {
    const float *scores;        // [rows, cols]
    const int32_t *num_cols;    // [rows] or NULL
    int32_t rows, cols, k;
    int32_t *idx;               // [rows, k]
    // Optional remap of column -> token position for the fine pass:
    // token = cand[row*ncand + col / b] * b + col % b.
    const int32_t *cand;
    int32_t ncand, b;
    uint32_t *status;
    // approx != 0: the stochastic early exit (the boundary bucket sampled
    // with splitmix64(seed, row + 1) instead of ranked)
    int32_t approx;
    uint64_t seed;
};

struct FineArgs {
    const uint16_t *q;          // [B, Hq, dk]
    CacheView ic;               // e4m3 index cache
    const int32_t *pt;
    const int32_t *lens;
    const int32_t *cand;        // [B, hkv, ncand] ascending, -1 padded
    int32_t batch, hq, max_blocks, ncand;
    float *fscores;             // [B*hkv, ncand*b]
    uint32_t *status;
    // the coarse-to-fine step's cluster kernel (c2f_fine.cu): it selects
    // the top ncand blocks of the coarse score rows coarse [B, max_blocks]
    // itself (written to cand_out [B, ncand] if not NULL), rescores their
    // tokens and writes the top tok_k into tok_idx [B, tok_k] (token
    // positions, ascending, -1 padded)
    const float *coarse;
    int32_t *cand_out;
    int32_t tok_k;
    int32_t *tok_idx;
    // indexer head weights [B, Hq] (NULL: the head-sum score): the fine
    // score is then sum_g w[r,g] ReLU(q_g . k_t) (weighted-ReLU kernel)
    const float *weights;
};

// PQ32 coarse-to-fine (pq.cu): PQ32 codes of the index keys, their
// coarse scores (LeanSparse Eq. 6 with the codebook centroids), the top-C
// coarse candidates, the miss filter and the exact rescoring.
struct PqArgs {
    const uint16_t *q;          // [B, Hq, 128] bf16
    const float *weights;       // [B, Hq] indexer head weights
    CacheView ic;               // e4m3 index cache, one KV head, dk = 128
    const uint8_t *codes;       // [num_pages, 1, b, 32]
    const uint16_t *codebook;   // [32, 256, 4] bf16
    const uint8_t *hit;         // [num_pages, 1, b] 1 = key cached, or NULL (all cached)
    const int32_t *pt;
    const int32_t *lens;
    int32_t batch, hq, max_blocks, sink, recent;
    int32_t ncand, tok_k;       // C coarse candidates, k final tokens
    float *coarse;              // [B, max_blocks * b] coarse scores (-inf: not a candidate)
    uint32_t *row_ext;          // [B][2] largest score key, complemented smallest (zero between calls)
    uint32_t *hist;             // [B][kPqBins] bucket counts of the coarse scores (zero between calls)
    int32_t *cand_out;          // [B, ncand] coarse candidates, ascending, -1 padded (or NULL)
    int32_t *tok_idx;           // [B, tok_k] selected token positions, ascending, -1 padded
    uint32_t *status;
    long long spin_budget;
    uint8_t *codes_out;         // encoding: [num_pages, 1, b, 32]
    FastDiv fd_b, fd_tpr;       // coarse scores: block size, 128-token tiles per request
};

constexpr int kPqBins = 2048;

struct AttnArgs {
    const uint16_t *q;          // [B, Hq, dk]
    CacheView c;
    const int32_t *pt;
    const int32_t *lens;
    const int32_t *idx;         // [B, hkv, nsel]
    int32_t batch, hq, max_blocks, nsel, token_mode;
    int32_t sink, recent;
    float scale_log2;           // softmax scale * log2(e)
    int32_t splits, items_per_split, nsub;
    // even split of all rows' item slots over fl_ctas CTAs (attention_flat.cu):
    // fl_ns item slots per row, fl_total = rows * fl_ns, at most fl_parts
    // CTAs per row; row_done: one counter per row, zero between calls.
    // The host keeps (fl_total + 1) * fl_ctas below 2^32, so the split's
    // index arithmetic fits 32 bits.
    int32_t fl_ns, fl_ctas, fl_parts;
    int64_t fl_total;
    uint32_t *row_done;
    // selection made by the attention kernel itself from fp32 score rows
    // [B*hkv, sel_cols] (NULL: read idx); sel_write: where it writes the
    // selection out [B*hkv, nsel], or NULL
    const float *sel_scores;
    int32_t sel_cols;
    // reciprocals of the run-time divisors: block size b, 16-token items per
    // block, KV heads, query subgroups per KV head, and (even split) item
    // slots per row, CTAs and items in all; gsize = hq / hkv
    FastDiv fd_b, fd_cpb, fd_hkv, fd_nsub, fd_ns, fd_nc, fd_total;
    int32_t gsize;
    // pdl_early: launched right after the score kernel of the same step on
    // the same stream, as a programmatic dependent.  Everything before that
    // score kernel had completed when it let this kernel launch, so q,
    // lens and the page table are final and the kernel reads them (and
    // sets up) before it waits for the score rows.
    int32_t pdl_early;
    int32_t *sel_write;
    float *o_part;              // [B*Hq, splits or fl_parts, dv]
    float *lse_part;            // [B*Hq, splits or fl_parts]   log2 domain
    uint16_t *out;              // [B, Hq, dv] bf16     (splits == 1)
    float *lse;                 // [B, Hq] natural log or NULL
    uint32_t *status;
    long long spin_budget;
    // tcgen05 kernel: merge the row's tiles inside the kernel (every CTA of
    // the grid resident at once): each tile CTA adds 1 to mrg_arrive[row],
    // waits (bounded) for it to reach the tile count, merges a slice of the
    // row's outputs, then adds 1 to mrg_done[row]; the last resets both
    int32_t merge_in_kernel;
    uint32_t *mrg_arrive, *mrg_done;
};

// A staged item: a run of token rows within one page (n > 0), nothing to
// attend (n == 0), or a list of single tokens resolved per row (n == -1).
struct ItemDesc {
    int32_t page;
    int16_t ts;
    int16_t n;
};

// Row multipliers of the 2-D [rows, dim] views the tensor-core attention
// kernel loads K and V tiles from: row = page*page_rows + head*head_rows + slot.
struct TcRows {
    int64_t k_page_rows, k_head_rows, v_page_rows, v_head_rows;
};

struct MergeArgs {
    const float *o_part;
    const float *lse_part;
    int32_t rows, splits, dv;
    uint16_t *out;
    float *lse;
};

// ---- launchers (return a cudaError_t from the launch; LSA_ERR_UNSUPPORTED
// is reported through *unsupported when no kernel instance fits the shape)
cudaError_t launch_build_summaries(const SummaryArgs &a, cudaStream_t s, bool quest);
cudaError_t launch_append(const SummaryArgs &a, cudaStream_t s, bool quest, bool *unsupported);
cudaError_t launch_score(const ScoreArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_score_quest(const ScoreArgs &a, cudaStream_t s, bool *unsupported);
bool score_quest_supported(int dk, int hkv, int group);
cudaError_t launch_topk(const TopkArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_fine_scores(const FineArgs &a, cudaStream_t s, bool *unsupported);
bool c2f_fine_supported(const CacheView &iv, int hq, int max_blocks, int ncand, int tok_k, bool weighted);
bool pq_supported(const CacheView &iv, int hq, int max_blocks, int ncand, int tok_k);
cudaError_t launch_pq_encode(const PqArgs &a, cudaStream_t s);
cudaError_t launch_pq_scores(const PqArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_pq_select(const PqArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_c2f_fine(const FineArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s);
int attention_flat_ctas_per_sm();
int attention_flat_warps();
int attention_flat_max_items_per_warp();
bool attention_flat_can_select(int cols, int k);
cudaError_t launch_attention_flat(const AttnArgs &a, int gs, cudaStream_t s, bool *unsupported);
bool launch_topk_fast(const TopkArgs &a, cudaStream_t s, cudaError_t *err);
cudaError_t launch_attention_tc(const AttnArgs &a, int gs, cudaStream_t s, bool *unsupported);
int attention_tc_group(int dk, int dv, int group, bool alias, bool token_mode, const CacheView &v);
int attention_tc_max_items_per_split(int dk);
bool attention_umma_supported(int dk, int dv, int group, bool alias);
int attention_umma_items_per_tile();
int attention_umma_ctas_per_sm(int dk, int dv, bool alias);
cudaError_t launch_attention_umma(const AttnArgs &a, cudaStream_t s, bool *unsupported);

// Shape support queries used by the planner.
bool score_supported(int dk, int hkv);
bool attention_supported(int dk, int dv, int group, bool alias, int *sub_group);
int attention_items_max(int sink, int recent, int b, int nsel, int token_mode);
int attention_max_items_per_split(int dk, int dv, bool alias, int token_mode);
int topk_max_cols();
int score_chunk(int batch, int max_blocks, int sms);

}  // namespace lsa

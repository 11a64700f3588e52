// Internal declarations shared by the translation units of liblsa.so:
// kernel argument blocks and the launchers each .cu file provides to the
// C-ABI layer (api.cu).  Not installed; the public interface is lsa.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/lsa.h"

namespace lsa {

// Tokens per staged item of the attention kernels.  Block sizes must be
// multiples of it, so an item never crosses a page.
constexpr int kChunk = 16;

// Default budget of a bounded wait, in SM clock cycles (about 1 s).
constexpr long long kSpinBudget = 2000000000LL;

// A paged cache as the kernels see it: byte pointers, element strides.
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
};

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
    float *o_part;              // [B*Hq, splits, dv]   (splits > 1)
    float *lse_part;            // [B*Hq, splits]       log2 domain
    uint16_t *out;              // [B, Hq, dv] bf16     (splits == 1)
    float *lse;                 // [B, Hq] natural log or NULL
    uint32_t *status;
    long long spin_budget;
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
cudaError_t launch_build_summaries(const SummaryArgs &a, cudaStream_t s);
cudaError_t launch_append(const SummaryArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_score(const ScoreArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_topk(const TopkArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_fine_scores(const FineArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t s, bool *unsupported);
cudaError_t launch_merge(const MergeArgs &a, cudaStream_t s);

// Shape support queries used by the planner.
bool score_supported(int dk, int hkv);
bool attention_supported(int dk, int dv, int group, bool alias, int *sub_group);
int attention_items_max(int sink, int recent, int b, int nsel, int token_mode);
int topk_max_cols();

}  // namespace lsa

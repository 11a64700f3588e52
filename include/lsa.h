/*
 * lsa.h -- block-sparse decode-step attention over a paged KV cache.
 *
 * C ABI of liblsa.so.  One decode step of block top-k sparse attention:
 *
 *   1. summaries  k_bar_j = mean key of the b tokens of block j, built once
 *                 when the block fills and reused at every later step
 *                 (Vortex blog post, "Block top-k attention", Figure 1 and
 *                 the block top-k equation; forward_cache of the vFlow
 *                 listing in "Writing an algorithm: vFlow").
 *   2. scores     s_j = q . k_bar_j, summed over the query heads of one KV
 *                 head's GQA group (same equation; the vFlow indexer reduces
 *                 the GeMM of summaries and queries over the head dimension).
 *   3. selection  I = top-k_j(s_j) per (request, KV head), ties to the lower
 *                 block index, with sink tokens and a recent window always
 *                 attended (ByteCross, Figure 1 caption and Appendix A
 *                 "Scored selection"; Vortex cites StreamingLLM for this).
 *   4. attention  o = softmax(q K_T^T * scale) V_T over the attended tokens
 *                 T = forced U selected blocks, split into parts whose partial
 *                 results are merged by log-sum-exp (ByteCross, Appendix A:
 *                 the sink call and the window call are merged by
 *                 log-sum-exp; split-K decode attention, Section 4.4).
 *   Coarse-to-fine variant (LeanSparse, Section 5 "Coarse-to-fine decode
 *   indexing", Figure 9): a coarse top-C over block summaries of FP8 index
 *   keys, then exact rescoring of every token of those C blocks with its FP8
 *   e4m3 key and fp32 scale (132 bytes per 128-d key), keeping the top tokens.
 *
 * Conventions for every call
 *   - All pointers named as device pointers must be device memory of the
 *     current CUDA device; host pointers are read during the call only.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *     unless stated otherwise.  No call allocates device memory; scratch
 *     comes from the caller's `workspace`.
 *   - The caller owns every buffer; no pointer is retained after return.
 *   - Host-side argument checks return a status immediately and launch
 *     nothing.  Data errors found on the device (page ids out of range,
 *     invalid selections, NaN scores, wait timeouts) are recorded in a
 *     per-device status word and never fault: the offending access is
 *     skipped.  Read it with lsa_get_device_status().
 *   - Token positions and block indices are logical (per request); the page
 *     table maps logical block j of request r to physical page
 *     page_table[r * max_blocks + j].  Pages may be shared between requests
 *     (prefix sharing); summaries are stored per physical page, so a shared
 *     page has one summary (Vortex, Figure 2 and "Running it: vTensor": named
 *     cache entries live in pages managed by the KV allocator).
 *   - seq_lens[r] counts the tokens of request r in the cache, the current
 *     step's token included (ByteCross, Appendix A: each step appends its own
 *     key and value before reading).
 */
#ifndef LSA_H
#define LSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *lsa_stream_t;

typedef enum lsa_status {
    LSA_OK = 0,
    LSA_ERR_INVALID_ARG = 1,  /* bad pointer, size, stride or alignment        */
    LSA_ERR_UNSUPPORTED = 2,  /* valid but not built (head dim, group size...)  */
    LSA_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than required        */
    LSA_ERR_BOUNDS = 4,       /* device: page id / index / length out of range  */
    LSA_ERR_TIMEOUT = 5,      /* device: a bounded wait gave up                 */
    LSA_ERR_CUDA = 6,         /* a CUDA runtime call failed                     */
    LSA_ERR_NAN = 7           /* device: a NaN score was skipped                */
} lsa_status;

typedef enum lsa_summary_kind {
    LSA_SUMMARY_MEAN = 0,     /* one mean key per block: [P, Hkv, dk]           */
    LSA_SUMMARY_MINMAX = 1    /* Quest: max and min keys: [P, Hkv, 2, dk]       */
} lsa_summary_kind;

typedef enum lsa_key_format {
    LSA_KEYS_BF16 = 0,        /* keys are bf16                                  */
    LSA_KEYS_E4M3 = 1         /* keys are FP8 e4m3 bytes + one fp32 scale/token */
} lsa_key_format;

/* A paged cache.  Element (page p, KV head h, token slot t, dim i) of K is at
 * k + p*k_page_stride + h*k_head_stride + t*k_token_stride + i, likewise V.
 * Strides are in elements.  Requirements: the innermost dim is contiguous;
 * pointers and every stride in bytes are multiples of 16; dk and dv in bytes
 * are multiples of 16.
 *   v == k with v strides equal to k strides and dv <= dk is a latent cache
 *   whose values are the first dv dims of the keys (MLA-shaped; Vortex,
 *   "Designing for a new architecture"); K bytes are then read once.
 * An index cache (coarse-to-fine) has key_format = LSA_KEYS_E4M3, k = the
 * e4m3 bytes, v = NULL, dv = 0, and k_scale[p*scale_page_stride +
 * h*scale_head_stride + t] = the fp32 scale of that token's key: the key's
 * value is scale * e4m3(byte). */
typedef struct lsa_cache {
    void *k;
    void *v;
    int64_t k_page_stride, k_head_stride, k_token_stride;
    int64_t v_page_stride, v_head_stride, v_token_stride;
    int32_t num_pages, block_size, num_kv_heads, dk, dv;
    int32_t key_format;                 /* lsa_key_format                  */
    const float *k_scale;               /* LSA_KEYS_E4M3 only              */
    int64_t scale_page_stride, scale_head_stride;
} lsa_cache;

/* Per-step parameters.  Forced tokens: F = [0, min(sink, L)) U
 * [max(L - recent, min(sink, L)), L).  Candidates: full blocks (j+1)*b <= L
 * none of whose tokens is in F.  The token budget of a step is
 * |F| + k_blocks * block_size (single stage) or |F| + c2f_tokens
 * (coarse-to-fine). */
typedef struct lsa_params {
    int32_t batch;            /* B requests                                    */
    int32_t num_q_heads;      /* Hq, a multiple of num_kv_heads; query head g
                                 belongs to KV head g / (Hq / Hkv)              */
    int32_t max_blocks;       /* page-table row length                         */
    int32_t k_blocks;         /* scored blocks selected per (request, KV head) */
    int32_t sink_tokens;
    int32_t recent_tokens;
    float softmax_scale;      /* <= 0 selects 1/sqrt(dk)                        */
    int32_t c2f_candidates;   /* > 0: coarse-to-fine with C candidate blocks    */
    int32_t c2f_tokens;       /* tokens kept by the fine pass                   */
    int32_t num_splits;       /* split-K parts per (request, KV head); 0 = auto */
    int32_t summary_kind;     /* lsa_summary_kind of the summaries passed in    */
    /* Coarse-to-fine fine score.  NULL: the head sum of dot products (as for
     * block scores).  Else device fp32 [batch, num_q_heads] indexer head
     * weights w, and the fine score of token t is the indexer's weighted
     * head aggregation sum_g w[r,g] * max(0, q[r,g,:] . k_t), k_t = scale_t
     * * e4m3(k8_t) (LeanSparse, Section 5, Eq. 6, on the exact keys);
     * needs 64 query heads per KV head. */
    const float *fine_head_weights;
    /* PQ32 coarse-to-fine (LeanSparse, Section 5: "Approximate scoring with
     * PQ" and "Retrieving and refining candidates"); pq_candidates > 0
     * selects it (c2f_candidates must then be 0).  Each token of a full block
     * carries a PQ32 code: 32 bytes, byte j the index of the centroid of
     * dims 4j .. 4j+3 of its index key among the 256 of codebook j.  A step
     *   1. scores every token of every full candidate block with Eq. 6,
     *        s~_t = sum_g w[r,g] max(0, sum_j q[r,g,4j:4j+4] . C_j[c_{t,j}])
     *      (w = fine_head_weights, required),
     *   2. keeps the pq_candidates tokens of largest s~ (ties to the lower
     *      token),
     *   3. drops a kept token whose original index key is not cached (a
     *      miss: pq_hit 0) when its s~ is below the candidates' c2f_tokens-th
     *      largest s~ minus the sample standard deviation (n - 1) of the
     *      candidates' s~ (no drop with at most c2f_tokens candidates),
     *   4. scores the remaining candidates and the tokens of the partial
     *      last block with their FP8 index keys (the weighted-ReLU score
     *      above, with the exact keys) and keeps the c2f_tokens best, whose
     *      positions are the selection.
     * pq_codes [num_pages, 1, block_size, 32] uint8 device (the index
     * cache's geometry, one KV head); pq_codebook [32, 256, 4] bf16 device;
     * pq_hit [num_pages, 1, block_size] uint8 device, 1 = the token's index
     * key is cached, or NULL (every key cached).  Needs 64 query heads over
     * one KV head, dk = 128.  The miss filter's threshold is computed in
     * fp64 from fp32 coarse scores. */
    int32_t pq_candidates;
    const uint8_t *pq_codes;
    const void *pq_codebook;
    const uint8_t *pq_hit;
} lsa_params;

/* Status and errors ------------------------------------------------------ */

const char *lsa_status_string(lsa_status s);

/* Reads the current device's status word (synchronises the device), returns
 * the most severe recorded code (LSA_OK if none) and, if clear != 0, resets
 * it.  *flags (may be NULL) receives the raw bit set: bit n set means code n
 * was recorded. */
lsa_status lsa_get_device_status(uint32_t *flags, int clear);

/* Step 1: summaries ------------------------------------------------------- */

/* Writes the bf16 summary of every full block referenced by the page tables:
 *   summaries[(p*Hkv + h)*dk + i] = bf16_rne( (1/b) * sum_t K[p,h,t,i] )
 * with the sum taken in fp64 (exact for bf16 keys of moderate exponent
 * spread), so the result does not depend on summation order.  For an e4m3
 * index cache the summed values are scale_t * e4m3(k8).  Blocks j with
 * (j+1)*b > seq_lens[r] (partial tails) are skipped.  A page referenced by
 * several requests is written with identical bits by each.
 *   page_table [batch, max_blocks] int32 device; seq_lens [batch] int32 device;
 *   summaries  [num_pages, Hkv, dk] bf16 device, caller-allocated.
 * Errors: LSA_ERR_INVALID_ARG for NULLs or batch < 0; device: LSA_ERR_BOUNDS
 * for page ids outside [0, num_pages) or lengths beyond max_blocks*b. */
lsa_status lsa_build_summaries(const lsa_cache *cache, const int32_t *page_table,
                               const int32_t *seq_lens, int32_t batch, int32_t max_blocks,
                               void *summaries, lsa_stream_t stream);

/* Quest's block summaries (Vortex blog post, end of "Why Long Generations
 * Are Expensive": each block keeps the element-wise maximum and minimum of
 * its keys; the Quest listing in "Writing an algorithm: vFlow"):
 *   summaries[((p*Hkv + h)*2 + 0)*dk + i] = max_t K[p,h,t,i]
 *   summaries[((p*Hkv + h)*2 + 1)*dk + i] = min_t K[p,h,t,i]
 * for every full block referenced by the page tables (exact: bf16 values).
 *   summaries [num_pages, Hkv, 2, dk] bf16 device, caller-allocated.
 * Scored with lsa_params.summary_kind = LSA_SUMMARY_MINMAX.  bf16 keys only
 * (LSA_ERR_UNSUPPORTED for e4m3).  Other arguments and errors as
 * lsa_build_summaries. */
lsa_status lsa_build_minmax_summaries(const lsa_cache *cache, const int32_t *page_table,
                                      const int32_t *seq_lens, int32_t batch, int32_t max_blocks,
                                      void *summaries, lsa_stream_t stream);

/* Appends one token per request: writes k_new[r, h, :] and v_new[r, h, :]
 * (bf16 [batch, Hkv, dk] / [batch, Hkv, dv], device) into slot L % b of page
 * page_table[r, L / b] with L = seq_lens[r], then increments seq_lens[r].
 * When the block becomes full, its summary is computed in the same kernel
 * (the summary is built once, when the block fills: Vortex, "Block top-k
 * attention").  v_new is ignored for a latent cache (v == k).
 * Errors as lsa_build_summaries; LSA_ERR_UNSUPPORTED for e4m3 caches. */
lsa_status lsa_append_block(const lsa_cache *cache, const void *k_new, const void *v_new,
                            const int32_t *page_table, int32_t *seq_lens, int32_t batch,
                            int32_t max_blocks, void *summaries, lsa_stream_t stream);

/* lsa_append_block for Quest summaries: when a block fills, its maximum and
 * minimum keys are written ([num_pages, Hkv, 2, dk], as
 * lsa_build_minmax_summaries). */
lsa_status lsa_append_block_minmax(const lsa_cache *cache, const void *k_new, const void *v_new,
                                   const int32_t *page_table, int32_t *seq_lens, int32_t batch,
                                   int32_t max_blocks, void *summaries, lsa_stream_t stream);

/* Step 2: scores ---------------------------------------------------------- */

/* scores[(r*Hkv + h)*max_blocks + j] = sum_{g in group(h)} q[r,g,:] .
 * summaries[page_table[r,j], h, :] in fp32 for every candidate block j of
 * request r; -inf for every other j < max_blocks.
 *   q [batch, Hq, dk] bf16 device, contiguous;  scores fp32 device.
 * `cache` supplies the geometry (num_kv_heads, block_size, dk, num_pages).
 * Supported: dk in {64, 128, 256, 576} with Hkv*dk/8 lanes tiling a warp or
 * Hkv == 1.  Otherwise LSA_ERR_UNSUPPORTED.
 * With params->summary_kind = LSA_SUMMARY_MINMAX the summaries are Quest's
 * ([num_pages, Hkv, 2, dk]) and the score of block j is the Quest bound
 *   max_{g in group(h)} sum_i max(q[r,g,i]*max_ji, q[r,g,i]*min_ji),
 * an upper bound on q_g . k_t for every token t of the block (the listing's
 * Max over heads of Sum over dims); supported for dk in {64, 128}, Hkv and
 * the group size in {1, 2, 4, 8}. */
lsa_status lsa_score(const void *q, const lsa_cache *cache, const void *summaries,
                     const int32_t *page_table, const int32_t *seq_lens, const lsa_params *params,
                     float *scores, lsa_stream_t stream);

/* Step 3: top-k ----------------------------------------------------------- */

/* Row-wise exact top-k: for each of `rows` rows of `scores` ([rows, cols]
 * fp32 device), among the first num_cols[row] entries (num_cols NULL: all
 * cols), the k largest by (score descending, index ascending).  -inf entries
 * are not candidates; NaN entries are skipped and flagged (LSA_ERR_NAN).
 * -0.0 and +0.0 compare equal.  idx [rows, k] int32 device receives the
 * chosen column indices in ascending order, padded with -1.
 * Supported: cols <= 32768.  The result is bit-exact (no floating point). */
lsa_status lsa_topk(const float *scores, const int32_t *num_cols, int32_t rows, int32_t cols,
                    int32_t k, int32_t *idx, lsa_stream_t stream);

/* Row-wise APPROXIMATE top-k, the stochastic early exit (Vortex blog post,
 * "Making it fast": a monotone remap spreads the scores over the buckets of
 * a radix-style select, and the select stops once it has enough confident
 * winners, sampling the rest from the boundary bucket).  Opt-in; it trades
 * recall of the exact top-k for speed.  Per row, over the candidates
 * (entries as for lsa_topk), keff = min(k, candidates):
 *   1. bucket(x) = floor((x - vmin) * (2048 / (vmax - vmin))), clamped to
 *      2047, in fp32 over the candidates' smallest and largest value (one
 *      bucket when they are equal or the span is not finite);
 *   2. the candidates in buckets above the one holding the keff-th largest
 *      value (the boundary bucket, cnt candidates) are all taken;
 *   3. the remaining `take` are the boundary bucket's candidates numbered,
 *      in column order, within `take` steps after off circularly:
 *      number n is taken iff (n - off) mod cnt < take, with
 *      off = splitmix64(seed, row + 1) mod cnt, where splitmix64(s, n) is
 *      output n of SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) seeded
 *      with s.
 * Every candidate above the boundary bucket is kept, and every one in it is
 * kept with probability take / cnt over the seed.  The result is a
 * deterministic function of (scores, k, seed, row).  idx as lsa_topk.
 * Supported: cols <= 32768.  Errors as lsa_topk. */
lsa_status lsa_topk_approx(const float *scores, const int32_t *num_cols, int32_t rows, int32_t cols,
                           int32_t k, uint64_t seed, int32_t *idx, lsa_stream_t stream);

/* Coarse-to-fine fine pass: for every token t of the candidate blocks
 * cand[r, h, :] (ascending, -1 padded, c2f_candidates per row) of request r,
 *   f_t = scale_t * sum_{g in group(h)} q[r,g,:] . e4m3(k8_t)
 * in fp32 (or the weighted-ReLU score when params->fine_head_weights is
 * set); keeps the c2f_tokens best by (f descending, token ascending).
 * tok_idx [batch, Hkv, c2f_tokens] int32 device: token positions, ascending,
 * -1 padded.  index_cache: an LSA_KEYS_E4M3 cache with dk = 128. */
lsa_status lsa_fine_topk(const void *q, const lsa_cache *index_cache, const int32_t *page_table,
                         const int32_t *seq_lens, const int32_t *cand, const lsa_params *params,
                         int32_t *tok_idx, void *workspace, size_t workspace_bytes,
                         lsa_stream_t stream);

/* Kernel launches one lsa_decode_step call with these shapes makes (the
 * selection and attention kernels the planner picks for them), or -1 when
 * the shapes are invalid.  index_cache: as for lsa_decode_step (NULL unless
 * coarse-to-fine).  No device work. */
int32_t lsa_decode_step_launches(const lsa_cache *cache, const lsa_cache *index_cache, const lsa_params *params);

/* PQ32 codes of the index keys of every full block of each request (the
 * encoded history): byte j of token t is the centroid of codebook j nearest
 * to dims 4j .. 4j+3 of scale_t * e4m3(k8_t) in squared Euclidean distance,
 * ties to the lower centroid (LeanSparse, Section 5: each completed page is
 * encoded when it is written).  The distance is evaluated in fp32 in one
 * fixed order (k = scale * e4m3; d_e = k_e - C_e; ((d0^2 + d1^2) + d2^2) +
 * d3^2, each step rounded, no fused multiply-add), so the codes are
 * reproducible bit for bit.  index_cache: LSA_KEYS_E4M3, one KV head, dk =
 * 128.  codebook [32, 256, 4] bf16 device; codes [num_pages, 1, block_size,
 * 32] uint8 device (pages of partial blocks are not written).  Errors as
 * lsa_build_summaries. */
lsa_status lsa_pq_encode(const lsa_cache *index_cache, const void *codebook, const int32_t *page_table,
                         const int32_t *seq_lens, int32_t batch, int32_t max_blocks, uint8_t *codes,
                         lsa_stream_t stream);

/* The PQ32 coarse scores s~_t (step 1 of the PQ32 coarse-to-fine in
 * lsa_params) of every token position t < max_blocks * block_size:
 * scores [batch, max_blocks * block_size] fp32 device, -inf for tokens that
 * are not in a full candidate block.  params: pq_codes, pq_codebook and
 * fine_head_weights are used; fp32 accumulation of exact bf16 products. */
lsa_status lsa_pq_scores(const void *q, const lsa_cache *index_cache, const int32_t *page_table,
                         const int32_t *seq_lens, const lsa_params *params, float *scores, lsa_stream_t stream);

/* Step 4: sparse attention ------------------------------------------------ */

/* Bytes of workspace lsa_sparse_decode needs for these shapes (partial
 * results and per-row counters).  The same rules as lsa_decode_step's
 * workspace apply. */
size_t lsa_sparse_decode_workspace_size(const lsa_cache *cache, const lsa_params *params);

/* Exact attention over T = F U selected for every query head:
 *   out[r, g, :] = bf16_rne( softmax_t(scale * q[r,g,:] . K_t) V_t ),
 *   lse[r, g]    = log sum_t exp(scale * q[r,g,:] . K_t)   (natural log),
 * split into parts whose partial (o, m, l) are merged by log-sum-exp.
 * idx [batch, Hkv, n] int32 device, ascending, -1 padded, where n = k_blocks
 * and entries are block indices (single stage), or n = c2f_tokens and
 * entries are token positions (c2f_candidates > 0 or pq_candidates > 0).
 * A selected block must be a candidate; a selected token must lie outside
 * the forced ranges (it may be in the partial last block).  Other entries
 * are skipped and flagged (LSA_ERR_BOUNDS).  A request with
 * seq_lens[r] == 0 gets out = 0 and lse = -inf.
 *   out [batch, Hq, dv] bf16 device; lse [batch, Hq] fp32 device or NULL.
 * workspace: device, >= lsa_sparse_decode_workspace_size bytes (may be NULL
 * when that size is 0). */
lsa_status lsa_sparse_decode(const void *q, const lsa_cache *cache, const int32_t *page_table,
                             const int32_t *seq_lens, const int32_t *idx, const lsa_params *params,
                             void *out, float *lse, void *workspace, size_t workspace_bytes,
                             lsa_stream_t stream);

/* lsa_sparse_decode without a caller workspace.  The pages have no
 * counterpart to this call: it exists for callers that cannot hand over
 * device memory -- a plain C host with no device allocator of its own, or a
 * serving loop whose memory plan is fixed before it starts and admits no
 * allocation afterwards.  It allocates nothing: its scratch is one buffer of
 * LSA_STATIC_SCRATCH_BYTES in the library's own static device memory, one
 * per device, zero at load, held until the process exits.
 *   - Shapes whose lsa_sparse_decode_workspace_size exceeds
 *     LSA_STATIC_SCRATCH_BYTES are rejected with LSA_ERR_WORKSPACE, and
 *     invalid pointers with LSA_ERR_INVALID_ARG, before anything is
 *     launched or cleared.
 *   - Counters in the buffer must be zero when a call starts; a call that
 *     completes leaves them zero for the next call with the same layout.  A
 *     call whose cache descriptor, parameters or attention plan (which
 *     LSA_ATTENTION_PATH can change) differs from the previous call's on
 *     that device first clears the bytes it needs, on its stream.  So does
 *     the first call after lsa_get_device_status reported a device error
 *     (a call that recorded one may leave counters non-zero): read the
 *     status after such a call before making the next one.
 *   - The first call on a device looks up the buffer's address once; make
 *     that first call before any stream capture begins.
 *   - All calls on a device share the one buffer, so calls that may run at
 *     the same time (several streams, or host threads without an order
 *     between their calls) race on it and must not use this entry point.
 * Arguments and results otherwise as lsa_sparse_decode. */
#define LSA_STATIC_SCRATCH_BYTES (8u << 20)
lsa_status lsa_sparse_decode_static_scratch(const void *q, const lsa_cache *cache,
                                            const int32_t *page_table, const int32_t *seq_lens,
                                            const int32_t *idx, const lsa_params *params, void *out,
                                            float *lse, lsa_stream_t stream);

/* Fused decode step ------------------------------------------------------- */

/* Bytes of workspace lsa_decode_step needs.  The workspace holds the
 * block scores, the selection, partial results and counters, some of which
 * must be zero when a call starts: zero-fill it before its first use (e.g.
 * cudaMemsetAsync after allocation).  Every call that completes without a
 * device error leaves those parts at zero again, so one workspace serves any
 * number of calls and CUDA-graph replays of the same shape (cache
 * descriptor and parameters) and implementation; zero it again before
 * using it for another shape or implementation, or after a call that
 * recorded LSA_ERR_TIMEOUT.  Calls that share a workspace must not overlap
 * in time. */
size_t lsa_decode_step_workspace_size(const lsa_cache *cache, const lsa_params *params);

/* Steps 2-4 in one call: score every candidate block against the summaries,
 * select top-k_blocks per (request, KV head), and attend F U selected.  With
 * c2f_candidates > 0 and an index cache: coarse top-C blocks over
 * `summaries` (built from the index keys), fine top-c2f_tokens tokens, then
 * attention.
 *   idx_out [batch, Hkv, k_blocks or c2f_tokens] int32 device or NULL.
 * Other arguments as in the calls above.
 *
 * Implementations (Vortex, "Making it fast", fuses the operators so block
 * scores never leave the chip; here they make one trip through L2):
 *   default: two launches.  The score kernel writes fp32 block scores to the
 *     workspace; the attention kernel selects each (request, KV head) row's
 *     blocks itself (exact top-k in the CTA), writes idx_out, and attends.
 *     It is launched as a programmatic dependent of the score kernel and
 *     reads q, seq_lens and the page table before it waits for the scores,
 *     which is safe because the score kernel starts only once all earlier
 *     work on the stream is complete.  With c2f_candidates > 0, rows of more
 *     than 8192 blocks, k_blocks > 512, an explicit split count, an odd GQA
 *     group, head dimensions other than dk = dv = 64 or 128, or a latent
 *     (aliased K/V) cache, the stages run as separate launches (score,
 *     top-k, attention).
 *   LSA_PDL=0 (environment): no programmatic dependent launch anywhere;
 *   LSA_PDL=1: every kernel of the library is launched as one. */
lsa_status lsa_decode_step(const void *q, const lsa_cache *cache, const void *summaries,
                           const lsa_cache *index_cache, const int32_t *page_table,
                           const int32_t *seq_lens, const lsa_params *params, int32_t *idx_out,
                           void *out, float *lse, void *workspace, size_t workspace_bytes,
                           lsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LSA_H */

// C-ABI entry points of liblsa.so: argument validation, work planning
// (split-K sizing from the device's SM count), workspace layout and the
// stream-ordered launch sequence of each call.  See include/lsa.h for the
// contract of every function.
#include <math.h>

#include <algorithm>
#include <mutex>
#include <stdlib.h>
#include <string.h>

#include "lsa_internal.h"

namespace lsa {
namespace {

constexpr int kMaxDevices = 64;

__device__ uint32_t d_status_word;

std::mutex g_mu;
uint32_t *g_status_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return (dev >= 0 && dev < kMaxDevices) ? dev : -1;
}

// Address of this device's status word (looked up once per device).
uint32_t *status_word()
{
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, d_status_word) == cudaSuccess) g_status_ptr[dev] = static_cast<uint32_t *>(p);
    }
    return g_status_ptr[dev];
}

int sm_count()
{
    const int dev = current_device();
    if (dev < 0) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool mult16(int64_t elems, int esz) { return ((elems * esz) & 15) == 0; }

size_t round_up(size_t x) { return (x + 255) & ~size_t(255); }

// CTAs per SM of the tcgen05 attention kernel for a shape (cached; the
// occupancy query is a host call).
int umma_ctas_per_sm(int dk, int dv, bool alias)
{
    static int cache[3] = {-1, -1, -1};
    const int idx = dk == 128 ? 0 : (alias ? 1 : 2);
    std::lock_guard<std::mutex> lk(g_mu);
    if (cache[idx] < 0) cache[idx] = attention_umma_ctas_per_sm(dk, dv, alias);
    return cache[idx];
}

// Validates a cache descriptor and converts it to the kernels' view.
lsa_status make_view(const lsa_cache *c, bool need_values, CacheView *v)
{
    if (!c || !c->k) return LSA_ERR_INVALID_ARG;
    if (c->num_pages <= 0 || c->block_size <= 0 || c->num_kv_heads <= 0 || c->dk <= 0) return LSA_ERR_INVALID_ARG;
    const bool e4m3 = c->key_format == LSA_KEYS_E4M3;
    if (!e4m3 && c->key_format != LSA_KEYS_BF16) return LSA_ERR_INVALID_ARG;
    const int esz = e4m3 ? 1 : 2;
    if (!aligned16(c->k) || !mult16(c->dk, esz) || !mult16(c->k_page_stride, esz) ||
        !mult16(c->k_head_stride, esz) || !mult16(c->k_token_stride, esz))
        return LSA_ERR_INVALID_ARG;
    if (c->k_token_stride < c->dk) return LSA_ERR_INVALID_ARG;
    memset(v, 0, sizeof *v);
    v->k = static_cast<const uint8_t *>(c->k);
    v->kps = c->k_page_stride;
    v->khs = c->k_head_stride;
    v->kts = c->k_token_stride;
    v->num_pages = c->num_pages;
    v->b = c->block_size;
    v->hkv = c->num_kv_heads;
    v->dk = c->dk;
    v->e4m3 = e4m3;
    if (e4m3) {
        if (!c->k_scale) return LSA_ERR_INVALID_ARG;
        v->kscale = c->k_scale;
        v->sps = c->scale_page_stride;
        v->shs = c->scale_head_stride;
    }
    if (need_values) {
        if (e4m3 || !c->v || c->dv <= 0) return LSA_ERR_INVALID_ARG;
        if (!aligned16(c->v) || !mult16(c->dv, 2) || !mult16(c->v_page_stride, 2) ||
            !mult16(c->v_head_stride, 2) || !mult16(c->v_token_stride, 2) || c->v_token_stride < c->dv)
            return LSA_ERR_INVALID_ARG;
        v->v = static_cast<const uint8_t *>(c->v);
        v->vps = c->v_page_stride;
        v->vhs = c->v_head_stride;
        v->vts = c->v_token_stride;
        v->dv = c->dv;
        v->v_alias = c->v == c->k && c->v_page_stride == c->k_page_stride &&
                     c->v_head_stride == c->k_head_stride && c->v_token_stride == c->k_token_stride &&
                     c->dv <= c->dk;
    }
    return LSA_OK;
}

lsa_status check_params(const lsa_params *p, const CacheView &v)
{
    if (!p) return LSA_ERR_INVALID_ARG;
    if (p->batch < 0 || p->num_q_heads <= 0 || p->num_q_heads % v.hkv != 0) return LSA_ERR_INVALID_ARG;
    if (p->batch > 0 && p->max_blocks <= 0) return LSA_ERR_INVALID_ARG;
    if (p->k_blocks < 0 || p->sink_tokens < 0 || p->recent_tokens < 0) return LSA_ERR_INVALID_ARG;
    if (p->c2f_candidates < 0 || p->c2f_tokens < 0 || p->num_splits < 0) return LSA_ERR_INVALID_ARG;
    if (p->batch > 65535 || (int64_t)p->max_blocks * v.b > INT32_MAX) return LSA_ERR_INVALID_ARG;
    if (p->summary_kind != LSA_SUMMARY_MEAN && p->summary_kind != LSA_SUMMARY_MINMAX) return LSA_ERR_INVALID_ARG;
    if (p->pq_candidates < 0 || (p->pq_candidates > 0 && p->c2f_candidates > 0)) return LSA_ERR_INVALID_ARG;
    return LSA_OK;
}

lsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LSA_OK : LSA_ERR_CUDA; }

// Whether the selection is of tokens (the two coarse-to-fine variants)
// rather than of blocks.
bool token_mode_of(const lsa_params *p) { return p->c2f_candidates > 0 || p->pq_candidates > 0; }

// Bounded waits give up after this many SM clock cycles (about a second
// by default).  LSA_SPIN_BUDGET (environment, cycles) overrides it; tests set
// a short budget to make a wait run out.
long long spin_budget()
{
    const char *e = getenv("LSA_SPIN_BUDGET");
    if (e && *e) {
        const long long v = strtoll(e, nullptr, 10);
        if (v > 0) return v;
    }
    return kSpinBudget;
}

float scale_of(const lsa_params *p, int dk)
{
    return p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / sqrtf((float)dk);
}

// Pointer checks of the attention call (lsa_sparse_decode and its
// no-workspace variant), made before anything is launched or cleared.
lsa_status check_decode_args(const void *q, const int32_t *page_table, const int32_t *seq_lens, const int32_t *idx,
                             const lsa_params *p, const void *out)
{
    const bool token_mode = token_mode_of(p);
    const int nsel = token_mode ? p->c2f_tokens : p->k_blocks;
    if (!q || !page_table || !seq_lens || !out || !aligned16(q) || (nsel > 0 && !idx)) return LSA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0) return LSA_ERR_INVALID_ARG;
    return LSA_OK;
}

// ---------------------------------------------------------------- planning

struct AttnPlan {
    int nsub, splits, items_per_split;
    int tc_group;          // > 0: tensor-core kernel with this many heads per CTA
    bool umma;             // tcgen05 kernel for groups of 64 heads, one tile of 128 tokens per CTA
    bool umma_merge;       // ... merging the row's tiles itself (every CTA resident at once)
    bool flat;             // even split of every row's items over the GPU (attention_flat.cu)
    int fl_ns, fl_ctas, fl_parts;
    int64_t fl_total;
    size_t ws_bytes;
};

lsa_status plan_attention(const CacheView &v, const lsa_params *p, bool token_mode, AttnPlan *pl)
{
    const int G = p->num_q_heads / v.hkv;
    int gs = 0;
    if (v.b % kChunk != 0) return LSA_ERR_UNSUPPORTED;
    memset(pl, 0, sizeof *pl);
    const char *path = getenv("LSA_ATTENTION_PATH");
    const bool allow_tc = !(path && strcmp(path, "cuda_core") == 0);
    pl->umma = allow_tc && attention_umma_supported(v.dk, v.dv, G, v.v_alias != 0);
    if (pl->umma) {
        // one CTA per 128-token tile of a row: the tiles are the split-K
        // parts (an explicit split count does not change them)
        const int nsel = token_mode ? p->c2f_tokens : p->k_blocks;
        const int items = attention_items_max(p->sink_tokens, p->recent_tokens, v.b, nsel, token_mode);
        const int ipt = attention_umma_items_per_tile();
        pl->tc_group = 0;
        pl->flat = false;
        pl->nsub = 1;
        pl->fl_ns = pl->fl_ctas = pl->fl_parts = 0;
        pl->fl_total = 0;
        pl->items_per_split = ipt;
        pl->splits = std::max(1, (items + ipt - 1) / ipt);
        pl->ws_bytes = 0;
        pl->umma_merge = false;
        const int64_t rows = (int64_t)p->batch * v.hkv;
        if (pl->splits > 1) {
            const size_t rowsq = (size_t)p->batch * p->num_q_heads * pl->splits;
            pl->ws_bytes = round_up(rowsq * v.dv * sizeof(float)) + round_up(rowsq * sizeof(float));
            // the tiles merge their row themselves when the whole grid is
            // resident at once (their wait for the row's other tiles then
            // always ends); otherwise the merge kernel does it
            const int per_sm = umma_ctas_per_sm(v.dk, v.dv, v.v_alias != 0);
            pl->umma_merge = per_sm > 0 && (int64_t)pl->splits * rows <= (int64_t)per_sm * sm_count();
            if (pl->umma_merge) pl->ws_bytes += round_up(2 * (size_t)rows * sizeof(uint32_t));
        }
        return rows > 65535 ? LSA_ERR_UNSUPPORTED : LSA_OK;
    }
    pl->tc_group = allow_tc ? attention_tc_group(v.dk, v.dv, G, v.v_alias != 0, token_mode, v) : 0;
    if (pl->tc_group > 0) {
        gs = pl->tc_group;
    } else if (!attention_supported(v.dk, v.dv, G, v.v_alias != 0, &gs)) {
        return LSA_ERR_UNSUPPORTED;
    }
    pl->nsub = G / gs;
    const int nsel = token_mode ? p->c2f_tokens : p->k_blocks;
    const int items = attention_items_max(p->sink_tokens, p->recent_tokens, v.b, nsel, token_mode);
    const int64_t rows = (int64_t)p->batch * v.hkv * pl->nsub;
    int s = p->num_splits;
    if (s <= 0) {
        const int64_t target = 2LL * sm_count();
        s = rows > 0 ? (int)((target + rows - 1) / rows) : 1;
    }
    s = s < 1 ? 1 : (s > items ? items : s);
    if (s > 65535) s = 65535;
    // every split's item descriptors must fit in shared memory
    const int max_ips = pl->tc_group > 0 ? attention_tc_max_items_per_split(v.dk)
                                          : attention_max_items_per_split(v.dk, v.dv, v.v_alias != 0, token_mode);
    if (max_ips < 1) return LSA_ERR_UNSUPPORTED;
    const int min_s = (items + max_ips - 1) / max_ips;
    if (s < min_s) s = min_s;
    pl->items_per_split = (items + s - 1) / s;
    pl->splits = (items + pl->items_per_split - 1) / pl->items_per_split;
    if (pl->splits < 1) pl->splits = 1;
    pl->ws_bytes = 0;
    if (pl->splits > 1) {
        const size_t rowsq = (size_t)p->batch * p->num_q_heads * pl->splits;
        pl->ws_bytes = round_up(rowsq * v.dv * sizeof(float)) + round_up(rowsq * sizeof(float));
    }
    // Without an explicit split count the tensor-core path splits all rows'
    // items evenly over the GPU instead: at most two rows per CTA (a piece is
    // no longer than a row) and at most the per-warp item limit per warp.
    pl->flat = pl->tc_group > 0 && p->num_splits <= 0 && !token_mode && items > 0 && rows > 0;
    if (pl->flat) {
        const int64_t T = rows * items;
        const int64_t per_cta = std::min<int64_t>(items, (int64_t)attention_flat_warps() *
                                                              attention_flat_max_items_per_warp());
        const int64_t slots = (int64_t)attention_flat_ctas_per_sm() * sm_count();
        int64_t nc;
        if (rows <= slots && items <= per_cta) {
            // every row has the same number of item slots: a whole number of
            // CTAs per row keeps the GPU balanced, and one CTA per row needs
            // no merge across CTAs
            nc = rows * (slots / rows);
        } else {
            nc = std::max<int64_t>(slots, (T + per_cta - 1) / per_cta);
        }
        nc = std::min<int64_t>(nc, T);
        // the kernel's index arithmetic is 32-bit (below 2^31: fdiv); larger
        // batches take the split-K plan above
        if ((T + 1) * nc >= (int64_t(1) << 31)) {
            pl->flat = false;
            return LSA_OK;
        }
        pl->fl_ns = items;
        pl->fl_total = T;
        pl->fl_ctas = (int)nc;
        const int64_t min_piece = T / nc;   // >= 1
        pl->fl_parts = (int)((items + min_piece - 1) / min_piece + 1);
        const size_t rowsq = (size_t)p->batch * p->num_q_heads * pl->fl_parts;
        pl->ws_bytes = round_up(rowsq * v.dv * sizeof(float)) + round_up(rowsq * sizeof(float)) +
                       round_up((size_t)rows * sizeof(uint32_t));
    }
    return LSA_OK;
}

// sel_scores: the attention kernel selects the blocks itself from these fp32
// score rows (only with the even-split plan, see attention_flat_can_select)
// and writes the selection to sel_write when that is not NULL.
lsa_status run_attention(const void *q, const CacheView &v, const int32_t *pt, const int32_t *lens,
                         const int32_t *idx, const lsa_params *p, bool token_mode, void *out, float *lse,
                         uint8_t *ws, size_t ws_bytes, cudaStream_t st, const float *sel_scores = nullptr,
                         int32_t *sel_write = nullptr)
{
    AttnPlan pl;
    lsa_status rc = plan_attention(v, p, token_mode, &pl);
    if (rc != LSA_OK) return rc;
    if (ws_bytes < pl.ws_bytes || (pl.ws_bytes && !ws)) return LSA_ERR_WORKSPACE;
    AttnArgs a;
    memset(&a, 0, sizeof a);
    a.q = static_cast<const uint16_t *>(q);
    a.c = v;
    a.pt = pt;
    a.lens = lens;
    a.idx = idx;
    a.batch = p->batch;
    a.hq = p->num_q_heads;
    a.max_blocks = p->max_blocks;
    a.nsel = token_mode ? p->c2f_tokens : p->k_blocks;
    a.token_mode = token_mode;
    a.sink = p->sink_tokens;
    a.recent = p->recent_tokens;
    a.scale_log2 = scale_of(p, v.dk) * 1.4426950408889634f;
    a.fd_b = make_fastdiv((uint32_t)v.b);
    a.fd_cpb = make_fastdiv((uint32_t)(v.b / kChunk));
    a.fd_hkv = make_fastdiv((uint32_t)v.hkv);
    a.gsize = p->num_q_heads / v.hkv;
    a.splits = pl.splits;
    a.items_per_split = pl.items_per_split;
    a.nsub = pl.nsub;
    a.fd_nsub = make_fastdiv((uint32_t)pl.nsub);
    a.out = static_cast<uint16_t *>(out);
    a.lse = lse;
    a.status = status_word();
    a.spin_budget = spin_budget();
    if (sel_scores && !pl.flat) return LSA_ERR_UNSUPPORTED;
    if (pl.flat) {
        a.sel_scores = sel_scores;
        a.sel_cols = p->max_blocks;
        // only the decode step passes score rows, right after scoring
        a.pdl_early = sel_scores && pdl_step_dependent() ? 1 : 0;
        a.sel_write = sel_write;
        a.fl_ns = pl.fl_ns;
        a.fl_total = pl.fl_total;
        a.fl_ctas = pl.fl_ctas;
        a.fl_parts = pl.fl_parts;
        a.fd_ns = make_fastdiv((uint32_t)pl.fl_ns);
        a.fd_nc = make_fastdiv((uint32_t)pl.fl_ctas);
        a.fd_total = make_fastdiv((uint32_t)pl.fl_total);
        const size_t rowsq = (size_t)p->batch * p->num_q_heads * pl.fl_parts;
        a.o_part = reinterpret_cast<float *>(ws);
        a.lse_part = reinterpret_cast<float *>(ws + round_up(rowsq * v.dv * sizeof(float)));
        a.row_done = reinterpret_cast<uint32_t *>(ws + round_up(rowsq * v.dv * sizeof(float)) +
                                                  round_up(rowsq * sizeof(float)));
        bool unsup = false;
        const cudaError_t e = launch_attention_flat(a, pl.tc_group, st, &unsup);
        if (unsup) return LSA_ERR_UNSUPPORTED;
        return e == cudaSuccess ? LSA_OK : LSA_ERR_CUDA;
    }
    const size_t rowsq = (size_t)p->batch * p->num_q_heads * pl.splits;
    if (pl.splits > 1) {
        a.o_part = reinterpret_cast<float *>(ws);
        a.lse_part = reinterpret_cast<float *>(ws + round_up(rowsq * v.dv * sizeof(float)));
    }
    if (pl.umma_merge) {
        a.merge_in_kernel = 1;
        a.mrg_arrive = reinterpret_cast<uint32_t *>(ws + round_up(rowsq * v.dv * sizeof(float)) +
                                                    round_up(rowsq * sizeof(float)));
        a.mrg_done = a.mrg_arrive + (size_t)p->batch * v.hkv;
    }
    bool unsup = false;
    cudaError_t e = pl.umma           ? launch_attention_umma(a, st, &unsup)
                    : pl.tc_group > 0 ? launch_attention_tc(a, pl.tc_group, st, &unsup)
                                      : launch_attention(a, st, &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return LSA_ERR_CUDA;
    if (pl.splits > 1 && !pl.umma_merge) {
        MergeArgs m;
        m.o_part = a.o_part;
        m.lse_part = a.lse_part;
        m.rows = p->batch * p->num_q_heads;
        m.splits = pl.splits;
        m.dv = v.dv;
        m.out = a.out;
        m.lse = lse;
        e = launch_merge(m, st);
        if (e != cudaSuccess) return LSA_ERR_CUDA;
    }
    return LSA_OK;
}

// Workspace of the decode step: [scores | selection | c2f extras | attention].
// PQ32 coarse-to-fine: [coarse scores of every token | selection |
// candidates | row extremes + bucket counts | attention].
struct StepLayout {
    size_t scores, sel, cand, fine, attn, total;
};

lsa_status step_layout(const CacheView &v, const CacheView *iv, const lsa_params *p, StepLayout *L)
{
    const bool c2f = p->c2f_candidates > 0, pq = p->pq_candidates > 0;
    const CacheView &sv = (c2f || pq) ? *iv : v;
    AttnPlan pl;
    lsa_status rc = plan_attention(v, p, c2f || pq, &pl);
    if (rc != LSA_OK) return rc;
    const size_t rows = (size_t)p->batch * sv.hkv;
    if (pq) {
        L->scores = round_up(rows * p->max_blocks * (size_t)sv.b * sizeof(float));
        L->sel = round_up(rows * (size_t)p->c2f_tokens * sizeof(int32_t));
        L->cand = round_up(rows * (size_t)p->pq_candidates * sizeof(int32_t));
        L->fine = round_up(rows * 2 * sizeof(uint32_t)) + round_up(rows * (size_t)kPqBins * sizeof(uint32_t));
    } else {
        L->scores = round_up(rows * p->max_blocks * sizeof(float));
        L->sel = round_up(rows * (size_t)(c2f ? p->c2f_tokens : p->k_blocks) * sizeof(int32_t));
        L->cand = c2f ? round_up(rows * (size_t)p->c2f_candidates * sizeof(int32_t)) : 0;
        L->fine = c2f ? round_up(rows * (size_t)p->c2f_candidates * sv.b * sizeof(float)) : 0;
    }
    L->attn = pl.ws_bytes;
    L->total = L->scores + L->sel + L->cand + L->fine + L->attn;
    return LSA_OK;
}

// The PQ arguments of a step or a scoring call (pointers the caller checked).
PqArgs pq_args(const void *q, const CacheView &iv, const int32_t *page_table, const int32_t *seq_lens,
               const lsa_params *p)
{
    PqArgs a;
    memset(&a, 0, sizeof a);
    a.q = static_cast<const uint16_t *>(q);
    a.weights = p->fine_head_weights;
    a.ic = iv;
    a.codes = p->pq_codes;
    a.codebook = static_cast<const uint16_t *>(p->pq_codebook);
    a.hit = p->pq_hit;
    a.pt = page_table;
    a.lens = seq_lens;
    a.batch = p->batch;
    a.hq = p->num_q_heads;
    a.max_blocks = p->max_blocks;
    a.sink = p->sink_tokens;
    a.recent = p->recent_tokens;
    a.ncand = p->pq_candidates;
    a.tok_k = p->c2f_tokens;
    a.status = status_word();
    a.spin_budget = spin_budget();
    return a;
}

bool pq_inputs_ok(const void *q, const lsa_params *p)
{
    return q && aligned16(q) && p->fine_head_weights && p->pq_codes && aligned16(p->pq_codes) && p->pq_codebook &&
           aligned16(p->pq_codebook);
}

}  // namespace
}  // namespace lsa

namespace lsa {
void static_scratch_forget(int dev);
}

using namespace lsa;

extern "C" {

const char *lsa_status_string(lsa_status s)
{
    switch (s) {
    case LSA_OK: return "ok";
    case LSA_ERR_INVALID_ARG: return "invalid argument";
    case LSA_ERR_UNSUPPORTED: return "unsupported shape";
    case LSA_ERR_WORKSPACE: return "workspace missing or too small";
    case LSA_ERR_BOUNDS: return "index, page id or length out of range (device)";
    case LSA_ERR_TIMEOUT: return "bounded wait timed out (device)";
    case LSA_ERR_CUDA: return "CUDA runtime error";
    case LSA_ERR_NAN: return "NaN score skipped (device)";
    }
    return "unknown status";
}

lsa_status lsa_get_device_status(uint32_t *flags, int clear)
{
    uint32_t *w = status_word();
    if (!w) return LSA_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, d_status_word, sizeof v) != cudaSuccess) return LSA_ERR_CUDA;
    if (clear) {
        const uint32_t z = 0;
        if (cudaMemcpyToSymbol(d_status_word, &z, sizeof z) != cudaSuccess) return LSA_ERR_CUDA;
    }
    if (flags) *flags = v;
    // a call that recorded a device error may have left counters of the
    // static scratch non-zero: the next no-workspace call clears it again
    if (v != 0) static_scratch_forget(current_device());
    const lsa_status order[] = {LSA_ERR_TIMEOUT, LSA_ERR_BOUNDS, LSA_ERR_NAN, LSA_ERR_INVALID_ARG};
    for (lsa_status s : order)
        if (v & (1u << s)) return s;
    return LSA_OK;
}

}  // extern "C"

namespace lsa {
namespace {

lsa_status build_summaries(const lsa_cache *cache, const int32_t *page_table, const int32_t *seq_lens,
                           int32_t batch, int32_t max_blocks, void *summaries, lsa_stream_t stream, bool quest)
{
    CacheView v;
    lsa_status rc = make_view(cache, false, &v);
    if (rc != LSA_OK) return rc;
    if (quest && v.e4m3) return LSA_ERR_UNSUPPORTED;
    if (batch < 0 || max_blocks < 0) return LSA_ERR_INVALID_ARG;
    if (batch == 0 || max_blocks == 0) return LSA_OK;
    if (!page_table || !seq_lens || !summaries || !aligned16(summaries)) return LSA_ERR_INVALID_ARG;
    SummaryArgs a;
    memset(&a, 0, sizeof a);
    a.c = v;
    a.pt = page_table;
    a.lens = const_cast<int32_t *>(seq_lens);
    a.batch = batch;
    a.max_blocks = max_blocks;
    a.summ = static_cast<uint16_t *>(summaries);
    a.status = status_word();
    return from_cuda(launch_build_summaries(a, reinterpret_cast<cudaStream_t>(stream), quest));
}

lsa_status append_block(const lsa_cache *cache, const void *k_new, const void *v_new, const int32_t *page_table,
                        int32_t *seq_lens, int32_t batch, int32_t max_blocks, void *summaries, lsa_stream_t stream,
                        bool quest)
{
    CacheView v;
    lsa_status rc = make_view(cache, cache && cache->key_format == LSA_KEYS_BF16, &v);
    if (rc != LSA_OK) return rc;
    if (v.e4m3) return LSA_ERR_UNSUPPORTED;
    if (batch < 0 || max_blocks < 0) return LSA_ERR_INVALID_ARG;
    if (batch == 0) return LSA_OK;
    if (!k_new || !page_table || !seq_lens || !summaries || !aligned16(k_new) || !aligned16(summaries))
        return LSA_ERR_INVALID_ARG;
    if (!v.v_alias && (!v_new || !aligned16(v_new))) return LSA_ERR_INVALID_ARG;
    SummaryArgs a;
    memset(&a, 0, sizeof a);
    a.c = v;
    a.pt = page_table;
    a.lens = seq_lens;
    a.batch = batch;
    a.max_blocks = max_blocks;
    a.summ = static_cast<uint16_t *>(summaries);
    a.k_new = static_cast<const uint16_t *>(k_new);
    a.v_new = static_cast<const uint16_t *>(v_new);
    a.status = status_word();
    bool unsup = false;
    cudaError_t e = launch_append(a, reinterpret_cast<cudaStream_t>(stream), quest, &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    return from_cuda(e);
}

// Block scores with the kernel the summaries call for.
cudaError_t launch_scores(const ScoreArgs &s, int summary_kind, cudaStream_t st, bool *unsup)
{
    return summary_kind == LSA_SUMMARY_MINMAX ? launch_score_quest(s, st, unsup) : launch_score(s, st, unsup);
}

bool scores_supported(const CacheView &v, const lsa_params *p)
{
    return p->summary_kind == LSA_SUMMARY_MINMAX ? score_quest_supported(v.dk, v.hkv, p->num_q_heads / v.hkv)
                                                 : score_supported(v.dk, v.hkv);
}

}  // namespace
}  // namespace lsa

extern "C" {

lsa_status lsa_build_summaries(const lsa_cache *cache, const int32_t *page_table, const int32_t *seq_lens,
                               int32_t batch, int32_t max_blocks, void *summaries, lsa_stream_t stream)
{
    return build_summaries(cache, page_table, seq_lens, batch, max_blocks, summaries, stream, false);
}

lsa_status lsa_build_minmax_summaries(const lsa_cache *cache, const int32_t *page_table, const int32_t *seq_lens,
                                      int32_t batch, int32_t max_blocks, void *summaries, lsa_stream_t stream)
{
    return build_summaries(cache, page_table, seq_lens, batch, max_blocks, summaries, stream, true);
}

lsa_status lsa_append_block(const lsa_cache *cache, const void *k_new, const void *v_new,
                            const int32_t *page_table, int32_t *seq_lens, int32_t batch, int32_t max_blocks,
                            void *summaries, lsa_stream_t stream)
{
    return append_block(cache, k_new, v_new, page_table, seq_lens, batch, max_blocks, summaries, stream, false);
}

lsa_status lsa_append_block_minmax(const lsa_cache *cache, const void *k_new, const void *v_new,
                                   const int32_t *page_table, int32_t *seq_lens, int32_t batch, int32_t max_blocks,
                                   void *summaries, lsa_stream_t stream)
{
    return append_block(cache, k_new, v_new, page_table, seq_lens, batch, max_blocks, summaries, stream, true);
}

lsa_status lsa_score(const void *q, const lsa_cache *cache, const void *summaries, const int32_t *page_table,
                     const int32_t *seq_lens, const lsa_params *params, float *scores, lsa_stream_t stream)
{
    CacheView v;
    lsa_status rc = make_view(cache, false, &v);
    if (rc != LSA_OK) return rc;
    if ((rc = check_params(params, v)) != LSA_OK) return rc;
    if (params->batch == 0) return LSA_OK;
    if (!q || !summaries || !page_table || !seq_lens || !scores || !aligned16(q) || !aligned16(summaries))
        return LSA_ERR_INVALID_ARG;
    if (!scores_supported(v, params)) return LSA_ERR_UNSUPPORTED;
    if (params->summary_kind == LSA_SUMMARY_MINMAX && v.e4m3) return LSA_ERR_UNSUPPORTED;
    ScoreArgs a;
    memset(&a, 0, sizeof a);
    a.q = static_cast<const uint16_t *>(q);
    a.summ = static_cast<const uint16_t *>(summaries);
    a.pt = page_table;
    a.lens = seq_lens;
    a.batch = params->batch;
    a.hq = params->num_q_heads;
    a.hkv = v.hkv;
    a.dk = v.dk;
    a.b = v.b;
    a.num_pages = v.num_pages;
    a.max_blocks = params->max_blocks;
    a.sink = params->sink_tokens;
    a.recent = params->recent_tokens;
    a.chunk = score_chunk(params->batch, params->max_blocks, sm_count());
    a.scores = scores;
    a.status = status_word();
    bool unsup = false;
    cudaError_t e = launch_scores(a, params->summary_kind, reinterpret_cast<cudaStream_t>(stream), &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    return from_cuda(e);
}

lsa_status lsa_topk(const float *scores, const int32_t *num_cols, int32_t rows, int32_t cols, int32_t k,
                    int32_t *idx, lsa_stream_t stream)
{
    if (rows < 0 || cols < 0 || k < 0) return LSA_ERR_INVALID_ARG;
    if (rows == 0 || k == 0) return LSA_OK;
    if (!idx || (cols > 0 && !scores)) return LSA_ERR_INVALID_ARG;
    TopkArgs a;
    memset(&a, 0, sizeof a);
    a.scores = scores;
    a.num_cols = num_cols;
    a.rows = rows;
    a.cols = cols;
    a.k = k;
    a.idx = idx;
    a.status = status_word();
    bool unsup = false;
    cudaError_t e = launch_topk(a, reinterpret_cast<cudaStream_t>(stream), &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    return from_cuda(e);
}

lsa_status lsa_topk_approx(const float *scores, const int32_t *num_cols, int32_t rows, int32_t cols, int32_t k,
                           uint64_t seed, int32_t *idx, lsa_stream_t stream)
{
    if (rows < 0 || cols < 0 || k < 0) return LSA_ERR_INVALID_ARG;
    if (rows == 0 || k == 0) return LSA_OK;
    if (!idx || (cols > 0 && !scores)) return LSA_ERR_INVALID_ARG;
    TopkArgs a;
    memset(&a, 0, sizeof a);
    a.scores = scores;
    a.num_cols = num_cols;
    a.rows = rows;
    a.cols = cols;
    a.k = k;
    a.idx = idx;
    a.status = status_word();
    a.approx = 1;
    a.seed = seed;
    bool unsup = false;
    cudaError_t e = launch_topk(a, reinterpret_cast<cudaStream_t>(stream), &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    return from_cuda(e);
}

lsa_status lsa_fine_topk(const void *q, const lsa_cache *index_cache, const int32_t *page_table,
                         const int32_t *seq_lens, const int32_t *cand, const lsa_params *params, int32_t *tok_idx,
                         void *workspace, size_t workspace_bytes, lsa_stream_t stream)
{
    CacheView iv;
    lsa_status rc = make_view(index_cache, false, &iv);
    if (rc != LSA_OK) return rc;
    if ((rc = check_params(params, iv)) != LSA_OK) return rc;
    if (!iv.e4m3 || params->c2f_candidates <= 0) return LSA_ERR_INVALID_ARG;
    if (params->batch == 0 || params->c2f_tokens == 0) return LSA_OK;
    if (!q || !page_table || !seq_lens || !cand || !tok_idx || !aligned16(q)) return LSA_ERR_INVALID_ARG;
    const size_t rows = (size_t)params->batch * iv.hkv;
    const int64_t cols = (int64_t)params->c2f_candidates * iv.b;
    if (cols > topk_max_cols()) return LSA_ERR_UNSUPPORTED;
    const size_t need = round_up(rows * cols * sizeof(float));
    if (!workspace || workspace_bytes < need) return LSA_ERR_WORKSPACE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    FineArgs f;
    memset(&f, 0, sizeof f);
    f.q = static_cast<const uint16_t *>(q);
    f.ic = iv;
    f.pt = page_table;
    f.lens = seq_lens;
    f.cand = cand;
    f.batch = params->batch;
    f.hq = params->num_q_heads;
    f.max_blocks = params->max_blocks;
    f.ncand = params->c2f_candidates;
    f.fscores = static_cast<float *>(workspace);
    f.status = status_word();
    f.weights = params->fine_head_weights;
    bool unsup = false;
    cudaError_t e = launch_fine_scores(f, st, &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return LSA_ERR_CUDA;
    TopkArgs t;
    memset(&t, 0, sizeof t);
    t.scores = f.fscores;
    t.rows = (int32_t)rows;
    t.cols = (int32_t)cols;
    t.k = params->c2f_tokens;
    t.idx = tok_idx;
    t.cand = cand;
    t.ncand = params->c2f_candidates;
    t.b = iv.b;
    t.status = f.status;
    e = launch_topk(t, st, &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    return from_cuda(e);
}

int32_t lsa_decode_step_launches(const lsa_cache *cache, const lsa_cache *index_cache, const lsa_params *params)
{
    CacheView v;
    if (make_view(cache, true, &v) != LSA_OK || check_params(params, v) != LSA_OK) return -1;
    if (params->batch == 0) return 0;
    AttnPlan pl;
    if (plan_attention(v, params, token_mode_of(params), &pl) != LSA_OK) return -1;
    const int32_t attn = pl.flat ? 1 : 1 + ((pl.splits > 1 && !pl.umma_merge) ? 1 : 0);
    if (params->pq_candidates > 0) return 3 + attn;   // coarse scores, bucket counts, selection
    if (params->c2f_candidates > 0) {
        CacheView iv;
        if (make_view(index_cache, false, &iv) != LSA_OK) return -1;
        const bool fused = params->c2f_tokens > 0 &&
                           c2f_fine_supported(iv, params->num_q_heads, params->max_blocks, params->c2f_candidates,
                                              params->c2f_tokens, params->fine_head_weights != nullptr);
        if (fused) return 2 + attn;   // coarse scores, the cluster kernel
        return 2 + (params->c2f_tokens > 0 ? 2 : 0) + attn;
    }
    if (pl.flat && attention_flat_can_select(params->max_blocks, params->k_blocks)) return 2;
    return 1 + (params->k_blocks > 0 ? 1 : 0) + attn;
}

lsa_status lsa_pq_encode(const lsa_cache *index_cache, const void *codebook, const int32_t *page_table,
                         const int32_t *seq_lens, int32_t batch, int32_t max_blocks, uint8_t *codes,
                         lsa_stream_t stream)
{
    CacheView iv;
    lsa_status rc = make_view(index_cache, false, &iv);
    if (rc != LSA_OK) return rc;
    if (batch < 0 || (batch > 0 && max_blocks <= 0) || batch > 65535) return LSA_ERR_INVALID_ARG;
    if (!iv.e4m3 || iv.dk != 128 || iv.hkv != 1) return LSA_ERR_UNSUPPORTED;
    if (batch == 0) return LSA_OK;
    if (!codebook || !aligned16(codebook) || !page_table || !seq_lens || !codes) return LSA_ERR_INVALID_ARG;
    if ((iv.kts & 3) || (iv.kps & 3) || (reinterpret_cast<uintptr_t>(iv.k) & 3)) return LSA_ERR_INVALID_ARG;
    PqArgs a;
    memset(&a, 0, sizeof a);
    a.ic = iv;
    a.codebook = static_cast<const uint16_t *>(codebook);
    a.pt = page_table;
    a.lens = seq_lens;
    a.batch = batch;
    a.max_blocks = max_blocks;
    a.codes_out = codes;
    a.status = status_word();
    return from_cuda(launch_pq_encode(a, reinterpret_cast<cudaStream_t>(stream)));
}

lsa_status lsa_pq_scores(const void *q, const lsa_cache *index_cache, const int32_t *page_table,
                         const int32_t *seq_lens, const lsa_params *params, float *scores, lsa_stream_t stream)
{
    CacheView iv;
    lsa_status rc = make_view(index_cache, false, &iv);
    if (rc != LSA_OK) return rc;
    if ((rc = check_params(params, iv)) != LSA_OK) return rc;
    if (!iv.e4m3 || iv.dk != 128 || iv.hkv != 1 || params->num_q_heads != 64) return LSA_ERR_UNSUPPORTED;
    if (params->batch == 0) return LSA_OK;
    if (!pq_inputs_ok(q, params) || !page_table || !seq_lens || !scores) return LSA_ERR_INVALID_ARG;
    PqArgs a = pq_args(q, iv, page_table, seq_lens, params);
    a.coarse = scores;   // no row extremes or counts: scores only
    bool unsup = false;
    cudaError_t e = launch_pq_scores(a, reinterpret_cast<cudaStream_t>(stream), &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    return from_cuda(e);
}

size_t lsa_sparse_decode_workspace_size(const lsa_cache *cache, const lsa_params *params)
{
    CacheView v;
    if (make_view(cache, true, &v) != LSA_OK || check_params(params, v) != LSA_OK) return 0;
    AttnPlan pl;
    if (plan_attention(v, params, token_mode_of(params), &pl) != LSA_OK) return 0;
    return pl.ws_bytes;
}

lsa_status lsa_sparse_decode(const void *q, const lsa_cache *cache, const int32_t *page_table,
                             const int32_t *seq_lens, const int32_t *idx, const lsa_params *params, void *out,
                             float *lse, void *workspace, size_t workspace_bytes, lsa_stream_t stream)
{
    CacheView v;
    lsa_status rc = make_view(cache, true, &v);
    if (rc != LSA_OK) return rc;
    if ((rc = check_params(params, v)) != LSA_OK) return rc;
    if (params->batch == 0) return LSA_OK;
    if ((rc = check_decode_args(q, page_table, seq_lens, idx, params, out)) != LSA_OK) return rc;
    const bool token_mode = token_mode_of(params);
    const int nsel = token_mode ? params->c2f_tokens : params->k_blocks;
    return run_attention(q, v, page_table, seq_lens, nsel > 0 ? idx : nullptr, params, token_mode, out, lse,
                         static_cast<uint8_t *>(workspace), workspace_bytes,
                         reinterpret_cast<cudaStream_t>(stream));
}

size_t lsa_decode_step_workspace_size(const lsa_cache *cache, const lsa_params *params)
{
    CacheView v;
    if (make_view(cache, true, &v) != LSA_OK || check_params(params, v) != LSA_OK) return 0;
    StepLayout L;
    CacheView iv = v;   // the index cache shares paging and geometry with the attention cache
    if (step_layout(v, &iv, params, &L) != LSA_OK) return 0;
    return L.total;
}

lsa_status lsa_decode_step(const void *q, const lsa_cache *cache, const void *summaries,
                           const lsa_cache *index_cache, const int32_t *page_table, const int32_t *seq_lens,
                           const lsa_params *params, int32_t *idx_out, void *out, float *lse, void *workspace,
                           size_t workspace_bytes, lsa_stream_t stream)
{
    CacheView v;
    lsa_status rc = make_view(cache, true, &v);
    if (rc != LSA_OK) return rc;
    if ((rc = check_params(params, v)) != LSA_OK) return rc;
    const bool c2f = params->c2f_candidates > 0, pq = params->pq_candidates > 0;
    CacheView iv;
    if (c2f || pq) {
        if ((rc = make_view(index_cache, false, &iv)) != LSA_OK) return rc;
        if (!iv.e4m3 || iv.hkv != v.hkv || iv.b != v.b || iv.dk != v.dk) return LSA_ERR_INVALID_ARG;
    } else {
        iv = v;
    }
    if (params->batch == 0) return LSA_OK;
    if (pq) {
        // PQ32 coarse-to-fine: coarse scores of every encoded token and the
        // rows' bucket counts, one cluster per request for the candidates,
        // the miss filter, the exact rescoring and the token selection, then
        // attention over the selected tokens
        if (!pq_inputs_ok(q, params) || !page_table || !seq_lens || !out) return LSA_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0) return LSA_ERR_INVALID_ARG;
        if (!pq_supported(iv, params->num_q_heads, params->max_blocks, params->pq_candidates, params->c2f_tokens))
            return LSA_ERR_UNSUPPORTED;
        StepLayout L;
        if ((rc = step_layout(v, &iv, params, &L)) != LSA_OK) return rc;
        if (L.total > 0 && (!workspace || workspace_bytes < L.total)) return LSA_ERR_WORKSPACE;
        cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        const size_t rows = (size_t)params->batch;
        PqArgs a = pq_args(q, iv, page_table, seq_lens, params);
        a.coarse = reinterpret_cast<float *>(ws);
        a.tok_idx = idx_out ? idx_out : reinterpret_cast<int32_t *>(ws + L.scores);
        a.cand_out = reinterpret_cast<int32_t *>(ws + L.scores + L.sel);
        a.row_ext = reinterpret_cast<uint32_t *>(ws + L.scores + L.sel + L.cand);
        a.hist = reinterpret_cast<uint32_t *>(ws + L.scores + L.sel + L.cand + round_up(rows * 2 * sizeof(uint32_t)));
        bool unsup = false;
        cudaError_t e = launch_pq_scores(a, st, &unsup);
        if (unsup) return LSA_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return LSA_ERR_CUDA;
        e = launch_pq_select(a, st, &unsup);
        if (unsup) return LSA_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return LSA_ERR_CUDA;
        return run_attention(q, v, page_table, seq_lens, a.tok_idx, params, true, out, lse,
                             ws + L.scores + L.sel + L.cand + L.fine, L.attn, st);
    }
    if (!q || !summaries || !page_table || !seq_lens || !out || !aligned16(q) || !aligned16(summaries))
        return LSA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0) return LSA_ERR_INVALID_ARG;
    StepLayout L;
    if ((rc = step_layout(v, &iv, params, &L)) != LSA_OK) return rc;
    if (L.total > 0 && (!workspace || workspace_bytes < L.total)) return LSA_ERR_WORKSPACE;
    if (!scores_supported(iv, params)) return LSA_ERR_UNSUPPORTED;
    if (c2f && params->summary_kind != LSA_SUMMARY_MEAN) return LSA_ERR_UNSUPPORTED;
    if ((int64_t)params->max_blocks > topk_max_cols()) return LSA_ERR_UNSUPPORTED;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *scores = reinterpret_cast<float *>(ws);
    int32_t *sel = idx_out ? idx_out : reinterpret_cast<int32_t *>(ws + L.scores);
    uint8_t *ws_attn = ws + L.scores + L.sel + L.cand + L.fine;
    uint32_t *status = status_word();
    const size_t rows = (size_t)params->batch * iv.hkv;

    // coarse (or only) stage: block scores against the summaries
    ScoreArgs s;
    memset(&s, 0, sizeof s);
    s.q = static_cast<const uint16_t *>(q);
    s.summ = static_cast<const uint16_t *>(summaries);
    s.pt = page_table;
    s.lens = seq_lens;
    s.batch = params->batch;
    s.hq = params->num_q_heads;
    s.hkv = iv.hkv;
    s.dk = iv.dk;
    s.b = iv.b;
    s.num_pages = iv.num_pages;
    s.max_blocks = params->max_blocks;
    s.sink = params->sink_tokens;
    s.recent = params->recent_tokens;
    s.chunk = score_chunk(params->batch, params->max_blocks, sm_count());
    s.scores = scores;
    s.status = status;
    int32_t *cand = reinterpret_cast<int32_t *>(ws + L.scores + L.sel);
    const bool fused = c2f && params->c2f_tokens > 0 &&
                       c2f_fine_supported(iv, params->num_q_heads, params->max_blocks, params->c2f_candidates,
                                          params->c2f_tokens, params->fine_head_weights != nullptr);
    bool unsup = false;
    cudaError_t e = launch_scores(s, params->summary_kind, st, &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return LSA_ERR_CUDA;

    TopkArgs t;
    memset(&t, 0, sizeof t);
    t.scores = scores;
    t.rows = (int32_t)rows;
    t.cols = params->max_blocks;
    t.status = status;
    if (!c2f) {
        // with the even-split attention the attention kernel selects the
        // blocks itself (no top-k launch, the selection stays on chip)
        AttnPlan apl;
        if (plan_attention(v, params, false, &apl) == LSA_OK && apl.flat &&
            attention_flat_can_select(params->max_blocks, params->k_blocks))
            return run_attention(q, v, page_table, seq_lens, nullptr, params, false, out, lse, ws_attn, L.attn, st,
                                 scores, idx_out);
        t.k = params->k_blocks;
        t.idx = sel;
        e = launch_topk(t, st, &unsup);
        if (unsup) return LSA_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return LSA_ERR_CUDA;
        return run_attention(q, v, page_table, seq_lens, params->k_blocks > 0 ? sel : nullptr, params, false,
                             out, lse, ws_attn, L.attn, st);
    }
    if (fused) {
        // one cluster per request selects the candidates, rescores their
        // tokens and selects the tokens; then attention over them
        FineArgs f;
        memset(&f, 0, sizeof f);
        f.q = static_cast<const uint16_t *>(q);
        f.ic = iv;
        f.pt = page_table;
        f.lens = seq_lens;
        f.batch = params->batch;
        f.hq = params->num_q_heads;
        f.max_blocks = params->max_blocks;
        f.ncand = params->c2f_candidates;
        f.status = status;
        f.weights = params->fine_head_weights;
        f.coarse = scores;
        f.cand_out = cand;
        f.tok_k = params->c2f_tokens;
        f.tok_idx = sel;
        e = launch_c2f_fine(f, st, &unsup);
        if (unsup) return LSA_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return LSA_ERR_CUDA;
        return run_attention(q, v, page_table, seq_lens, sel, params, true, out, lse, ws_attn, L.attn, st);
    }
    // coarse-to-fine in separate stages: top-C candidate blocks, exact FP8
    // rescoring, token top-k
    t.k = params->c2f_candidates;
    t.idx = cand;
    e = launch_topk(t, st, &unsup);
    if (unsup) return LSA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return LSA_ERR_CUDA;
    rc = lsa_fine_topk(q, index_cache, page_table, seq_lens, cand, params, sel, ws + L.scores + L.sel + L.cand,
                       L.fine, stream);
    if (rc != LSA_OK) return rc;
    return run_attention(q, v, page_table, seq_lens, params->c2f_tokens > 0 ? sel : nullptr, params, true, out,
                         lse, ws_attn, L.attn, st);
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation variant
//
// lsa_sparse_decode_static_scratch: the scratch that lsa_sparse_decode takes
// from the caller lives here instead, in a file-scope static device array
// (zero-initialised when the module loads).  Nothing is allocated per call;
// the array's address is looked up once per device with that device current.

namespace lsa {
namespace {

constexpr size_t kStaticScratchBytes = LSA_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {};
// What the buffer of each device last served.  A call leaves the counters
// it needs at zero for the next call with the same layout, but another
// shape, or another attention plan for the same shape (LSA_ATTENTION_PATH
// picks the kernel per call), lays its counters over bytes the previous
// one used for data.
struct ScratchUse {
    lsa_cache cache;
    lsa_params params;
    AttnPlan plan;
    bool valid;
};
ScratchUse g_static_use[kMaxDevices] = {};

bool same_plan(const AttnPlan &a, const AttnPlan &b)
{
    return a.nsub == b.nsub && a.splits == b.splits && a.items_per_split == b.items_per_split &&
           a.tc_group == b.tc_group && a.umma == b.umma && a.umma_merge == b.umma_merge && a.flat == b.flat && a.fl_ns == b.fl_ns && a.fl_ctas == b.fl_ctas &&
           a.fl_parts == b.fl_parts && a.fl_total == b.fl_total && a.ws_bytes == b.ws_bytes;
}

// The device's buffer; when the call's shape or plan differs from the one
// the buffer served last (or a device error was reported since), the bytes
// it needs are cleared first (on the call's stream: a memset, no
// allocation).
lsa_status static_scratch_for_current_device(const lsa_cache *cache, const lsa_params *params, const AttnPlan &plan,
                                             cudaStream_t st, void **ptr)
{
    const int dev = current_device();
    if (dev < 0) return LSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return LSA_ERR_CUDA;
        g_static_ptr[dev] = p;
    }
    ScratchUse &u = g_static_use[dev];
    const bool same = u.valid && same_plan(u.plan, plan) && memcmp(&u.cache, cache, sizeof *cache) == 0 &&
                      memcmp(&u.params, params, sizeof *params) == 0;
    if (!same) {
        u.valid = false;
        if (plan.ws_bytes > 0 && cudaMemsetAsync(g_static_ptr[dev], 0, plan.ws_bytes, st) != cudaSuccess)
            return LSA_ERR_CUDA;
        u.cache = *cache;
        u.params = *params;
        u.plan = plan;
        u.valid = true;
    }
    *ptr = g_static_ptr[dev];
    return LSA_OK;
}

}  // namespace

void static_scratch_forget(int dev)
{
    if (dev < 0 || dev >= kMaxDevices) return;
    std::lock_guard<std::mutex> lock(g_static_mu);
    g_static_use[dev].valid = false;
}

}  // namespace lsa

extern "C" lsa_status lsa_sparse_decode_static_scratch(const void *q, const lsa_cache *cache,
                                                       const int32_t *page_table, const int32_t *seq_lens,
                                                       const int32_t *idx, const lsa_params *params, void *out,
                                                       float *lse, lsa_stream_t stream)
{
    CacheView v;
    lsa_status rc = make_view(cache, true, &v);
    if (rc != LSA_OK) return rc;
    if ((rc = check_params(params, v)) != LSA_OK) return rc;
    AttnPlan plan;
    if ((rc = plan_attention(v, params, token_mode_of(params), &plan)) != LSA_OK) return rc;
    if (plan.ws_bytes > kStaticScratchBytes) return LSA_ERR_WORKSPACE;
    if (params->batch == 0) return LSA_OK;
    if ((rc = check_decode_args(q, page_table, seq_lens, idx, params, out)) != LSA_OK) return rc;
    void *scratch = nullptr;
    if ((rc = static_scratch_for_current_device(cache, params, plan, reinterpret_cast<cudaStream_t>(stream),
                                                &scratch)) != LSA_OK)
        return rc;
    return lsa_sparse_decode(q, cache, page_table, seq_lens, idx, params, out, lse, scratch, kStaticScratchBytes,
                             stream);
}

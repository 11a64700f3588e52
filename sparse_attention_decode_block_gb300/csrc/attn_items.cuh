// Item planning shared by the split-K attention kernels: the attended token
// set of one (request, KV head) row is walked in 16-token items -- forced
// sink tokens, then the selected blocks (or single selected tokens), then the
// forced recent tokens -- and each item is resolved to a run of token rows
// within one page.
#pragma once

#include "lsa_device.cuh"

namespace lsa {
namespace {

// Row plan of one (request): forced ranges and item counts.
struct RowPlan {
    int L, se, rs;
    int nsc, nsel_items, nrc, n_items;
};

__device__ __forceinline__ RowPlan plan_of_len(const AttnArgs &a, int L, bool flag_bad)
{
    RowPlan pl;
    if (L < 0 || (int64_t)L > (int64_t)a.max_blocks * a.c.b) {
        if (flag_bad) flag_error(a.status, LSA_ERR_BOUNDS);
        L = 0;
    }
    pl.L = L;
    pl.se = min(a.sink, L);
    pl.rs = max(L - a.recent, pl.se);
    pl.nsc = (pl.se + kChunk - 1) / kChunk;
    pl.nsel_items = a.token_mode ? (a.nsel + kChunk - 1) / kChunk : a.nsel * (a.c.b / kChunk);
    pl.nrc = L > pl.rs ? (L + kChunk - 1) / kChunk - pl.rs / kChunk : 0;
    pl.n_items = pl.nsc + pl.nsel_items + pl.nrc;
    return pl;
}

__device__ __forceinline__ RowPlan make_plan(const AttnArgs &a, int r, bool flag_bad)
{
    return plan_of_len(a, a.lens[r], flag_bad);
}

// Selected-block item k of a row: the selection entry it reads and the one
// before it (for the ascending check), or (-1, -1) when k is not a
// selected-block item under a plan whose sink covers nsc items.
__device__ __forceinline__ int2 item_sel_entries(const AttnArgs &a, int r, int h, int nsc, int i)
{
    const int k = i - nsc, cpb = (int)a.fd_cpb.d;
    if (a.token_mode || k < 0 || k >= a.nsel * cpb) return make_int2(-1, -1);
    const int ei = (int)fdiv((uint32_t)k, a.fd_cpb);
    const int32_t *irow = a.idx + ((int64_t)r * a.c.hkv + h) * a.nsel;
    return make_int2(irow[ei], ei > 0 ? irow[ei - 1] : -1);
}

// Resolves item i of row (r, h) to a run of token rows within one page:
// d = {page, slot of the first token, rows}; rows = 0 for nothing to attend,
// rows = -1 for a token-list item (rows resolved per token).
__device__ ItemDesc describe_item_sel(const AttnArgs &a, const RowPlan &pl, int r, int h, int i, int2 sel);

__device__ ItemDesc describe_item(const AttnArgs &a, const RowPlan &pl, int r, int h, int i)
{
    const int2 sel = (i >= pl.nsc && i < pl.nsc + pl.nsel_items) ? item_sel_entries(a, r, h, pl.nsc, i)
                                                                  : make_int2(-1, -1);
    return describe_item_sel(a, pl, r, h, i, sel);
}

// As describe_item, with the item's selection entries (item_sel_entries
// under this plan) already loaded and the page id of block j of request r
// read by page_of(r, j).
template <class PageOf>
__device__ __forceinline__ ItemDesc describe_item_with(const AttnArgs &a, const RowPlan &pl, int r, int h, int i,
                                                       int2 sel, PageOf page_of)
{
    const int b = a.c.b;
    ItemDesc d;
    d.page = -1;
    d.ts = 0;
    d.n = 0;
    int t0 = 0, n = 0;
    if (i < pl.nsc) {
        t0 = i * kChunk;
        n = min(kChunk, pl.se - t0);
    } else if (i < pl.nsc + pl.nsel_items) {
        if (a.token_mode) {
            d.n = -1;
            return d;
        }
        const int k = i - pl.nsc;
        const int ck = (int)fmodu((uint32_t)k, a.fd_cpb);
        const int e = sel.x, prev = sel.y;
        const bool valid = e >= 0 && e < a.max_blocks && (int64_t)e * b >= pl.se &&
                           (int64_t)(e + 1) * b <= pl.rs && prev < e;
        if (!valid && e != -1 && ck == 0) flag_error(a.status, LSA_ERR_BOUNDS);
        if (valid) {
            t0 = e * b + ck * kChunk;
            n = kChunk;
        }
    } else {
        const int k = i - pl.nsc - pl.nsel_items;
        const int blk16 = pl.rs / kChunk + k;
        t0 = max(pl.rs, blk16 * kChunk);
        n = min(pl.L, blk16 * kChunk + kChunk) - t0;
    }
    if (n <= 0) return d;
    const uint32_t tb = fdiv((uint32_t)t0, a.fd_b);
    const int p = page_of(r, (int)tb);
    if (p < 0 || p >= a.c.num_pages) {
        flag_error(a.status, LSA_ERR_BOUNDS);
        return d;
    }
    d.page = p;
    d.ts = (int16_t)(t0 - (int)tb * b);
    d.n = (int16_t)n;
    return d;
}

__device__ ItemDesc describe_item_sel(const AttnArgs &a, const RowPlan &pl, int r, int h, int i, int2 sel)
{
    return describe_item_with(a, pl, r, h, i, sel,
                              [&](int rq, int j) { return a.pt[(int64_t)rq * a.max_blocks + j]; });
}

// Token-list rows: entry u of token-list item i -> (page, slot) or page -1.
__device__ int2 describe_token(const AttnArgs &a, const RowPlan &pl, int r, int h, int i, int u)
{
    const int b = a.c.b;
    int2 row = make_int2(-1, 0);
    const int ei = (i - pl.nsc) * kChunk + u;
    if (ei >= a.nsel) return row;
    const int32_t *irow = a.idx + ((int64_t)r * a.c.hkv + h) * a.nsel;
    const int t = irow[ei];
    const int prev = ei > 0 ? irow[ei - 1] : -1;
    if (t == -1) return row;
    const int j = t / b;
    // a selected token is any token outside the forced ranges (it may lie in
    // the partial last block: the PQ32 selection rescores that tail)
    const bool valid = t >= 0 && (int64_t)t >= pl.se && (int64_t)t < pl.rs && prev < t;
    if (!valid) {
        flag_error(a.status, LSA_ERR_BOUNDS);
        return row;
    }
    const int p = a.pt[(int64_t)r * a.max_blocks + j];
    if (p < 0 || p >= a.c.num_pages) {
        flag_error(a.status, LSA_ERR_BOUNDS);
        return row;
    }
    return make_int2(p, t % b);
}

}  // namespace
}  // namespace lsa

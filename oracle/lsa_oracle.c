/*
 * lsa_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * block-sparse decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the bench's
 * CPU-baseline leg are the only callers.  It shares no source, header, table
 * or helper with the CUDA library; the two meet only through the seeded
 * input generator (the `workloads` package), which holds none of the
 * method's arithmetic.
 *
 * Everything is computed in double precision from the bf16 / e4m3 inputs.
 * The method, as the pages define it:
 *
 *   summary   k_bar_j = mean of the b keys of block j, built once the block
 *             is full (Vortex blog post, "Block top-k attention", Figure 1
 *             and the forward_cache of the vFlow listing); stored as bf16.
 *   score     s_j = q . k_bar_j (Vortex, block top-k equation), summed over
 *             the query heads of a KV head's GQA group (the vFlow listing
 *             reduces the GeMM output over the head dimension; a sum equals
 *             that mean times the group size, which orders blocks the same).
 *   select    I = top-k_j(s_j), ties to the lower block index, with the sink
 *             tokens and the most recent tokens always attended (ByteCross,
 *             Figure 1 caption and Appendix A "Scored selection"; Vortex
 *             cites StreamingLLM for sinks plus a recent window).
 *   attend    o = softmax(q K_T^T * scale) V_T over the attended token set T
 *             (Vortex, block top-k equation).
 *   coarse-to-fine: a coarse top-C over block summaries of the index keys,
 *             then an exact rescoring of every token of the C blocks with its
 *             FP8 e4m3 index key and per-token scale, keeping the top tokens
 *             (LeanSparse, Section 5 "Coarse-to-fine decode indexing",
 *             Figure 9; 132-byte FP8 key + scale).
 *   merge     partial results over a partition of T combine by log-sum-exp
 *             (ByteCross, Appendix A: sink call and window call merged by
 *             log-sum-exp).
 *   Quest     an alternative summary and score (Vortex blog post, end of
 *             "Why Long Generations Are Expensive", and the Quest listing in
 *             "Writing an algorithm: vFlow"): each block keeps the
 *             element-wise maximum and minimum of its keys, and a block's
 *             score for query head g is sum_i max(q_gi * max_i, q_gi * min_i),
 *             an upper bound on q_g . k_t for every token t of the block;
 *             the listing's Max over the query heads of the GQA group makes
 *             the block score.
 *
 * Readings where the pages leave a step open are stated beside each step.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 bit pattern -> double (bf16 is the top half of an IEEE binary32). */
double orc_bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> bf16, round to nearest, ties to even, in one rounding step.
 * bf16 keeps 8 significant bits; normal numbers start at 2^-126 and the
 * subnormal spacing is 2^-133 (binary32's exponent range). */
uint16_t orc_f64_to_bf16(double x)
{
    if (isnan(x))
        return 0x7fc0;
    uint16_t s = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a))
        return s | 0x7f80;
    if (a == 0.0)
        return s;
    int e;
    (void)frexp(a, &e);            /* a = m * 2^e, m in [0.5, 1) */
    int qe = e - 8;                /* spacing of 8-significant-bit numbers */
    if (qe < -133)
        qe = -133;
    double r = nearbyint(ldexp(a, -qe));   /* default mode: ties to even */
    double y = ldexp(r, qe);
    if (y >= 0x1p128)
        return s | 0x7f80;
    float f = (float)y;            /* exact: y is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return s | (uint16_t)(u >> 16);
}

/* OCP FP8 E4M3 ("fn": no infinities, S.1111.111 is NaN), bias 7. */
double orc_e4m3_to_f64(uint8_t c)
{
    int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7)
        return NAN;
    double v = (e == 0) ? ldexp((double)m, -9)         /* m/8 * 2^-6      */
                        : ldexp((double)(8 + m), e - 10); /* (1+m/8) 2^(e-7) */
    return sgn ? -v : v;
}

/* ------------------------------------------------------------------ */
/* Inputs                                                              */
/* ------------------------------------------------------------------ */

typedef struct {
    int32_t num_pages, num_kv_heads, block_size, dk, dv;
    const uint16_t *k;        /* [P, Hkv, b, dk] bf16, contiguous       */
    const uint16_t *v;        /* [P, Hkv, b, dv] bf16, contiguous       */
    const uint8_t *k8;        /* [P, Hkv, b, dk] e4m3 index keys or NULL */
    const float *k8_scale;    /* [P, Hkv, b] per-token scale or NULL     */
} orc_cache;

typedef struct {
    int32_t batch, num_q_heads, max_blocks;
    int32_t k_blocks;          /* scored blocks to select, forced excluded */
    int32_t sink, recent;      /* forced token ranges                      */
    double scale;              /* softmax scale                            */
    int32_t c2f_candidates;    /* 0: single stage                          */
    int32_t c2f_tokens;
    int32_t summary_kind;      /* 0: mean keys; 1: Quest min/max keys      */
    const float *fine_weights; /* NULL, or [batch, num_q_heads] indexer
                                  head weights of the weighted-ReLU fine score */
    /* PQ32 coarse-to-fine (pq_candidates > 0): token-level coarse scores
     * from product-quantised index keys, a miss filter, then the exact
     * weighted-ReLU rescoring (fine_weights required) */
    int32_t pq_candidates;     /* C: token candidates of the coarse pass    */
    const uint8_t *pq_codes;   /* [P, Hkv, b, 32] one byte per 4-dim subvector */
    const uint16_t *pq_codebook; /* [32, 256, 4] bf16 centroids            */
    const uint8_t *pq_hit;     /* [P, Hkv, b] 1: the token's original index
                                  key is cached (NULL: every token is)      */
} orc_params;

enum { ORC_OK = 0, ORC_BAD_PAGE = 1, ORC_BAD_ARG = 2, ORC_NOMEM = 3 };

static double key_elem(const orc_cache *c, int use_k8, int64_t p, int h, int t, int i)
{
    int64_t base = ((p * c->num_kv_heads + h) * (int64_t)c->block_size + t);
    if (use_k8)
        return (double)c->k8_scale[base] * orc_e4m3_to_f64(c->k8[base * c->dk + i]);
    return orc_bf16_to_f64(c->k[base * c->dk + i]);
}

static double val_elem(const orc_cache *c, int64_t p, int h, int t, int i)
{
    int64_t base = ((p * c->num_kv_heads + h) * (int64_t)c->block_size + t);
    return orc_bf16_to_f64(c->v[base * c->dv + i]);
}

/* Forced ranges F = [0, sink_end) U [rec_start, L), with the recent range
 * clipped so that the two never overlap.  Reading: when L < sink + recent
 * the two ranges cover every token. */
static void forced_ranges(int64_t L, int32_t sink, int32_t recent,
                          int64_t *sink_end, int64_t *rec_start)
{
    int64_t se = sink < L ? sink : L;
    int64_t rs = L - recent;
    if (rs < se)
        rs = se;
    *sink_end = se;
    *rec_start = rs;
}

/* Block j is a scoring candidate iff it is full and none of its tokens is
 * forced.  Reading: a partial tail block has no summary until it fills, and
 * a block touching a forced range is attended (in part) anyway. */
static int is_candidate(int64_t j, int32_t b, int64_t sink_end, int64_t rec_start)
{
    return j * b >= sink_end && (j + 1) * b <= rec_start;
}

/* ------------------------------------------------------------------ */
/* Step: block summaries                                               */
/* ------------------------------------------------------------------ */

/* Mean of the b keys of (page p, head h), exact fp64 sum, one rounding. */
static void summary_of(const orc_cache *c, int use_k8, int64_t p, int h, double *out)
{
    const int b = c->block_size;
    for (int i = 0; i < c->dk; ++i) {
        double sum = 0.0;
        for (int t = 0; t < b; ++t)
            sum += key_elem(c, use_k8, p, h, t, i);
        out[i] = orc_bf16_to_f64(orc_f64_to_bf16(sum / (double)b));
    }
}

/* Summaries of every full block referenced by the page tables.
 * summ: [P, Hkv, dk] bf16 bits (untouched for pages with no full block);
 * valid: [P] set to 1 for pages written (may be NULL). */
int orc_summaries(const orc_cache *c, int use_k8, const int32_t *pt, const int32_t *lens,
                  int32_t batch, int32_t max_blocks, uint16_t *summ, uint8_t *valid)
{
    double *tmp = (double *)malloc(sizeof(double) * (size_t)c->dk);
    if (!tmp)
        return ORC_NOMEM;
    for (int r = 0; r < batch; ++r) {
        int64_t nfull = lens[r] / c->block_size;
        for (int64_t j = 0; j < nfull; ++j) {
            int64_t p = pt[(int64_t)r * max_blocks + j];
            if (p < 0 || p >= c->num_pages) {
                free(tmp);
                return ORC_BAD_PAGE;
            }
            for (int h = 0; h < c->num_kv_heads; ++h) {
                summary_of(c, use_k8, p, h, tmp);
                for (int i = 0; i < c->dk; ++i)
                    summ[((int64_t)p * c->num_kv_heads + h) * c->dk + i] = orc_f64_to_bf16(tmp[i]);
            }
            if (valid)
                valid[p] = 1;
        }
    }
    free(tmp);
    return ORC_OK;
}

/* Quest summaries of (page p, head h): element-wise maximum and minimum of
 * the b keys (exact: they are key values). */
static void quest_summary_of(const orc_cache *c, int64_t p, int h, double *mx, double *mn)
{
    const int b = c->block_size;
    for (int i = 0; i < c->dk; ++i) {
        double hi = -INFINITY, lo = INFINITY;
        for (int t = 0; t < b; ++t) {
            double x = key_elem(c, 0, p, h, t, i);
            if (x > hi)
                hi = x;
            if (x < lo)
                lo = x;
        }
        mx[i] = hi;
        mn[i] = lo;
    }
}

/* Quest summaries of every full block referenced by the page tables:
 * summ [P, Hkv, 2, dk] bf16 bits, the maximum keys then the minimum keys
 * (untouched for pages with no full block); valid: [P] (may be NULL). */
int orc_quest_summaries(const orc_cache *c, const int32_t *pt, const int32_t *lens, int32_t batch,
                        int32_t max_blocks, uint16_t *summ, uint8_t *valid)
{
    double *mx = (double *)malloc(sizeof(double) * 2 * (size_t)c->dk);
    if (!mx)
        return ORC_NOMEM;
    double *mn = mx + c->dk;
    for (int r = 0; r < batch; ++r) {
        int64_t nfull = lens[r] / c->block_size;
        for (int64_t j = 0; j < nfull; ++j) {
            int64_t p = pt[(int64_t)r * max_blocks + j];
            if (p < 0 || p >= c->num_pages) {
                free(mx);
                return ORC_BAD_PAGE;
            }
            for (int h = 0; h < c->num_kv_heads; ++h) {
                quest_summary_of(c, p, h, mx, mn);
                uint16_t *dst = summ + ((int64_t)p * c->num_kv_heads + h) * 2 * c->dk;
                for (int i = 0; i < c->dk; ++i) {
                    dst[i] = orc_f64_to_bf16(mx[i]);
                    dst[c->dk + i] = orc_f64_to_bf16(mn[i]);
                }
            }
            if (valid)
                valid[p] = 1;
        }
    }
    free(mx);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Step: block scores                                                  */
/* ------------------------------------------------------------------ */

static void load_summary(const orc_cache *c, int use_k8, const uint16_t *summ,
                         int64_t p, int h, double *out)
{
    if (summ) {
        for (int i = 0; i < c->dk; ++i)
            out[i] = orc_bf16_to_f64(summ[((int64_t)p * c->num_kv_heads + h) * c->dk + i]);
    } else {
        summary_of(c, use_k8, p, h, out);
    }
}

/* s_j = sum over the group's query heads g of q_g . k_bar_j, for every
 * candidate block j; -inf for every other j < max_blocks. */
static int row_scores(const uint16_t *q, const orc_cache *c, int use_k8, const uint16_t *summ,
                      const int32_t *pt, int64_t L, const orc_params *prm, int r, int h,
                      double *scores)
{
    const int b = c->block_size, dk = c->dk;
    const int G = prm->num_q_heads / c->num_kv_heads;
    int64_t se, rs;
    forced_ranges(L, prm->sink, prm->recent, &se, &rs);
    double *sv = (double *)malloc(sizeof(double) * 2 * (size_t)dk);
    if (!sv)
        return ORC_NOMEM;
    for (int64_t j = 0; j < prm->max_blocks; ++j) {
        scores[j] = -INFINITY;
        if (!is_candidate(j, b, se, rs))
            continue;
        int64_t p = pt[(int64_t)r * prm->max_blocks + j];
        if (p < 0 || p >= c->num_pages) {
            free(sv);
            return ORC_BAD_PAGE;
        }
        if (prm->summary_kind == 1) {
            /* Quest: max over the group's heads of sum_i max(q*max, q*min) */
            double best = -INFINITY;
            if (summ) {
                const uint16_t *src = summ + ((int64_t)p * c->num_kv_heads + h) * 2 * dk;
                for (int i = 0; i < dk; ++i) {
                    sv[i] = orc_bf16_to_f64(src[i]);
                    sv[dk + i] = orc_bf16_to_f64(src[dk + i]);
                }
            } else {
                quest_summary_of(c, p, h, sv, sv + dk);
            }
            for (int g = 0; g < G; ++g) {
                const uint16_t *qg = q + ((int64_t)r * prm->num_q_heads + h * G + g) * dk;
                double s = 0.0;
                for (int i = 0; i < dk; ++i) {
                    double qi = orc_bf16_to_f64(qg[i]);
                    double a = qi * sv[i], bb = qi * sv[dk + i];
                    s += a > bb ? a : bb;
                }
                if (s > best)
                    best = s;
            }
            scores[j] = best;
            continue;
        }
        load_summary(c, use_k8, summ, p, h, sv);
        double s = 0.0;
        for (int g = 0; g < G; ++g) {
            const uint16_t *qg = q + ((int64_t)r * prm->num_q_heads + h * G + g) * dk;
            for (int i = 0; i < dk; ++i)
                s += orc_bf16_to_f64(qg[i]) * sv[i];
        }
        scores[j] = s;
    }
    free(sv);
    return ORC_OK;
}

int orc_block_scores(const uint16_t *q, const orc_cache *c, int use_k8, const uint16_t *summ,
                     const int32_t *pt, const int32_t *lens, const orc_params *prm,
                     double *scores /* [B, Hkv, max_blocks] */)
{
    for (int r = 0; r < prm->batch; ++r)
        for (int h = 0; h < c->num_kv_heads; ++h) {
            int rc = row_scores(q, c, use_k8, summ, pt, lens[r], prm, r, h,
                                scores + ((int64_t)r * c->num_kv_heads + h) * prm->max_blocks);
            if (rc)
                return rc;
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Step: top-k                                                         */
/* ------------------------------------------------------------------ */

typedef struct {
    double s;
    int64_t j;
} scored;

/* Order: larger score first; equal scores -> lower index first. */
static int by_score_then_index(const void *a, const void *b)
{
    const scored *x = (const scored *)a, *y = (const scored *)b;
    if (x->s > y->s)
        return -1;
    if (x->s < y->s)
        return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int by_index(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x < y) ? -1 : (x > y);
}

/* The k best of the n entries by (score desc, index asc).  Entries that are
 * -inf or NaN are not candidates.  Output: the chosen indices in ascending
 * order, then -1 padding up to k.  Returns the number chosen. */
static int64_t select_topk(const double *s, const int64_t *ids, int64_t n, int64_t k, int64_t *out)
{
    scored *v = (scored *)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(s[i]) || s[i] == -INFINITY)
            continue;
        v[m].s = s[i];
        v[m].j = ids ? ids[i] : i;
        ++m;
    }
    qsort(v, (size_t)m, sizeof(scored), by_score_then_index);
    int64_t take = m < k ? m : k;
    for (int64_t i = 0; i < take; ++i)
        out[i] = v[i].j;
    qsort(out, (size_t)take, sizeof(int64_t), by_index);
    for (int64_t i = take; i < k; ++i)
        out[i] = -1;
    free(v);
    return take;
}

int orc_topk(const double *scores, int32_t n, int32_t k, int32_t *out)
{
    int64_t *tmp = (int64_t *)malloc(sizeof(int64_t) * (size_t)(k > 0 ? k : 1));
    if (!tmp)
        return ORC_NOMEM;
    select_topk(scores, NULL, n, k, tmp);
    for (int i = 0; i < k; ++i)
        out[i] = (int32_t)tmp[i];
    free(tmp);
    return ORC_OK;
}

/* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): the state advances by the golden-ratio
 * increment 0x9e3779b97f4a7c15 and each output is the state passed through
 * the variant-13 finaliser (xor-shift 30, multiply, xor-shift 27, multiply,
 * xor-shift 31).  Used counter-style: output n (n >= 1) of the generator
 * seeded with `seed` is mix(seed + n * increment). */
uint64_t orc_splitmix64(uint64_t seed, uint64_t n)
{
    uint64_t z = seed + n * 0x9e3779b97f4a7c15ULL;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

/* Approximate top-k with a stochastic early exit (Vortex blog post, "Making
 * it fast": a monotone remap spreads the scores over the buckets, and the
 * selection stops once it has enough confident winners, sampling the rest
 * from the boundary bucket).  The steps, in that order, for one row of n
 * fp32 scores (-inf and NaN are not candidates; keff = min(k, candidates)):
 *   1. remap: bucket(x) = floor((x - vmin) * (nbins / (vmax - vmin))),
 *      clamped to nbins - 1, over the candidates' smallest and largest
 *      value, in fp32 (one bucket when vmax == vmin or the span is not
 *      finite); larger values never fall in lower buckets;
 *   2. the boundary bucket B holds the keff-th largest value: the G
 *      candidates in buckets above B are the confident winners (G < keff);
 *   3. the remaining keff - G are sampled from the cnt candidates of B: in
 *      column order they are numbered 0 .. cnt-1, and those whose number is
 *      within keff - G steps after off = splitmix64(seed, row + 1) mod cnt,
 *      circularly, are taken (every one of them is taken with probability
 *      (keff - G) / cnt over the seed).
 * Output: the chosen columns ascending, -1 padded to k. */
int orc_topk_approx(const float *scores, int32_t n, int32_t k, int32_t nbins, uint64_t seed, int64_t row,
                    int32_t *out)
{
    if (nbins < 1)
        return ORC_BAD_ARG;
    int32_t m = 0;
    float vmin = INFINITY, vmax = -INFINITY;
    for (int32_t i = 0; i < n; ++i) {
        const float x = scores[i];
        if (isnan(x) || x == -INFINITY)
            continue;
        ++m;
        if (x < vmin)
            vmin = x;
        if (x > vmax)
            vmax = x;
    }
    const int32_t keff = k < m ? (k > 0 ? k : 0) : m;
    int32_t nout = 0;
    if (keff == m) {
        for (int32_t i = 0; i < n; ++i)
            if (!(isnan(scores[i]) || scores[i] == -INFINITY))
                out[nout++] = i;
    } else if (keff > 0) {
        const float span = vmax - vmin;
        const float scale = (span > 0.0f && span < INFINITY) ? (float)nbins / span : 0.0f;
        int32_t *bucket = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
        int64_t *count = (int64_t *)calloc((size_t)nbins, sizeof(int64_t));
        if (!bucket || !count) {
            free(bucket);
            free(count);
            return ORC_NOMEM;
        }
        for (int32_t i = 0; i < n; ++i) {
            const float x = scores[i];
            bucket[i] = -1;
            if (isnan(x) || x == -INFINITY)
                continue;
            int32_t bk = 0;
            if (scale != 0.0f) {
                const float y = (x - vmin) * scale;
                bk = y >= (float)(nbins - 1) ? nbins - 1 : (int32_t)y;
            }
            bucket[i] = bk;
            count[bk]++;
        }
        int64_t above = 0;
        int32_t B = nbins - 1;
        while (above + count[B] < keff) {
            above += count[B];
            --B;
        }
        const int64_t cnt = count[B], take = keff - above;
        const int64_t off = (int64_t)(orc_splitmix64(seed, (uint64_t)row + 1) % (uint64_t)cnt);
        int64_t rank = 0;
        for (int32_t i = 0; i < n; ++i) {
            if (bucket[i] > B) {
                out[nout++] = i;
            } else if (bucket[i] == B) {
                if ((rank - off + cnt) % cnt < take)
                    out[nout++] = i;
                ++rank;
            }
        }
        free(bucket);
        free(count);
    }
    for (int32_t i = nout; i < k; ++i)
        out[i] = -1;
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Step: attention over a token set                                    */
/* ------------------------------------------------------------------ */

/* o = softmax(scale * q K_T^T) V_T over the listed token positions of
 * request r, KV head h; lse = log sum exp(scale * q K_T^T).  An empty set
 * gives o = 0 and lse = -inf (reading: nothing to attend). */
static int attend(const double *qd, const orc_cache *c, const int32_t *pt_row, int64_t ntok,
                  const int64_t *tok, int h, double scale, double *o, double *lse)
{
    const int b = c->block_size, dk = c->dk, dv = c->dv;
    for (int i = 0; i < dv; ++i)
        o[i] = 0.0;
    if (ntok == 0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    double *z = (double *)malloc(sizeof(double) * (size_t)ntok);
    if (!z)
        return ORC_NOMEM;
    double zmax = -INFINITY;
    for (int64_t n = 0; n < ntok; ++n) {
        int64_t t = tok[n];
        int64_t p = pt_row[t / b];
        if (p < 0 || p >= c->num_pages) {
            free(z);
            return ORC_BAD_PAGE;
        }
        double d = 0.0;
        for (int i = 0; i < dk; ++i)
            d += qd[i] * key_elem(c, 0, p, h, (int)(t % b), i);
        z[n] = scale * d;
        if (z[n] > zmax)
            zmax = z[n];
    }
    double denom = 0.0;
    for (int64_t n = 0; n < ntok; ++n) {
        int64_t t = tok[n];
        int64_t p = pt_row[t / b];
        double w = exp(z[n] - zmax);
        denom += w;
        for (int i = 0; i < dv; ++i)
            o[i] += w * val_elem(c, p, h, (int)(t % b), i);
    }
    for (int i = 0; i < dv; ++i)
        o[i] /= denom;
    *lse = zmax + log(denom);
    free(z);
    return ORC_OK;
}

/* Attention of every query head of (r, h) over a given token list.
 * out: [Hq, dv] doubles for this request (rows h*G .. h*G+G-1 written). */
static int attend_group(const uint16_t *q, const orc_cache *c, const int32_t *pt_row,
                        const orc_params *prm, int r, int h, int64_t ntok, const int64_t *tok,
                        uint16_t *out, double *lse_out)
{
    const int G = prm->num_q_heads / c->num_kv_heads, dk = c->dk, dv = c->dv;
    double *qd = (double *)malloc(sizeof(double) * (size_t)dk);
    double *o = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!qd || !o) {
        free(qd);
        free(o);
        return ORC_NOMEM;
    }
    int rc = ORC_OK;
    for (int g = 0; g < G && rc == ORC_OK; ++g) {
        int hq = h * G + g;
        const uint16_t *qg = q + ((int64_t)r * prm->num_q_heads + hq) * dk;
        for (int i = 0; i < dk; ++i)
            qd[i] = orc_bf16_to_f64(qg[i]);
        double lse;
        rc = attend(qd, c, pt_row, ntok, tok, h, prm->scale, o, &lse);
        for (int i = 0; i < dv; ++i)
            out[((int64_t)r * prm->num_q_heads + hq) * dv + i] = orc_f64_to_bf16(o[i]);
        lse_out[(int64_t)r * prm->num_q_heads + hq] = lse;
    }
    free(qd);
    free(o);
    return rc;
}

/* ------------------------------------------------------------------ */
/* Step: coarse-to-fine token rescoring                                */
/* ------------------------------------------------------------------ */

/* f_t = scale_t * sum_g q_g . e4m3(k8_t) for every token of the given
 * blocks (ascending), written to f / tok (n = nblocks * b entries).
 * With head weights w (prm->fine_weights), the indexer's weighted head
 * aggregation instead (LeanSparse, Section 5, Eq. 6, applied to the exact
 * FP8 keys rather than their PQ centroids):
 *   f_t = sum_g w[r, g] * max(0, q_g . k_t),  k_t = scale_t * e4m3(k8_t). */
static int fine_scores(const uint16_t *q, const orc_cache *c, const int32_t *pt_row,
                       const orc_params *prm, int r, int h, int64_t nblocks, const int64_t *blocks,
                       double *f, int64_t *tok)
{
    const int b = c->block_size, dk = c->dk;
    const int G = prm->num_q_heads / c->num_kv_heads;
    int64_t n = 0;
    for (int64_t u = 0; u < nblocks; ++u) {
        int64_t j = blocks[u];
        int64_t p = pt_row[j];
        if (p < 0 || p >= c->num_pages)
            return ORC_BAD_PAGE;
        for (int t = 0; t < b; ++t) {
            int64_t base = ((int64_t)p * c->num_kv_heads + h) * b + t;
            if (prm->fine_weights) {
                const double sc = (double)c->k8_scale[base];
                double f_t = 0.0;
                for (int g = 0; g < G; ++g) {
                    const uint16_t *qg = q + ((int64_t)r * prm->num_q_heads + h * G + g) * dk;
                    double d = 0.0;
                    for (int i = 0; i < dk; ++i)
                        d += orc_bf16_to_f64(qg[i]) * (sc * orc_e4m3_to_f64(c->k8[base * dk + i]));
                    const double w = (double)prm->fine_weights[(int64_t)r * prm->num_q_heads + h * G + g];
                    f_t += w * (d > 0.0 ? d : 0.0);
                }
                f[n] = f_t;
                tok[n] = j * b + t;
                ++n;
                continue;
            }
            double s = 0.0;
            for (int g = 0; g < G; ++g) {
                const uint16_t *qg = q + ((int64_t)r * prm->num_q_heads + h * G + g) * dk;
                for (int i = 0; i < dk; ++i)
                    s += orc_bf16_to_f64(qg[i]) * orc_e4m3_to_f64(c->k8[base * dk + i]);
            }
            f[n] = (double)c->k8_scale[base] * s;
            tok[n] = j * b + t;
            ++n;
        }
    }
    return ORC_OK;
}

int orc_fine_scores(const uint16_t *q, const orc_cache *idx, const int32_t *pt,
                    const orc_params *prm, int r, int h, int64_t nblocks, const int64_t *blocks,
                    double *f, int64_t *tok)
{
    return fine_scores(q, idx, pt + (int64_t)r * prm->max_blocks, prm, r, h, nblocks, blocks, f, tok);
}

/* ------------------------------------------------------------------ */
/* Step: PQ32 coarse scores and the miss filter                        */
/* ------------------------------------------------------------------ */

/* PQ32 (LeanSparse, Section 5, "Approximate scoring with PQ"): a 128-dim
 * index key is split into 32 four-dim subvectors, each stored as a one-byte
 * index c_j into a codebook C_j of 256 centroids.  The coarse score of
 * token t (Eq. 6) substitutes the centroids for the subvectors inside the
 * indexer's weighted head aggregation:
 *   s~_t = sum_g w_g * max(0, sum_j q_{g,j} . C_j[c_{t,j}])
 * over the query heads g of the KV head's group (q_{g,j}: dims 4j .. 4j+3
 * of head g's query). */
static double pq_score(const uint16_t *q, const float *w, const uint8_t *codes, const uint16_t *codebook,
                       int G, int dk)
{
    double s = 0.0;
    for (int g = 0; g < G; ++g) {
        const uint16_t *qg = q + (int64_t)g * dk;
        double d = 0.0;
        for (int j = 0; j < dk / 4; ++j) {
            const uint16_t *cj = codebook + ((int64_t)j * 256 + codes[j]) * 4;
            for (int e = 0; e < 4; ++e)
                d += orc_bf16_to_f64(qg[4 * j + e]) * orc_bf16_to_f64(cj[e]);
        }
        s += (double)w[g] * (d > 0.0 ? d : 0.0);
    }
    return s;
}

/* s~ of the tokens [t0, t0 + n) of request r, KV head h (full blocks). */
int orc_pq_scores(const uint16_t *q, const orc_cache *c, const int32_t *pt, const orc_params *prm,
                  int r, int h, int64_t t0, int64_t n, double *out)
{
    const int b = c->block_size, dk = c->dk, G = prm->num_q_heads / c->num_kv_heads;
    if (dk != 128 || !prm->pq_codes || !prm->pq_codebook || !prm->fine_weights)
        return ORC_BAD_ARG;
    const uint16_t *qr = q + ((int64_t)r * prm->num_q_heads + h * G) * dk;
    const float *wr = prm->fine_weights + (int64_t)r * prm->num_q_heads + h * G;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t t = t0 + i;
        const int64_t p = pt[(int64_t)r * prm->max_blocks + t / b];
        if (p < 0 || p >= c->num_pages)
            return ORC_BAD_PAGE;
        const uint8_t *codes = prm->pq_codes + (((int64_t)p * c->num_kv_heads + h) * b + t % b) * 32;
        out[i] = pq_score(qr, wr, codes, prm->pq_codebook, G, dk);
    }
    return ORC_OK;
}

/* PQ32 encoding of index keys: per subvector, the nearest centroid by
 * squared Euclidean distance to the dequantised key scale_t * e4m3(k8_t),
 * ties to the lower centroid.  The distance decides an integer, so it is
 * evaluated in fp32 in a fixed order: k = scale * e4m3 (one rounding),
 * diff_e = k_e - C_e, dist = ((diff_0^2 + diff_1^2) + diff_2^2) + diff_3^2,
 * each operation rounded to fp32 (no fused multiply-add).  tokens: n
 * positions (page p, slot t) pairs flattened as p * b + t. */
int orc_pq_encode(const orc_cache *c, const uint16_t *codebook, int64_t n, const int64_t *slots, uint8_t *codes)
{
    if (c->dk != 128 || !c->k8 || !c->k8_scale || c->num_kv_heads != 1)
        return ORC_BAD_ARG;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t base = slots[i];   /* (p * Hkv + h) * b + t with Hkv = 1 */
        const float sc = c->k8_scale[base];
        for (int j = 0; j < 32; ++j) {
            volatile float kk[4];
            for (int e = 0; e < 4; ++e)
                kk[e] = sc * (float)orc_e4m3_to_f64(c->k8[base * 128 + 4 * j + e]);
            int best = 0;
            float bd = INFINITY;
            for (int cc = 0; cc < 256; ++cc) {
                const uint16_t *cj = codebook + ((int64_t)j * 256 + cc) * 4;
                volatile float d0 = kk[0] - (float)orc_bf16_to_f64(cj[0]);
                volatile float d1 = kk[1] - (float)orc_bf16_to_f64(cj[1]);
                volatile float d2 = kk[2] - (float)orc_bf16_to_f64(cj[2]);
                volatile float d3 = kk[3] - (float)orc_bf16_to_f64(cj[3]);
                volatile float s0 = d0 * d0, s1 = d1 * d1, s2 = d2 * d2, s3 = d3 * d3;
                volatile float a = s0 + s1;
                volatile float b2 = a + s2;
                volatile float dist = b2 + s3;
                if (dist < bd) {
                    bd = dist;
                    best = cc;
                }
            }
            codes[i * 32 + j] = (uint8_t)best;
        }
    }
    return ORC_OK;
}

static int by_value_desc(const void *a, const void *b)
{
    const double x = *(const double *)a, y = *(const double *)b;
    return (x > y) ? -1 : (x < y);
}

/* The miss filter (LeanSparse, Section 5, "Retrieving and refining
 * candidates"): candidates whose original index key is cached (hits) are
 * kept; a miss is dropped when its coarse score is below the candidates'
 * k-th largest coarse score minus one sample standard deviation of the
 * candidates' coarse scores.  With at most k candidates every one is kept
 * (there is no k-th largest to compare with).  keep[i] = 1 / 0; returns
 * the number kept.  The threshold is written to *tau (-inf when every
 * candidate is kept). */
static int64_t miss_filter(const double *s, const uint8_t *hit, int64_t n, int64_t k, uint8_t *keep, double *tau)
{
    *tau = -INFINITY;
    if (n <= k) {
        for (int64_t i = 0; i < n; ++i)
            keep[i] = 1;
        return n;
    }
    double *srt = (double *)malloc(sizeof(double) * (size_t)n);
    if (!srt)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        srt[i] = s[i];
    qsort(srt, (size_t)n, sizeof(double), by_value_desc);   /* k-th largest */
    const double sk = srt[k - 1];
    free(srt);
    double mean = 0.0;
    for (int64_t i = 0; i < n; ++i)
        mean += s[i];
    mean /= (double)n;
    double var = 0.0;
    for (int64_t i = 0; i < n; ++i)
        var += (s[i] - mean) * (s[i] - mean);
    var /= (double)(n - 1);
    *tau = sk - sqrt(var);
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i) {
        keep[i] = (hit[i] || s[i] >= *tau) ? 1 : 0;
        m += keep[i];
    }
    return m;
}

int orc_miss_filter(const double *s, const uint8_t *hit, int64_t n, int64_t k, uint8_t *keep, double *tau)
{
    return miss_filter(s, hit, n, k, keep, tau) < 0 ? ORC_NOMEM : ORC_OK;
}

/* Exact weighted-ReLU index scores of explicit tokens of request r, KV
 * head h: f_t = sum_g w_g max(0, q_g . scale_t e4m3(k8_t)). */
static int token_scores_wrelu(const uint16_t *q, const orc_cache *c, const int32_t *pt_row, const orc_params *prm,
                              int r, int h, int64_t n, const int64_t *tok, double *f)
{
    const int b = c->block_size, dk = c->dk, G = prm->num_q_heads / c->num_kv_heads;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t t = tok[i];
        const int64_t p = pt_row[t / b];
        if (p < 0 || p >= c->num_pages)
            return ORC_BAD_PAGE;
        const int64_t base = ((int64_t)p * c->num_kv_heads + h) * b + t % b;
        const double sc = (double)c->k8_scale[base];
        double s = 0.0;
        for (int g = 0; g < G; ++g) {
            const uint16_t *qg = q + ((int64_t)r * prm->num_q_heads + h * G + g) * dk;
            double d = 0.0;
            for (int e = 0; e < dk; ++e)
                d += orc_bf16_to_f64(qg[e]) * (sc * orc_e4m3_to_f64(c->k8[base * dk + e]));
            s += (double)prm->fine_weights[(int64_t)r * prm->num_q_heads + h * G + g] * (d > 0.0 ? d : 0.0);
        }
        f[i] = s;
    }
    return ORC_OK;
}

int orc_token_scores_wrelu(const uint16_t *q, const orc_cache *c, const int32_t *pt, const orc_params *prm,
                           int r, int h, int64_t n, const int64_t *tok, double *f)
{
    if (!prm->fine_weights || !c->k8 || !c->k8_scale)
        return ORC_BAD_ARG;
    return token_scores_wrelu(q, c, pt + (int64_t)r * prm->max_blocks, prm, r, h, n, tok, f);
}

/* The PQ coarse-to-fine selection of one (request, KV head), in the order
 * of LeanSparse Section 5 and Figure 9:
 *   1. coarse: s~_t for every token of the full candidate blocks (the
 *      encoded history), top-C tokens (pq_candidates) by s~;
 *   2. miss filter over the C candidates (hits kept, misses below the
 *      k-th largest s~ minus one sample standard deviation dropped);
 *   3. fine: exact weighted-ReLU scores of the kept candidates and of the
 *      tokens of the partial last block (the unencoded tail, always scored
 *      from its original keys), top-k (c2f_tokens) by f.
 * chosen: the k tokens, ascending, -1 padded; cand (may be NULL): the C
 * coarse candidates ascending, -1 padded; kept (may be NULL): 1 / 0 per
 * cand entry.  Returns the number chosen through *nchosen. */
static int pq_select(const uint16_t *q, const orc_cache *ic, const int32_t *pt, int64_t L, const orc_params *prm,
                     int r, int h, int64_t *chosen, int64_t *nchosen, int32_t *cand, uint8_t *kept_out, double *tau_out)
{
    const int b = ic->block_size;
    const int32_t *pt_row = pt + (int64_t)r * prm->max_blocks;
    int64_t se, rs;
    forced_ranges(L, prm->sink, prm->recent, &se, &rs);
    const int64_t nfull = L / b;
    const int64_t C = prm->pq_candidates, k = prm->c2f_tokens;
    /* 1. coarse over the encoded history */
    int64_t ntok = 0;
    for (int64_t j = 0; j < nfull; ++j)
        if (is_candidate(j, b, se, rs))
            ntok += b;
    int64_t cap = ntok + b + 1;
    double *s = (double *)malloc(sizeof(double) * (size_t)cap);
    int64_t *ids = (int64_t *)malloc(sizeof(int64_t) * (size_t)cap);
    int64_t *cb = (int64_t *)malloc(sizeof(int64_t) * (size_t)(C > 0 ? C : 1));
    double *cs = (double *)malloc(sizeof(double) * (size_t)(C > 0 ? C : 1));
    uint8_t *hit = (uint8_t *)malloc((size_t)(C > 0 ? C : 1));
    uint8_t *keep = (uint8_t *)malloc((size_t)(C > 0 ? C : 1));
    int64_t *ft = (int64_t *)malloc(sizeof(int64_t) * (size_t)(C + b + 1));
    double *f = (double *)malloc(sizeof(double) * (size_t)(C + b + 1));
    int rc = ORC_OK;
    if (!s || !ids || !cb || !cs || !hit || !keep || !ft || !f) {
        rc = ORC_NOMEM;
        goto out;
    }
    {
        int64_t n = 0;
        for (int64_t j = 0; j < nfull && rc == ORC_OK; ++j) {
            if (!is_candidate(j, b, se, rs))
                continue;
            rc = orc_pq_scores(q, ic, pt, prm, r, h, j * b, b, s + n);
            for (int t = 0; t < b; ++t)
                ids[n + t] = j * b + t;
            n += b;
        }
        if (rc)
            goto out;
        const int64_t ncb = select_topk(s, ids, n, C, cb);
        if (cand)
            for (int64_t i = 0; i < C; ++i)
                cand[i] = (int32_t)cb[i];
        /* coarse scores and hits of the candidates */
        for (int64_t i = 0; i < ncb; ++i) {
            const int64_t t = cb[i];
            int64_t lo = 0, hi = n - 1;   /* ids ascend: binary search */
            while (lo < hi) {
                const int64_t mid = (lo + hi) / 2;
                if (ids[mid] < t)
                    lo = mid + 1;
                else
                    hi = mid;
            }
            cs[i] = s[lo];
            const int64_t p = pt_row[t / b];
            hit[i] = prm->pq_hit ? prm->pq_hit[((int64_t)p * ic->num_kv_heads + h) * b + t % b] : 1;
        }
        /* 2. miss filter */
        double tau;
        if (miss_filter(cs, hit, ncb, k, keep, &tau) < 0) {
            rc = ORC_NOMEM;
            goto out;
        }
        if (tau_out)
            *tau_out = tau;
        if (kept_out)
            for (int64_t i = 0; i < C; ++i)
                kept_out[i] = i < ncb ? keep[i] : 0;
        /* 3. fine over the kept candidates and the tail */
        int64_t m = 0;
        for (int64_t i = 0; i < ncb; ++i)
            if (keep[i])
                ft[m++] = cb[i];
        for (int64_t t = nfull * b; t < L; ++t)
            if (t >= se && t < rs)
                ft[m++] = t;
        rc = token_scores_wrelu(q, ic, pt_row, prm, r, h, m, ft, f);
        if (rc)
            goto out;
        *nchosen = select_topk(f, ft, m, k, chosen);
    }
out:
    free(s);
    free(ids);
    free(cb);
    free(cs);
    free(hit);
    free(keep);
    free(ft);
    free(f);
    return rc;
}

int orc_pq_select(const uint16_t *q, const orc_cache *ic, const int32_t *pt, const int32_t *lens,
                  const orc_params *prm, int r, int h, int32_t *chosen, int32_t *cand, uint8_t *kept, double *tau)
{
    if (prm->pq_candidates <= 0 || !prm->fine_weights)
        return ORC_BAD_ARG;
    int64_t *ch = (int64_t *)malloc(sizeof(int64_t) * (size_t)(prm->c2f_tokens > 0 ? prm->c2f_tokens : 1));
    if (!ch)
        return ORC_NOMEM;
    int64_t nch = 0;
    int rc = pq_select(q, ic, pt, lens[r], prm, r, h, ch, &nch, cand, kept, tau);
    for (int64_t i = 0; i < prm->c2f_tokens; ++i)
        chosen[i] = (int32_t)ch[i];
    free(ch);
    return rc;
}

/* ------------------------------------------------------------------ */
/* The decode step                                                     */
/* ------------------------------------------------------------------ */

/* One (request, KV head) unit: forced ranges, candidates, scores,
 * selection, token set, attention. */
static int decode_unit(const uint16_t *q, const orc_cache *c, const uint16_t *summ,
                       const orc_cache *ic, const uint16_t *isumm, const int32_t *pt,
                       const int32_t *lens, const orc_params *prm, int r, int h,
                       uint16_t *out, double *lse, int32_t *sel, int32_t *cand)
{
    const int b = c->block_size;
    const int64_t L = lens[r];
    const int32_t *pt_row = pt + (int64_t)r * prm->max_blocks;
    const int c2f = prm->c2f_candidates > 0 || prm->pq_candidates > 0;
    const int64_t ksel = c2f ? prm->c2f_tokens : prm->k_blocks;
    int64_t se, rs;
    forced_ranges(L, prm->sink, prm->recent, &se, &rs);

    double *scores = (double *)malloc(sizeof(double) * (size_t)(prm->max_blocks > 0 ? prm->max_blocks : 1));
    int64_t *chosen = (int64_t *)malloc(sizeof(int64_t) * (size_t)(ksel > 0 ? ksel : 1));
    int64_t cap = se + (L - rs) + (c2f ? prm->c2f_tokens : (int64_t)prm->k_blocks * b);
    int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
    int rc = ORC_OK;
    if (!scores || !chosen || !tok) {
        rc = ORC_NOMEM;
        goto done;
    }

    int64_t nchosen = 0;
    if (prm->pq_candidates > 0) {
        rc = pq_select(q, ic, pt, L, prm, r, h, chosen, &nchosen,
                       cand ? cand + ((int64_t)r * c->num_kv_heads + h) * prm->pq_candidates : NULL, NULL, NULL);
        if (rc)
            goto done;
    } else if (!c2f) {
        rc = row_scores(q, c, 0, summ, pt, L, prm, r, h, scores);
        if (rc)
            goto done;
        nchosen = select_topk(scores, NULL, prm->max_blocks, ksel, chosen);
    } else {
        /* coarse: top-C blocks over summaries of the dequantised index keys */
        int64_t C = prm->c2f_candidates;
        int64_t *cb = (int64_t *)malloc(sizeof(int64_t) * (size_t)C);
        if (!cb) {
            rc = ORC_NOMEM;
            goto done;
        }
        rc = row_scores(q, ic, 1, isumm, pt, L, prm, r, h, scores);
        if (rc) {
            free(cb);
            goto done;
        }
        int64_t ncb = select_topk(scores, NULL, prm->max_blocks, C, cb);
        if (cand)
            for (int64_t i = 0; i < C; ++i)
                cand[((int64_t)r * c->num_kv_heads + h) * C + i] = (int32_t)cb[i];
        /* fine: exact FP8 rescoring of every token of the C blocks */
        double *f = (double *)malloc(sizeof(double) * (size_t)(ncb * b > 0 ? ncb * b : 1));
        int64_t *ft = (int64_t *)malloc(sizeof(int64_t) * (size_t)(ncb * b > 0 ? ncb * b : 1));
        if (!f || !ft) {
            free(cb);
            free(f);
            free(ft);
            rc = ORC_NOMEM;
            goto done;
        }
        rc = fine_scores(q, ic, pt_row, prm, r, h, ncb, cb, f, ft);
        if (rc == ORC_OK)
            nchosen = select_topk(f, ft, ncb * b, ksel, chosen);
        free(cb);
        free(f);
        free(ft);
        if (rc)
            goto done;
    }
    if (sel)
        for (int64_t i = 0; i < ksel; ++i)
            sel[((int64_t)r * c->num_kv_heads + h) * ksel + i] = (int32_t)chosen[i];

    /* token set T = F U selected, ascending */
    int64_t ntok = 0;
    for (int64_t t = 0; t < se; ++t)
        tok[ntok++] = t;
    for (int64_t i = 0; i < nchosen; ++i) {
        if (c2f) {
            tok[ntok++] = chosen[i];
        } else {
            for (int t = 0; t < b; ++t)
                tok[ntok++] = chosen[i] * b + t;
        }
    }
    for (int64_t t = rs; t < L; ++t)
        tok[ntok++] = t;

    rc = attend_group(q, c, pt_row, prm, r, h, ntok, tok, out, lse);
done:
    free(scores);
    free(chosen);
    free(tok);
    return rc;
}

/* The whole decode step for every (request, KV head).
 *   out  [B, Hq, dv] bf16 bits;  lse [B, Hq] double (natural log)
 *   sel  [B, Hkv, ksel]: selected block indices (single stage, ksel =
 *        k_blocks) or token positions (coarse-to-fine, ksel = c2f_tokens),
 *        ascending, -1 padded.  May be NULL.
 *   cand [B, Hkv, c2f_candidates] coarse blocks (coarse-to-fine only, may be NULL)
 *   summ / isumm: precomputed summaries (bf16 bits, [P, Hkv, dk]) of the
 *        attention keys / index keys, or NULL to compute them from the keys.
 * nthreads > 1 runs units in parallel when built with OpenMP. */
int orc_decode(const uint16_t *q, const orc_cache *c, const uint16_t *summ,
               const orc_cache *ic, const uint16_t *isumm, const int32_t *pt,
               const int32_t *lens, const orc_params *prm, int nthreads,
               uint16_t *out, double *lse, int32_t *sel, int32_t *cand)
{
    if (prm->num_q_heads % c->num_kv_heads != 0)
        return ORC_BAD_ARG;
    if ((prm->c2f_candidates > 0 || prm->pq_candidates > 0) && (!ic || !ic->k8 || !ic->k8_scale))
        return ORC_BAD_ARG;
    if (prm->pq_candidates > 0 && (!prm->pq_codes || !prm->pq_codebook || !prm->fine_weights))
        return ORC_BAD_ARG;
    const int64_t units = (int64_t)prm->batch * c->num_kv_heads;
    int rc = ORC_OK;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int r = (int)(u / c->num_kv_heads), h = (int)(u % c->num_kv_heads);
        int e = decode_unit(q, c, summ, ic, isumm, pt, lens, prm, r, h, out, lse, sel, cand);
        if (e) {
#ifdef _OPENMP
#pragma omp critical
#endif
            rc = e;
        }
    }
    return rc;
}

/* Dense attention over [0, L) for every query head (tests only). */
int orc_dense(const uint16_t *q, const orc_cache *c, const int32_t *pt, const int32_t *lens,
              const orc_params *prm, uint16_t *out, double *lse)
{
    for (int r = 0; r < prm->batch; ++r) {
        int64_t L = lens[r];
        int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(L > 0 ? L : 1));
        if (!tok)
            return ORC_NOMEM;
        for (int64_t t = 0; t < L; ++t)
            tok[t] = t;
        for (int h = 0; h < c->num_kv_heads; ++h) {
            int rc = attend_group(q, c, pt + (int64_t)r * prm->max_blocks, prm, r, h, L, tok, out, lse);
            if (rc) {
                free(tok);
                return rc;
            }
        }
        free(tok);
    }
    return ORC_OK;
}

/* Attention of one query head (fp64 query) over an explicit token list of
 * request r, KV head h; o: [dv] doubles. */
int orc_attend_tokens(const double *qd, const orc_cache *c, const int32_t *pt_row, int64_t ntok,
                      const int64_t *tok, int h, double scale, double *o, double *lse)
{
    return attend(qd, c, pt_row, ntok, tok, h, scale, o, lse);
}

/* Log-sum-exp merge of partial results over a partition of the token set:
 * part s has normalised output o_s and log-sum-exp lse_s; the union has
 * weights exp(lse_s - M) with M the largest lse_s.  Empty parts (lse = -inf)
 * contribute nothing; all parts empty gives o = 0, lse = -inf. */
void orc_lse_merge(int nparts, int dv, const double *o, const double *lse,
                   double *o_out, double *lse_out)
{
    double M = -INFINITY;
    for (int s = 0; s < nparts; ++s)
        if (lse[s] > M)
            M = lse[s];
    for (int i = 0; i < dv; ++i)
        o_out[i] = 0.0;
    if (M == -INFINITY) {
        *lse_out = -INFINITY;
        return;
    }
    double wsum = 0.0;
    for (int s = 0; s < nparts; ++s) {
        if (lse[s] == -INFINITY)
            continue;
        double w = exp(lse[s] - M);
        wsum += w;
        for (int i = 0; i < dv; ++i)
            o_out[i] += w * o[(int64_t)s * dv + i];
    }
    for (int i = 0; i < dv; ++i)
        o_out[i] /= wsum;
    *lse_out = M + log(wsum);
}

/* Attention over T = F U (given selection) for every (request, KV head):
 * the definition behind a sparse decode call that receives its selection
 * (block indices, or token positions when token_mode != 0; ascending, -1
 * padded, nsel per row).  Blocks that are not candidates, tokens inside the
 * forced ranges, and entries that do not ascend are skipped. */
int orc_attend_selection(const uint16_t *q, const orc_cache *c, const int32_t *pt, const int32_t *lens,
                         const orc_params *prm, const int32_t *sel, int32_t nsel, int token_mode,
                         uint16_t *out, double *lse)
{
    const int b = c->block_size;
    for (int r = 0; r < prm->batch; ++r) {
        const int64_t L = lens[r];
        int64_t se, rs;
        forced_ranges(L, prm->sink, prm->recent, &se, &rs);
        const int32_t *pt_row = pt + (int64_t)r * prm->max_blocks;
        int64_t cap = se + (L - rs) + (int64_t)nsel * (token_mode ? 1 : b);
        int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
        if (!tok)
            return ORC_NOMEM;
        for (int h = 0; h < c->num_kv_heads; ++h) {
            const int32_t *srow = sel + ((int64_t)r * c->num_kv_heads + h) * nsel;
            int64_t ntok = 0, prev = -1;
            for (int64_t t = 0; t < se; ++t)
                tok[ntok++] = t;
            for (int i = 0; i < nsel; ++i) {
                int64_t e = srow[i];
                if (e < 0 || e <= prev)
                    continue;
                /* a selected block must be a candidate; a selected token
                 * need only lie outside the forced ranges (the PQ32
                 * selection rescores the unencoded tail and may keep it) */
                if (token_mode ? !(e >= se && e < rs) : !is_candidate(e, b, se, rs))
                    continue;
                prev = e;
                if (token_mode)
                    tok[ntok++] = e;
                else
                    for (int t = 0; t < b; ++t)
                        tok[ntok++] = e * b + t;
            }
            for (int64_t t = rs; t < L; ++t)
                tok[ntok++] = t;
            int rc = attend_group(q, c, pt_row, prm, r, h, ntok, tok, out, lse);
            if (rc) {
                free(tok);
                return rc;
            }
        }
        free(tok);
    }
    return ORC_OK;
}

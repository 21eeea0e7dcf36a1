/*
 * CPU oracle for query-aware sparse paged decode -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision statement of what the decode path computes.
 * Only the test suite, the package's smoke check and the benchmark's CPU
 * baseline leg load this file's library; the product path never does, and it
 * shares no code, header or table with the CUDA library.
 *
 * Sources (web pages on the method):
 *   [TS]  TinyServe query-aware page selection article:
 *         s1 "paged KV cache, 16 tokens per page", s2.1 "metadata structure"
 *         (per-page element-wise min m_j and max M_j of the keys),
 *         s2.2 "relevance score" (score_j = sum_i q[i] * (q[i] > 0 ? M_j[i] : m_j[i])),
 *         s2.3 "four stages" (score all pages, top-K pages, load only those,
 *         attention over them).
 *   [PA]  CS336 Lecture 10 "Inference", s9.2 PagedAttention (block table maps
 *         logical blocks to physical blocks; shared prefixes map to the same
 *         physical blocks) and s2.3 (decode attention softmax(q K^T / sqrt(d)) V).
 *   [QU]  Quail AI-SQL engine article, section "the inference engine as an
 *         execution engine" (partial attention results combined by
 *         log-sum-exp rescaling, as in flash decoding).
 *   [VXR] Vortex digest, method overview item 3: a lossy radix Top-K that
 *         stops once enough high-confidence candidates are collected and
 *         draws the rest at random from the threshold bin (recall@k > 0.97).
 *   [SM]  SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 *         number generators", OOPSLA 2014): state_i = seed + i * gamma,
 *         output_i = mix(state_i), used as a counter-based generator.
 *   [VX]  Vortex sparse-attention digest, method overview item 1: a
 *         query-independent cache phase computes per-block summaries such as
 *         the block's mean key ("centroids"); the query-dependent indexer
 *         phase scores each block from q and its summary, keeps the top-K
 *         blocks and attends over them ("Block Top-K").
 *
 * Readings taken where the pages are silent (listed with the design notes):
 *   - the comparator lost in the extracted formula is "q[i] > 0";
 *   - with grouped-query attention one selection serves the G query heads of a
 *     KV head; its page score is the maximum of the G heads' bounds;
 *   - ties in the top-K go to the lower logical page index; the selected list
 *     is returned in ascending page order, padded with -1;
 *   - only tokens t < seq_len count, in metadata and in attention;
 *   - Block Top-K: a page's centroid is the mean of its valid keys, its
 *     score for one query head is q . centroid, and with grouped-query
 *     attention the page score is the maximum over the group's heads (the
 *     same aggregation as for the bound);
 *   - an empty softmax (no token) gives output 0 and lse -inf.
 *
 * Element types: KV pools are read raw, as IEEE fp32 or as bfloat16 (the top
 * 16 bits of an fp32), and widened exactly to double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1 };

/* Thread count for the row loops (n <= 0 keeps the current one); returns it. */
int orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

static double load_elem(const void *base, int dtype, int64_t i) {
    if (dtype == ORC_F32) return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Index of element (page p, kv head g, token t, dim i) in a [Npool][Hkv][P][d] pool. */
static int64_t pool_index(int64_t p, int hkv, int g, int page_size, int t, int d, int i) {
    return (((p * hkv + g) * page_size + t) * (int64_t)d) + i;
}

/*
 * [TS s2.1] Metadata of the listed physical pages: for every KV head g and
 * dimension i, m[i] = min over the page's valid tokens of K[t][i] and
 * M[i] = the max over the same tokens.  meta is [n_pool][hkv][2][d] (the min
 * row, then the max row); pages not listed are left untouched.
 * Returns 0, or -1 if a page id or a valid-token count is out of range.
 */
int orc_meta(const void *k_pool, int kv_dtype, int64_t n_pool, int hkv, int page_size, int d,
             const int32_t *page_ids, const int32_t *valid_tokens, int64_t n_list, double *meta) {
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t e = 0; e < n_list; e++) {
        int64_t p = page_ids[e];
        int valid = valid_tokens[e];
        if (p < 0 || p >= n_pool || valid < 1 || valid > page_size) {
            bad = 1;
            continue;
        }
        for (int g = 0; g < hkv; g++) {
            double *mn = meta + ((p * hkv + g) * 2) * (int64_t)d;
            double *mx = mn + d;
            for (int i = 0; i < d; i++) {
                double lo = load_elem(k_pool, kv_dtype, pool_index(p, hkv, g, page_size, 0, d, i));
                double hi = lo;
                for (int t = 1; t < valid; t++) {
                    double x = load_elem(k_pool, kv_dtype, pool_index(p, hkv, g, page_size, t, d, i));
                    if (x < lo) lo = x;
                    if (x > hi) hi = x;
                }
                mn[i] = lo;
                mx[i] = hi;
            }
        }
    }
    return bad ? -1 : 0;
}

/* [TS s2.2] Upper-bound relevance of one page for one query vector. */
double orc_bound(const double *q, const double *m, const double *M, int d) {
    double s = 0.0;
    for (int i = 0; i < d; i++) s += q[i] * (q[i] > 0.0 ? M[i] : m[i]);
    return s;
}

/*
 * [TS s2.2-2.3] Scores of logical pages 0..n_b-1 of one sequence for KV head g:
 * S(j) = max over the G query heads h of the group of bound(q_h, m_p, M_p),
 * p = table_row[j].  q_group is [G][d].  Returns 0, or -1 on a bad page id
 * (that page's score is then -inf).
 */
int orc_row_scores(const double *q_group, int G, const double *meta, int64_t n_pool, int hkv,
                   int g, int d, const int32_t *table_row, int n_b, double *scores) {
    int rc = 0;
    for (int j = 0; j < n_b; j++) {
        int64_t p = table_row[j];
        if (p < 0 || p >= n_pool) {
            scores[j] = -INFINITY;
            rc = -1;
            continue;
        }
        const double *mn = meta + ((p * hkv + g) * 2) * (int64_t)d;
        const double *mx = mn + d;
        double best = -INFINITY;
        for (int h = 0; h < G; h++) {
            double s = orc_bound(q_group + (int64_t)h * d, mn, mx, d);
            if (s > best) best = s;
        }
        scores[j] = best;
    }
    return rc;
}

/*
 * [VX item 1] Block summaries of the listed physical pages: for every KV head
 * g, c[i] = (1 / valid) * sum over the page's valid tokens t of K[t][i].
 * cent is [n_pool][hkv][d]; pages not listed are left untouched.
 * Returns 0, or -1 if a page id or a valid-token count is out of range.
 */
int orc_centroid(const void *k_pool, int kv_dtype, int64_t n_pool, int hkv, int page_size, int d,
                 const int32_t *page_ids, const int32_t *valid_tokens, int64_t n_list, double *cent) {
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t e = 0; e < n_list; e++) {
        int64_t p = page_ids[e];
        int valid = valid_tokens[e];
        if (p < 0 || p >= n_pool || valid < 1 || valid > page_size) {
            bad = 1;
            continue;
        }
        for (int g = 0; g < hkv; g++) {
            double *c = cent + (p * hkv + g) * (int64_t)d;
            for (int i = 0; i < d; i++) {
                double sum = 0.0;
                for (int t = 0; t < valid; t++)
                    sum += load_elem(k_pool, kv_dtype, pool_index(p, hkv, g, page_size, t, d, i));
                c[i] = sum / valid;
            }
        }
    }
    return bad ? -1 : 0;
}

/*
 * [VX item 1] Block Top-K scores of logical pages 0..n_b-1 of one sequence
 * for KV head g: S(j) = max over the G query heads h of q_h . c_p,
 * p = table_row[j].  Returns 0, or -1 on a bad page id (score -inf).
 */
int orc_centroid_scores(const double *q_group, int G, const double *cent, int64_t n_pool, int hkv, int g, int d,
                        const int32_t *table_row, int n_b, double *scores) {
    int rc = 0;
    for (int j = 0; j < n_b; j++) {
        int64_t p = table_row[j];
        if (p < 0 || p >= n_pool) {
            scores[j] = -INFINITY;
            rc = -1;
            continue;
        }
        const double *c = cent + (p * hkv + g) * (int64_t)d;
        double best = -INFINITY;
        for (int h = 0; h < G; h++) {
            double s = 0.0;
            for (int i = 0; i < d; i++) s += q_group[(int64_t)h * d + i] * c[i];
            if (s > best) best = s;
        }
        scores[j] = best;
    }
    return rc;
}

typedef struct {
    double score;
    int32_t index;
} ranked_page;

/* Higher score first; among equal scores the lower page index first. */
static int by_score_desc(const void *a, const void *b) {
    const ranked_page *x = (const ranked_page *)a, *y = (const ranked_page *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->index > y->index) - (x->index < y->index);
}

static int by_int_asc(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * [TS s2.3] Top-K pages of one row: the top_k largest scores (all n_b pages if
 * top_k >= n_b), returned as ascending logical page indices in selected[0..top_k),
 * padded with -1.  Returns the number selected.
 */
int orc_select(const double *scores, int n_b, int top_k, int32_t *selected) {
    int n_sel = top_k < n_b ? top_k : n_b;
    if (n_sel < 0) n_sel = 0;
    if (top_k >= n_b) {
        for (int j = 0; j < n_b; j++) selected[j] = j;
    } else {
        ranked_page *r = (ranked_page *)malloc(sizeof(ranked_page) * (size_t)(n_b > 0 ? n_b : 1));
        for (int j = 0; j < n_b; j++) {
            r[j].score = scores[j];
            r[j].index = j;
        }
        qsort(r, (size_t)n_b, sizeof(ranked_page), by_score_desc);
        for (int k = 0; k < n_sel; k++) selected[k] = r[k].index;
        free(r);
        qsort(selected, (size_t)n_sel, sizeof(int32_t), by_int_asc);
    }
    for (int k = n_sel; k < top_k; k++) selected[k] = -1;
    return n_sel;
}

/*
 * [PA s2.3, s9.2; TS s2.3] Attention of the G query heads of KV head g of one
 * sequence over the tokens of the listed logical pages (pages[0..n_list)), each
 * mapped through table_row to a physical page; only tokens at positions
 * < seq_len count.  For head h:  l_t = sm_scale * (q_h . k_t),
 * out_h = sum_t softmax(l)_t v_t,  lse_h = log sum_t exp(l_t).
 * q_group is [G][d]; out is [G][d]; lse is [G] (may be NULL).
 * Returns the number of tokens attended, or -1 on a bad page id or index
 * (such a page is skipped).
 */
int orc_attend_row(const double *q_group, int G, const void *k_pool, const void *v_pool, int kv_dtype,
                   int64_t n_pool, int hkv, int g, int page_size, int d, const int32_t *table_row,
                   int n_b, int seq_len, const int32_t *pages, int n_list, double sm_scale,
                   double *out, double *lse) {
    int rc = 0;
    /* collect (physical page, token) pairs in the listed order */
    int cap = n_list * page_size;
    int64_t *tok_base = (int64_t *)malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
    int n_tok = 0;
    for (int e = 0; e < n_list; e++) {
        int j = pages[e];
        if (j < 0 || j >= n_b) {
            rc = -1;
            continue;
        }
        int64_t p = table_row[j];
        if (p < 0 || p >= n_pool) {
            rc = -1;
            continue;
        }
        for (int t = 0; t < page_size; t++) {
            if ((int64_t)j * page_size + t >= seq_len) break;
            tok_base[n_tok++] = pool_index(p, hkv, g, page_size, t, d, 0);
        }
    }
    double *logit = (double *)malloc(sizeof(double) * (size_t)(n_tok > 0 ? n_tok : 1));
    for (int h = 0; h < G; h++) {
        const double *q = q_group + (int64_t)h * d;
        double *o = out + (int64_t)h * d;
        for (int i = 0; i < d; i++) o[i] = 0.0;
        if (n_tok == 0) {
            if (lse) lse[h] = -INFINITY;
            continue;
        }
        double mx = -INFINITY;
        for (int t = 0; t < n_tok; t++) {
            double dot = 0.0;
            for (int i = 0; i < d; i++) dot += q[i] * load_elem(k_pool, kv_dtype, tok_base[t] + i);
            logit[t] = sm_scale * dot;
            if (logit[t] > mx) mx = logit[t];
        }
        double sum = 0.0;
        for (int t = 0; t < n_tok; t++) {
            logit[t] = exp(logit[t] - mx); /* now the unnormalised weight */
            sum += logit[t];
        }
        for (int t = 0; t < n_tok; t++) {
            double w = logit[t] / sum;
            for (int i = 0; i < d; i++) o[i] += w * load_elem(v_pool, kv_dtype, tok_base[t] + i);
        }
        if (lse) lse[h] = mx + log(sum);
    }
    free(logit);
    free(tok_base);
    return rc < 0 ? -1 : n_tok;
}

/* [SM] Output i (i >= 1) of SplitMix64 started at `seed`. */
uint64_t orc_splitmix64(uint64_t seed, uint64_t i) {
    uint64_t z = seed + i * 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

/* fp32 score -> unsigned key with the same order (-0 and +0 share a key). */
static uint32_t key_of(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

/*
 * [VXR] Approximate top-K of one row of fp32 scores (the reading taken for
 * the digest's lossy radix Top-K):
 *   1. scores become order-preserving 32-bit keys;
 *   2. MSB-first radix passes over the four 8-bit digits of the key (bits
 *      31..24, then 23..16, 15..8, 7..0): each pass counts the keys of the
 *      current bucket per digit and moves into the digit bucket that holds
 *      the `need`-th largest key; keys in higher digit buckets are certain
 *      to be in the top-K and leave `need`;
 *   3. early exit: before a pass, if need <= need_max (= floor(eps * K)),
 *      stop; also stop when the bucket is taken whole or fully resolved;
 *   4. the keys above the final bucket are all kept; `need` keys of the
 *      bucket (m keys, ranked t = 0..m-1 in page order) are kept: exactly
 *      those t with floor(((t + 1) need + o) / m) - floor((t need + o) / m) = 1,
 *      o = splitmix64(seed, row + 1) mod m (systematic sampling with a random
 *      start: every key of the bucket is kept with probability need / m).
 *      need_max = 0 gives the exact rule instead: the first `need` in page
 *      order (ties -> lower index).
 * selected gets the kept indices ascending, -1 padded to top_k; returns the
 * count min(top_k, n).
 */
int orc_select_approx(const float *scores, int n, int top_k, int need_max, uint64_t seed, int64_t row,
                      int32_t *selected) {
    if (top_k >= n) {
        for (int i = 0; i < top_k; i++) selected[i] = i < n ? i : -1;
        return n;
    }
    uint32_t *key = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(n > 0 ? n : 1));
    for (int i = 0; i < n; i++) key[i] = key_of(scores[i]);
    /* the bucket is the keys whose bits >= hi equal those of `prefix` */
    int hi = 32;
    uint64_t prefix = 0;
    int need = top_k, lo = hi;
    while (hi > 0) {
        if (need_max > 0 && need <= need_max) break;
        lo = hi > 8 ? hi - 8 : 0;
        uint64_t count[256] = {0};
        for (int i = 0; i < n; i++)
            if (((uint64_t)key[i] >> hi) == (prefix >> hi)) count[(key[i] >> lo) & ((1u << (hi - lo)) - 1u)]++;
        uint64_t above = 0;
        int bin = -1;
        for (int d = (1 << (hi - lo)) - 1; d >= 0; d--) {
            if (above + count[d] >= (uint64_t)need) {
                bin = d;
                break;
            }
            above += count[d];
        }
        prefix |= (uint64_t)bin << lo;
        need -= (int)above;
        if ((int)count[bin] == need) break;
        hi = lo;
    }
    uint64_t thr = prefix >> lo;
    int64_t m = 0;
    for (int i = 0; i < n; i++) m += ((uint64_t)key[i] >> lo) == thr;
    uint64_t o = need_max > 0 ? orc_splitmix64(seed, (uint64_t)row + 1u) % (uint64_t)m : 0;
    int out = 0;
    int64_t t = 0;
    for (int i = 0; i < n; i++) {
        uint64_t k = (uint64_t)key[i] >> lo;
        if (k > thr) {
            selected[out++] = i;
        } else if (k == thr) {
            int take = need_max > 0 ? (int)(((uint64_t)(t + 1) * need + o) / (uint64_t)m -
                                             ((uint64_t)t * need + o) / (uint64_t)m)
                                    : t < need;
            if (take) selected[out++] = i;
            t++;
        }
    }
    for (int i = out; i < top_k; i++) selected[i] = -1;
    free(key);
    return out;
}

/*
 * One full decode step for the listed rows (row r = b * hkv + g):
 * [TS s2.2] scores -> [TS s2.3] top-K -> attention over the selected pages.
 * top_k <= 0 means every page (dense paged decode).
 *
 *   q            [B][Hq][d] double
 *   meta         scorer 0: [n_pool][hkv][2][d] min/max rows; scorer 1: [n_pool][hkv][d]
 *                centroids (double; ignored when dense)
 *   scorer       0 = TinyServe bound [TS s2.2], 1 = Block Top-K centroid score [VX item 1]
 *   page_table   [B][max_pages] int32, seq_lens [B] int32
 *   selected_out [n_rows][max(top_k,1)] int32, n_sel_out [n_rows] (may be NULL when dense)
 *   scores_out   [n_rows][max_pages] double or NULL (-inf past n_b)
 *   out          [n_rows][G][d] double, lse [n_rows][G] double
 *
 * Rows are independent; they are spread over OpenMP threads.  Returns the
 * number of threads used, or -1 if any row met a bad index.
 */
int orc_step(const double *q, const void *k_pool, const void *v_pool, int kv_dtype, const double *meta,
             int scorer, const int32_t *page_table, const int32_t *seq_lens, int batch, int hq, int hkv, int d,
             int page_size, int max_pages, int64_t n_pool, int top_k, double sm_scale,
             const int32_t *rows, int n_rows, int32_t *selected_out, int32_t *n_sel_out,
             double *scores_out, double *out, double *lse) {
    int G = hq / hkv;
    int bad = 0;
    int threads = 1;
#pragma omp parallel reduction(| : bad)
    {
#ifdef _OPENMP
#pragma omp single
        threads = omp_get_num_threads();
#endif
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_pages);
        int32_t *all = (int32_t *)malloc(sizeof(int32_t) * (size_t)max_pages);
#pragma omp for schedule(dynamic, 1)
        for (int e = 0; e < n_rows; e++) {
            int r = rows[e];
            int b = r / hkv, g = r % hkv;
            if (b < 0 || b >= batch) {
                bad = 1;
                continue;
            }
            int seq_len = seq_lens[b];
            int n_b = (seq_len + page_size - 1) / page_size;
            if (n_b > max_pages) {
                bad = 1;
                n_b = max_pages;
            }
            const int32_t *table_row = page_table + (int64_t)b * max_pages;
            const double *q_group = q + ((int64_t)b * hq + (int64_t)g * G) * d;
            const int32_t *list;
            int n_list;
            if (top_k > 0) {
                int src = scorer == 1
                              ? orc_centroid_scores(q_group, G, meta, n_pool, hkv, g, d, table_row, n_b, scores)
                              : orc_row_scores(q_group, G, meta, n_pool, hkv, g, d, table_row, n_b, scores);
                if (src < 0) bad = 1;
                if (scores_out) {
                    for (int j = 0; j < max_pages; j++)
                        scores_out[(int64_t)e * max_pages + j] = j < n_b ? scores[j] : -INFINITY;
                }
                int32_t *sel = selected_out + (int64_t)e * top_k;
                n_list = orc_select(scores, n_b, top_k, sel);
                if (n_sel_out) n_sel_out[e] = n_list;
                list = sel;
            } else {
                for (int j = 0; j < n_b; j++) all[j] = j;
                n_list = n_b;
                if (n_sel_out) n_sel_out[e] = n_b;
                list = all;
            }
            if (orc_attend_row(q_group, G, k_pool, v_pool, kv_dtype, n_pool, hkv, g, page_size, d, table_row,
                               n_b, seq_len, list, n_list, sm_scale, out + (int64_t)e * G * d,
                               lse + (int64_t)e * G) < 0)
                bad = 1;
        }
        free(scores);
        free(all);
    }
    return bad ? -1 : threads;
}

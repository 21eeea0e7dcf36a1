/*
 * qskv.h -- query-aware sparse paged KV decode for GB300 (sm_103a).
 *
 * C ABI of libqskv.so.  Three calls make one decode step:
 *
 *   qskv_kv_meta_build       per-page min/max key metadata          (cache phase)
 *   qskv_page_select         bound score of every page + top-K      (indexer phase)
 *   qskv_sparse_paged_decode softmax(q K^T * scale) V over the selected pages,
 *                            split over warps and merged by log-sum-exp
 *
 * (qskv_page_select_refresh does the first two in one launch: the last
 * pages' metadata refresh inside the scoring grid; qskv_select_decode does
 * the whole step in one call: one launch when the rows fit one wave of
 * decode CTAs and a CTA's share of a row's metadata fits its shared memory,
 * else two or three),
 *
 * with an alternative block score (the mean key of each page, "Block Top-K"):
 *
 *   qskv_kv_centroid_build     per-page mean key (fp32)
 *   qskv_page_select_centroid  q . centroid of every page + top-K
 *
 * and a dense decode for batches that share a prefix of pages:
 *
 *   qskv_cascade_paged_decode  the shared prefix once per KV head on the
 *                              tensor cores, each row's own pages paged,
 *                              merged by log-sum-exp
 *
 * Sources (web pages on the method):
 *   TinyServe query-aware page selection article: s1 (fixed-size KV pages,
 *   selection per page), s2.1 (metadata m_j, M_j), s2.2 (bound score),
 *   s2.3 (score all pages, top-K, load only those pages, attend), s5.3
 *   (metadata refreshed every decode step).
 *   Vortex sparse-attention digest, method overview item 1: a query-
 *   independent cache phase (per-block summaries) and a query-dependent
 *   indexer phase (score, top-K, attend).
 *   CS336 Lecture 10 "Inference": s2.3 (decode attention), s5.1 (GQA: G query
 *   heads share one KV head), s9.2 (PagedAttention block table; shared
 *   prefixes map to the same physical blocks).
 *   Quail AI-SQL engine article, "the inference engine as an execution
 *   engine": partial attention results combined by log-sum-exp rescaling.
 *   Vortex digest, method overview item 1 (per-block mean keys scored by q,
 *   "Block Top-K").
 *
 * Layouts (row-major, all on the device unless stated; q, out and lse may
 * also be pinned host memory the device can address, which the kernels then
 * read and write directly, e.g. over GB300's NVLink-C2C host link; q, out
 * and lse are only read or written with plain loads and stores):
 *   k_pool, v_pool  [num_pool_pages][num_kv_heads][page_size][head_dim]  (kv dtype)
 *   meta            [num_pool_pages][num_kv_heads][2][head_dim]          (kv dtype)
 *                   row 0 = element-wise min m, row 1 = max M, over the
 *                   page's valid tokens
 *   q               [batch][num_q_heads][head_dim]                       (q dtype)
 *   page_table      [batch][max_pages] int32 physical page ids; entries
 *                   at or past ceil(seq_len / page_size) are never read;
 *                   several rows may name the same physical page (prefix sharing)
 *   seq_lens        [batch] int32 tokens per sequence, 0 <= seq_len <= max_pages*page_size
 *   selected        [batch][num_kv_heads][top_k] int32 logical page indices,
 *                   ascending, -1 padded
 *   n_selected      [batch][num_kv_heads] int32
 *   scores          [batch][num_kv_heads][max_pages] fp32
 *   out             [batch][num_q_heads][head_dim] fp32
 *   lse             [batch][num_q_heads] fp32 natural-log log-sum-exp of the
 *                   scaled logits
 * Query head h reads KV head h / G, G = num_q_heads / num_kv_heads.
 *
 * Supported: head_dim 64 or 128; page_size 16 or 32; G in {1, 2, 4, 8};
 * kv dtype fp32 or bf16 (meta has the kv dtype); q dtype fp32 or bf16;
 * batch * num_kv_heads <= 65535 (every call returns QSKV_ERR_UNSUPPORTED
 * beyond).
 * Every device pointer that is read or written in 16-byte vectors (q, k_pool,
 * v_pool, meta, out) must be 16-byte aligned; int32 arrays 4-byte aligned.
 *
 * Ownership: the caller allocates every buffer, including the workspace.  The
 * library allocates no device memory, keeps no state besides a per-device
 * attribute cache, launches only on the given stream (a cudaStream_t passed
 * as void*, NULL for the legacy default stream) and never synchronises,
 * except in qskv_get_error.
 *
 * Errors: a call returns a non-OK status before any launch when an argument
 * fails a host check (qskv_last_error_message() then says which), or
 * QSKV_ERR_CUDA when a launch fails.  Problems only the device can see (a
 * page id outside [0, num_pool_pages), a selected index outside the
 * sequence, seq_len beyond the table, a valid-token count outside
 * [1, page_size], a wait that timed out) never trap: the offending page is
 * skipped and a flag is raised in the workspace, which qskv_get_error reports.
 * Inputs must be finite except in slots past seq_len, which are never used.
 */
#ifndef QSKV_H
#define QSKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QSKV_OK = 0,
    QSKV_ERR_INVALID_ARG = 1,  /* a host-side argument check failed */
    QSKV_ERR_UNSUPPORTED = 2,  /* shape or dtype outside the supported set */
    QSKV_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small */
    QSKV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    QSKV_ERR_DEVICE_INDEX = 5, /* the device met an out-of-range index (page skipped) */
    QSKV_ERR_DEVICE_TIMEOUT = 6 /* a bounded device wait gave up (work abandoned) */
} qskv_status;

typedef enum { QSKV_F32 = 0, QSKV_BF16 = 1 } qskv_dtype;

/* Page score of the selection calls: the TinyServe bound over min/max
 * metadata, or the Block Top-K dot product with the mean key. */
typedef enum { QSKV_SCORE_BOUND = 0, QSKV_SCORE_CENTROID = 1 } qskv_scorer;

typedef struct {
    int32_t batch;          /* B: sequences */
    int32_t num_q_heads;    /* Hq */
    int32_t num_kv_heads;   /* Hkv; Hq % Hkv == 0 */
    int32_t head_dim;       /* d */
    int32_t page_size;      /* P: tokens per page */
    int32_t max_pages;      /* page_table row length */
    int32_t num_pool_pages; /* physical pages in k_pool / v_pool / meta */
} qskv_shape;

/*
 * Bytes of workspace one decode step needs on the current device (the three
 * calls may share one buffer).  The workspace must be 256-byte aligned and
 * zero-filled once before first use (e.g. cudaMemsetAsync); every call
 * leaves it ready for the next one.  It holds the device error word, a
 * counter per (sequence, KV head) row, a score buffer for callers that pass
 * none, and the split partial outputs of decode (one slot per row plus one
 * per decode warp).  Calls sharing a workspace must not run concurrently on
 * different streams.
 * Returns 0 if the shape is invalid or the device cannot be queried.
 */
size_t qskv_workspace_size(const qskv_shape *shape);

/*
 * Metadata build (TinyServe s2.1; refreshed every decode step, s5.3; the
 * cache phase of the Vortex two-phase split).
 * For each listed physical page p = page_ids[i] and every KV head g:
 *   meta[p][g][0][c] = min over t < valid_tokens[i] of k_pool[p][g][t][c]
 *   meta[p][g][1][c] = max over the same tokens
 * exactly, in the kv dtype.  Other pages' metadata is left untouched.  At
 * prefill list every page; at a decode step list each sequence's last page.
 *   page_ids, valid_tokens  [n_pages] int32 device arrays
 *   n_pages >= 0 (0 is a no-op)
 * Device errors: page id out of range or valid_tokens outside [1, page_size]
 * -> that entry is skipped, QSKV_ERR_DEVICE_INDEX is flagged.
 */
qskv_status qskv_kv_meta_build(const void *k_pool, qskv_dtype kv_dtype, const qskv_shape *shape,
                               const int32_t *page_ids, const int32_t *valid_tokens, int32_t n_pages,
                               void *meta, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Page selection (TinyServe s2.2-2.3; the indexer phase of the Vortex split).
 * For sequence b, KV head g and each logical page j < n_b = ceil(seq_len/P),
 * with p = page_table[b][j] and m, M the page's metadata:
 *   s_h(j)  = sum_c q[b][h][c] * (q[b][h][c] > 0 ? M[c] : m[c])  for each
 *             query head h of the group (an upper bound of max_t q_h . k_t)
 *   S(j)    = max over the group's heads of s_h(j)
 * selected[b][g][0..n) = the n = min(top_k, n_b) pages of largest S(j)
 * (equal scores: the lower page index wins), in ascending page order, -1 past
 * n; n_selected[b][g] = n.  Scores are computed in fp32; when `scores` is
 * non-NULL, S(j) is written to scores[b][g][j] for every j < n_b (entries
 * past n_b are left untouched), else a workspace buffer is used.
 * Device errors: a bad page id scores -inf and flags QSKV_ERR_DEVICE_INDEX.
 */
qskv_status qskv_page_select(const void *q, qskv_dtype q_dtype, const void *meta, qskv_dtype meta_dtype,
                             const int32_t *page_table, const int32_t *seq_lens, const qskv_shape *shape,
                             int32_t top_k, int32_t *selected, int32_t *n_selected, float *scores,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Metadata refresh of the pages the sequences append to, fused with page
 * selection (TinyServe s5.3: the metadata is refreshed at every decode step;
 * s2.2-2.3: score every page, keep the top K).  For every sequence b with
 * n_b >= 1 pages, its last page p = page_table[b][n_b - 1] holds
 * valid = seq_len - (n_b - 1) * page_size tokens: meta[p][g] is recomputed
 * from k_pool for every KV head g exactly as qskv_kv_meta_build does, and the
 * selection then runs exactly as qskv_page_select, scoring that page with its
 * new metadata.  The result is that of qskv_kv_meta_build over the last
 * pages followed by qskv_page_select, in one launch less.
 * meta is read and written ([num_pool_pages][num_kv_heads][2][head_dim],
 * bf16); the other pages' metadata must be current (built once at prefill).
 * A sequence's last page must not appear in another sequence's table (it is
 * being written to).  bf16 KV only (QSKV_ERR_UNSUPPORTED otherwise: use the
 * two calls); q fp32 or bf16.  Same workspace and device errors as
 * qskv_page_select.
 */
qskv_status qskv_page_select_refresh(const void *q, qskv_dtype q_dtype, const void *k_pool, void *meta,
                                     qskv_dtype kv_dtype, const int32_t *page_table, const int32_t *seq_lens,
                                     const qskv_shape *shape, int32_t top_k, int32_t *selected, int32_t *n_selected,
                                     float *scores, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Block summaries for the Block Top-K scorer (Vortex sparse-attention digest,
 * method overview item 1: the query-independent cache phase keeps each
 * block's mean key, "centroids").  For each listed physical page p and every
 * KV head g:
 *   centroids[p][g][c] = (1 / valid_tokens[i]) * sum over t < valid_tokens[i]
 *                        of k_pool[p][g][t][c]
 * in fp32 (sums of fp32 values, whatever the kv dtype), layout
 * [num_pool_pages][num_kv_heads][head_dim] fp32, 16-byte aligned.  Other
 * pages are left untouched.  Same list semantics and device errors as
 * qskv_kv_meta_build.
 */
qskv_status qskv_kv_centroid_build(const void *k_pool, qskv_dtype kv_dtype, const qskv_shape *shape,
                                   const int32_t *page_ids, const int32_t *valid_tokens, int32_t n_pages,
                                   float *centroids, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Page selection with the Block Top-K score (Vortex digest, method overview
 * item 1: the query-dependent indexer phase scores blocks from q and their
 * summaries and keeps the top-K).  For sequence b, KV head g and each logical
 * page j < n_b, with p = page_table[b][j]:
 *   S(j) = max over the group's query heads h of sum_c q[b][h][c] * centroids[p][g][c]
 * computed in fp32; then exactly as qskv_page_select: the n = min(top_k, n_b)
 * best pages (ties -> lower index), ascending, -1 padded; scores written to
 * `scores` (or a workspace buffer); same workspace and device errors.
 */
qskv_status qskv_page_select_centroid(const void *q, qskv_dtype q_dtype, const float *centroids,
                                      const int32_t *page_table, const int32_t *seq_lens, const qskv_shape *shape,
                                      int32_t top_k, int32_t *selected, int32_t *n_selected, float *scores,
                                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Page selection with a lossy top-K (Vortex digest, method overview item 3:
 * a radix Top-K that stops once enough high-confidence candidates are
 * collected and draws the rest at random from the threshold bin; the digest
 * reports recall@k > 0.97 at 1.3-1.6x the exact kernel's speed).
 * Scores as qskv_page_select (scorer QSKV_SCORE_BOUND: meta = [m | M] rows in
 * meta_dtype) or qskv_page_select_centroid (QSKV_SCORE_CENTROID: meta = fp32
 * centroids, meta_dtype QSKV_F32).  Ranking: the fp32 scores become
 * order-preserving 32-bit keys, and exact MSB-first radix passes over the
 * key's four 8-bit digits (bits 31..24, 23..16, 15..8, 7..0) narrow down
 * the threshold digit bucket until at most need_max keys are undecided,
 *   need_max = floor(epsilon * top_k)   (one IEEE double multiplication),
 * checked before each pass; every key above the threshold bucket is kept,
 * and the `need` still missing are drawn from that bucket's m keys (ranked
 * t = 0..m-1 in page order) by systematic sampling: key t is kept iff
 * floor(((t+1) need + o) / m) - floor((t need + o) / m) = 1, with
 * o = SplitMix64 output (row + 1) from `seed` (Steele, Lea and Flood 2014),
 * mod m.  Hence recall@top_k >= 1 - epsilon against the exact top-K of the
 * same fp32 scores, exactly min(top_k, n_b) pages, ascending.
 * epsilon in [0, 1); need_max = 0 (e.g. epsilon = 0) gives exactly
 * qskv_page_select's result.
 */
qskv_status qskv_page_select_approx(qskv_scorer scorer, const void *q, qskv_dtype q_dtype, const void *meta,
                                    qskv_dtype meta_dtype, const int32_t *page_table, const int32_t *seq_lens,
                                    const qskv_shape *shape, int32_t top_k, double epsilon, uint64_t seed,
                                    int32_t *selected, int32_t *n_selected, float *scores, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * Sparse paged decode attention (TinyServe s2.3 stages 3-4; split-K with a
 * log-sum-exp merge, Quail / flash decoding).
 * For each query head h of sequence b (KV head g = h / G), over the tokens
 * t < seq_len of the pages listed in selected[b][g][0..n_selected[b][g]):
 *   l_t = sm_scale * (q_h . k_t),  out[b][h] = sum_t softmax(l)_t v_t,
 *   lse[b][h] = log sum_t exp(l_t).
 * selected == NULL means every page j < n_b (exact dense paged decode);
 * n_selected and top_k are then ignored.  sm_scale == 0 means 1/sqrt(d).
 * Work split: when the (sequence, KV head) rows fit one wave of decode CTAs
 * (at most two per SM, at most 1024 units per row), each row goes to k CTAs
 * (k = 1 with at least one row per SM, else up to 8) whose warps' partial
 * results are combined in the CTA and, with k > 1, across the k CTAs by the
 * CTA drawing the row's last ticket (a per-row counter in the workspace);
 * otherwise the units are split evenly over the warps of a persistent grid
 * and a split row is combined by its last warp (when its pieces fit one
 * warp's single round of loads) or by a second kernel.  The per-row
 * counters are zero between calls (a zeroed workspace starts them so).
 * q, page_table and seq_lens may be read before the previous kernel in the
 * stream has completed when that kernel is one of this library's (which
 * never writes them); a kernel of the caller's is always waited for.
 * A sequence with no token gives out = 0 and lse = -inf.  lse may be NULL.
 * Device errors: a bad page id or selected index skips that page and flags
 * QSKV_ERR_DEVICE_INDEX.
 */
qskv_status qskv_sparse_paged_decode(const void *q, qskv_dtype q_dtype, const void *k_pool, const void *v_pool,
                                     qskv_dtype kv_dtype, const int32_t *page_table, const int32_t *seq_lens,
                                     const qskv_shape *shape, const int32_t *selected, const int32_t *n_selected,
                                     int32_t top_k, float sm_scale, float *out, float *lse, void *workspace,
                                     size_t workspace_bytes, void *stream);

/*
 * One decode step in one call (TinyServe query-aware page selection, s2.3:
 * score every page from its metadata, keep the top-K, load only those pages
 * and attend; s3.2 fuses those stages into one kernel; s5.3: the metadata of
 * the page the new token went into is refreshed every step).  The result is
 * exactly qskv_page_select_refresh(q, k_pool, meta, ..., top_k, selected,
 * n_selected, scores) followed by qskv_sparse_paged_decode(q, k_pool,
 * v_pool, ..., selected, n_selected, top_k, sm_scale, out, lse): the same
 * metadata update, the same selection (written to selected / n_selected, and
 * the scores to `scores` when it is not NULL), the same outputs, bit for bit.
 * Launches, by shape (rows = batch x num_kv_heads, k = decode CTAs per row as
 * in qskv_sparse_paged_decode):
 *   - k >= 2 and ceil(max_pages / k) pages of metadata fit a decode CTA's
 *     staging memory (368 pages for head_dim 64, 176 for 128): one launch.
 *     The k CTAs of a row form one thread-block cluster; the last one
 *     refreshes the last page's metadata, each scores its share of the
 *     row's pages, and after a cluster barrier each ranks the whole row and
 *     decodes its share of the selected pages (on a device where no cluster
 *     of k such CTAs fits, the two-launch form below instead);
 *   - otherwise k >= 1: the scoring grid (with the refresh), then the decode,
 *     whose CTAs rank their own rows first: two launches;
 *   - otherwise (more rows than fit one wave): scoring, ranking, decode.
 * bf16 KV only (QSKV_ERR_UNSUPPORTED otherwise); q fp32 or bf16; exact top-K
 * with the bound score.  Workspace: qskv_workspace_size(shape).  Same
 * argument checks and device errors as the two calls.
 */
qskv_status qskv_select_decode(const void *q, qskv_dtype q_dtype, const void *k_pool, const void *v_pool, void *meta,
                               qskv_dtype kv_dtype, const int32_t *page_table, const int32_t *seq_lens,
                               const qskv_shape *shape, int32_t top_k, float sm_scale, int32_t *selected,
                               int32_t *n_selected, float *scores, float *out, float *lse, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * qskv_sparse_paged_decode without a workspace, for callers that cannot
 * allocate device memory: for example a serving engine whose memory planner
 * hands out every byte of HBM up front and forbids later cudaMalloc calls,
 * or a latency-critical decode loop where cudaMalloc (which may synchronise
 * the device) is not allowed.  The pages have no counterpart of this call.
 *
 * Same arguments and results as qskv_sparse_paged_decode minus the
 * workspace.  The split partials, the row counters and the error word live
 * in an 8 MiB array of device memory built into the library (every GPU that
 * loads the library holds it until the process exits).  A shape whose
 * scratch (about 256 B + rows x 4 B + (rows + 12 x SM count) x G x
 * (head_dim + 1) x 4 B, rows = batch x num_kv_heads) exceeds 8 MiB is
 * rejected with QSKV_ERR_WORKSPACE before any launch.  Each call clears the
 * error word and the row counters with cudaMemsetAsync on `stream`; nothing
 * is allocated or freed.  Device-side index errors still
 * skip the offending page but are not reported (no workspace to read them
 * from): use qskv_sparse_paged_decode to diagnose.
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.  All calls
 * share the one array: calls that may overlap on the GPU (other streams,
 * other host threads) race and corrupt each other's results.
 */
qskv_status qskv_sparse_paged_decode_noalloc(const void *q, qskv_dtype q_dtype, const void *k_pool,
                                             const void *v_pool, qskv_dtype kv_dtype, const int32_t *page_table,
                                             const int32_t *seq_lens, const qskv_shape *shape,
                                             const int32_t *selected, const int32_t *n_selected, int32_t top_k,
                                             float sm_scale, float *out, float *lse, void *stream);

/*
 * Shared-prefix cascade decode (prefix sharing: CS336 Lecture 10 s9.2 --
 * sequences that start alike map their first logical blocks to the same
 * physical blocks; the attention over a shared anchor and over each
 * sequence's own suffix merged by log-sum-exp rescaling: Quail AI-SQL engine
 * article).
 *
 * Computes exactly what qskv_sparse_paged_decode computes with selected ==
 * NULL (dense attention over every token t < seq_len), for a batch whose
 * rows share their first `prefix_pages` pages: page_table[b][j] ==
 * page_table[0][j] for every b and every j < prefix_pages, and seq_len >=
 * prefix_pages * page_size for every b.  The prefix part is computed once
 * per KV head for all batch x G query rows as a dense product on the
 * tensor cores (reading the prefix pages once per call, not once per
 * sequence); each row's own pages j >= prefix_pages go through the paged
 * decode; the two are merged by log-sum-exp.
 *   prefix_pages  0 <= prefix_pages <= max_pages (0: plain dense decode)
 *   workspace     qskv_cascade_workspace_size(shape, prefix_pages) bytes,
 *                 256-byte aligned, zero-filled once (as for the other calls)
 * KV must be bf16 (QSKV_ERR_UNSUPPORTED otherwise); q fp32 or bf16.
 * Device errors: a row that breaks the sharing contract above flags
 * QSKV_ERR_DEVICE_INDEX (its output is then unspecified, nothing is read out
 * of bounds); bad page ids are skipped and flagged as in the other calls.
 */
size_t qskv_cascade_workspace_size(const qskv_shape *shape, int32_t prefix_pages);

qskv_status qskv_cascade_paged_decode(const void *q, qskv_dtype q_dtype, const void *k_pool, const void *v_pool,
                                      qskv_dtype kv_dtype, const int32_t *page_table, const int32_t *seq_lens,
                                      const qskv_shape *shape, int32_t prefix_pages, float sm_scale, float *out,
                                      float *lse, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Synchronises `stream`, reads and clears the workspace's device error flags,
 * and returns QSKV_OK, QSKV_ERR_DEVICE_INDEX, QSKV_ERR_DEVICE_TIMEOUT or
 * QSKV_ERR_CUDA.  The only call that blocks the host.
 */
qskv_status qskv_get_error(void *workspace, void *stream);

/* Static, human-readable name of a status. */
const char *qskv_status_string(qskv_status status);

/* Detail of the last non-OK status returned on this host thread ("" if none). */
const char *qskv_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* QSKV_H */

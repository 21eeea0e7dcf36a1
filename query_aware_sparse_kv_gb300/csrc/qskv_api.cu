// C ABI of libqskv.so: argument checks, workspace layout, TMA descriptors and
// kernel launches.  See include/qskv.h for the contract of each call.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>

#include "qskv.h"
#include "qskv_device.cuh"
#include "qskv_internal.h"

namespace qskv {

DecodeGrid decode_grid(int num_sms, int head_dim) {
    DecodeGrid g;
    g.ctas = kDecodeCtasPerSm * num_sms;
    g.warps_per_cta = decode_warps_per_cta(head_dim);
    g.total_warps = int64_t(g.ctas) * g.warps_per_cta;
    return g;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WorkspaceLayout workspace_layout(int64_t rows, int group, int head_dim, int max_pages, int num_sms,
                                 int extra_per_row) {
    WorkspaceLayout w;
    size_t off = 0;
    w.flags = off;
    off += 256;
    w.tickets = off;
    off = align256(off + size_t(rows) * 4);
    w.scores = off;
    off = align256(off + size_t(rows) * size_t(max_pages) * 4);
    w.slots = rows + decode_grid(num_sms, head_dim).total_warps + rows * extra_per_row;
    w.part_o = off;
    off = align256(off + size_t(w.slots) * group * head_dim * 4);
    w.part_lse = off;
    off = align256(off + size_t(w.slots) * group * 4);
    w.total = off;
    return w;
}

int l2_cache_bytes() {
    static std::atomic<int> cache[128];  // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 128) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 128) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace qskv

using namespace qskv;

namespace {

thread_local std::string g_last_error;

qskv_status fail(qskv_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

qskv_status ok() {
    g_last_error.clear();
    return QSKV_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// SM count of the current device (cached per device).
int current_sm_count(int *device_out) {
    static std::atomic<int> cache[128];  // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (device_out) *device_out = dev;
    if (dev >= 0 && dev < 128) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 128) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

qskv_status check_shape(const qskv_shape *s) {
    if (!s) return fail(QSKV_ERR_INVALID_ARG, "shape is NULL");
    if (s->batch < 1 || s->num_q_heads < 1 || s->num_kv_heads < 1 || s->max_pages < 1 || s->num_pool_pages < 1)
        return fail(QSKV_ERR_INVALID_ARG, "shape fields must be >= 1 (batch %d, Hq %d, Hkv %d, max_pages %d, pool %d)",
                    s->batch, s->num_q_heads, s->num_kv_heads, s->max_pages, s->num_pool_pages);
    if (s->num_q_heads % s->num_kv_heads != 0)
        return fail(QSKV_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", s->num_q_heads,
                    s->num_kv_heads);
    const int G = s->num_q_heads / s->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(QSKV_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", G);
    if (s->head_dim != 64 && s->head_dim != 128)
        return fail(QSKV_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", s->head_dim);
    if (s->page_size != 16 && s->page_size != 32)
        return fail(QSKV_ERR_UNSUPPORTED, "page_size must be 16 or 32 (got %d)", s->page_size);
    const int64_t rows = int64_t(s->batch) * s->num_kv_heads;
    if (rows > 65535) return fail(QSKV_ERR_UNSUPPORTED, "batch * num_kv_heads must be <= 65535 (got %lld)", (long long)rows);
    if (int64_t(s->num_pool_pages) >= (int64_t(1) << 25))
        return fail(QSKV_ERR_UNSUPPORTED, "num_pool_pages must be < 2^25");
    if (int64_t(s->num_pool_pages) * s->num_kv_heads * s->page_size >= (int64_t(1) << 31))
        return fail(QSKV_ERR_UNSUPPORTED, "num_pool_pages * num_kv_heads * page_size must be < 2^31");
    if (int64_t(s->max_pages) * s->page_size >= (int64_t(1) << 31))
        return fail(QSKV_ERR_UNSUPPORTED, "max_pages * page_size must be < 2^31");
    return QSKV_OK;
}

qskv_status check_dtype(int dt, const char *what) {
    if (dt != QSKV_F32 && dt != QSKV_BF16) return fail(QSKV_ERR_UNSUPPORTED, "%s dtype must be F32 or BF16 (%d)", what, dt);
    return QSKV_OK;
}

qskv_status check_workspace(void *ws, size_t bytes, size_t need) {
    if (!ws) return fail(QSKV_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(QSKV_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (bytes < need)
        return fail(QSKV_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", bytes, need);
    return QSKV_OK;
}

#define QSKV_TRY(expr)                    \
    do {                                  \
        qskv_status _s = (expr);          \
        if (_s != QSKV_OK) return _s;     \
    } while (0)

// ---------------------------------------------------------- TMA descriptors --
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// The pool viewed as a 2-D bf16 tensor [rows = Npool*Hkv*P][D], loaded in
// boxes of 16 token rows x 64 dims with 128-byte swizzle.
qskv_status make_pool_map(CUtensorMap *map, const void *pool, const qskv_shape *s) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(QSKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    const cuuint64_t dims[2] = {cuuint64_t(s->head_dim),
                                cuuint64_t(s->num_pool_pages) * s->num_kv_heads * s->page_size};
    const cuuint64_t strides[1] = {cuuint64_t(s->head_dim) * 2};
    const cuuint32_t box[2] = {64, 16};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QSKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return QSKV_OK;
}

qskv_status launched(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(QSKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

}  // namespace

extern "C" {

size_t qskv_workspace_size(const qskv_shape *shape) {
    if (check_shape(shape) != QSKV_OK) return 0;
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) {
        fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
        return 0;
    }
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    return workspace_layout(rows, shape->num_q_heads / shape->num_kv_heads, shape->head_dim, shape->max_pages, sms)
        .total;
}

qskv_status qskv_kv_meta_build(const void *k_pool, qskv_dtype kv_dtype, const qskv_shape *shape,
                               const int32_t *page_ids, const int32_t *valid_tokens, int32_t n_pages, void *meta,
                               void *workspace, size_t workspace_bytes, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(kv_dtype, "kv"));
    if (n_pages < 0) return fail(QSKV_ERR_INVALID_ARG, "n_pages must be >= 0 (got %d)", n_pages);
    QSKV_TRY(check_workspace(workspace, workspace_bytes, 256));
    if (n_pages == 0) return ok();
    if (!k_pool || !page_ids || !valid_tokens || !meta)
        return fail(QSKV_ERR_INVALID_ARG, "k_pool, page_ids, valid_tokens and meta must be non-NULL");
    if (!aligned(k_pool, 16) || !aligned(meta, 16)) return fail(QSKV_ERR_INVALID_ARG, "k_pool and meta must be 16-byte aligned");
    if (!aligned(page_ids, 4) || !aligned(valid_tokens, 4))
        return fail(QSKV_ERR_INVALID_ARG, "page_ids and valid_tokens must be 4-byte aligned");
    MetaArgs a;
    a.k_pool = k_pool;
    a.page_ids = page_ids;
    a.valid_tokens = valid_tokens;
    a.meta = meta;
    a.flags = static_cast<uint32_t *>(workspace);
    a.n_list = n_pages;
    a.num_kv_heads = shape->num_kv_heads;
    a.page_size = shape->page_size;
    a.num_pool_pages = shape->num_pool_pages;
    return launched(launch_meta_build(a, kv_dtype, shape->head_dim, static_cast<cudaStream_t>(stream)),
                    "kv_meta_build launch");
}

qskv_status qskv_page_select(const void *q, qskv_dtype q_dtype, const void *meta, qskv_dtype meta_dtype,
                             const int32_t *page_table, const int32_t *seq_lens, const qskv_shape *shape,
                             int32_t top_k, int32_t *selected, int32_t *n_selected, float *scores, void *workspace,
                             size_t workspace_bytes, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(q_dtype, "q"));
    QSKV_TRY(check_dtype(meta_dtype, "meta"));
    if (top_k < 1) return fail(QSKV_ERR_INVALID_ARG, "top_k must be >= 1 (got %d)", top_k);
    if (!q || !meta || !page_table || !seq_lens || !selected || !n_selected)
        return fail(QSKV_ERR_INVALID_ARG, "q, meta, page_table, seq_lens, selected and n_selected must be non-NULL");
    if (!aligned(q, 16) || !aligned(meta, 16)) return fail(QSKV_ERR_INVALID_ARG, "q and meta must be 16-byte aligned");
    if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(selected, 4) || !aligned(n_selected, 4) ||
        !aligned(scores, 4))
        return fail(QSKV_ERR_INVALID_ARG, "index and score arrays must be 4-byte aligned");
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) return fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const WorkspaceLayout L = workspace_layout(rows, G, shape->head_dim, shape->max_pages, sms);
    QSKV_TRY(check_workspace(workspace, workspace_bytes, L.total));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    SelectArgs a;
    a.k_pool = nullptr;
    a.meta_w = nullptr;
    a.q = q;
    a.meta = meta;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.selected = selected;
    a.n_selected = n_selected;
    a.scores = scores ? scores : reinterpret_cast<float *>(ws + L.scores);
    a.flags = reinterpret_cast<uint32_t *>(ws + L.flags);
    a.batch = shape->batch;
    a.num_q_heads = shape->num_q_heads;
    a.num_kv_heads = shape->num_kv_heads;
    a.group = G;
    a.page_size = shape->page_size;
    a.max_pages = shape->max_pages;
    a.num_pool_pages = shape->num_pool_pages;
    a.top_k = top_k;
    a.need_max = 0;
    a.seed = 0;
    a.meta_evict_first = 0;
    a.head_quads = 0;
    return launched(launch_page_select(a, q_dtype, meta_dtype, shape->head_dim, static_cast<cudaStream_t>(stream),
                                       scores != nullptr),
                    "page_select launch");
}

qskv_status qskv_page_select_refresh(const void *q, qskv_dtype q_dtype, const void *k_pool, void *meta,
                                     qskv_dtype kv_dtype, const int32_t *page_table, const int32_t *seq_lens,
                                     const qskv_shape *shape, int32_t top_k, int32_t *selected, int32_t *n_selected,
                                     float *scores, void *workspace, size_t workspace_bytes, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(q_dtype, "q"));
    QSKV_TRY(check_dtype(kv_dtype, "kv"));
    if (kv_dtype != QSKV_BF16)
        return fail(QSKV_ERR_UNSUPPORTED, "the fused refresh needs a bf16 KV cache (use qskv_kv_meta_build + qskv_page_select)");
    if (top_k < 1) return fail(QSKV_ERR_INVALID_ARG, "top_k must be >= 1 (got %d)", top_k);
    if (!q || !k_pool || !meta || !page_table || !seq_lens || !selected || !n_selected)
        return fail(QSKV_ERR_INVALID_ARG,
                    "q, k_pool, meta, page_table, seq_lens, selected and n_selected must be non-NULL");
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(meta, 16))
        return fail(QSKV_ERR_INVALID_ARG, "q, k_pool and meta must be 16-byte aligned");
    if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(selected, 4) || !aligned(n_selected, 4) ||
        !aligned(scores, 4))
        return fail(QSKV_ERR_INVALID_ARG, "index and score arrays must be 4-byte aligned");
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) return fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const WorkspaceLayout L = workspace_layout(rows, G, shape->head_dim, shape->max_pages, sms);
    QSKV_TRY(check_workspace(workspace, workspace_bytes, L.total));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    SelectArgs a;
    a.k_pool = k_pool;
    a.meta_w = meta;
    a.q = q;
    a.meta = meta;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.selected = selected;
    a.n_selected = n_selected;
    a.scores = scores ? scores : reinterpret_cast<float *>(ws + L.scores);
    a.flags = reinterpret_cast<uint32_t *>(ws + L.flags);
    a.batch = shape->batch;
    a.num_q_heads = shape->num_q_heads;
    a.num_kv_heads = shape->num_kv_heads;
    a.group = G;
    a.page_size = shape->page_size;
    a.max_pages = shape->max_pages;
    a.num_pool_pages = shape->num_pool_pages;
    a.top_k = top_k;
    a.need_max = 0;
    a.seed = 0;
    a.meta_evict_first = 0;
    a.head_quads = 0;
    return launched(launch_page_select(a, q_dtype, kv_dtype, shape->head_dim, static_cast<cudaStream_t>(stream),
                                       scores != nullptr, 1),
                    "page_select_refresh launch");
}

qskv_status qskv_kv_centroid_build(const void *k_pool, qskv_dtype kv_dtype, const qskv_shape *shape,
                                   const int32_t *page_ids, const int32_t *valid_tokens, int32_t n_pages,
                                   float *centroids, void *workspace, size_t workspace_bytes, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(kv_dtype, "kv"));
    if (n_pages < 0) return fail(QSKV_ERR_INVALID_ARG, "n_pages must be >= 0 (got %d)", n_pages);
    QSKV_TRY(check_workspace(workspace, workspace_bytes, 256));
    if (n_pages == 0) return ok();
    if (!k_pool || !page_ids || !valid_tokens || !centroids)
        return fail(QSKV_ERR_INVALID_ARG, "k_pool, page_ids, valid_tokens and centroids must be non-NULL");
    if (!aligned(k_pool, 16) || !aligned(centroids, 16))
        return fail(QSKV_ERR_INVALID_ARG, "k_pool and centroids must be 16-byte aligned");
    if (!aligned(page_ids, 4) || !aligned(valid_tokens, 4))
        return fail(QSKV_ERR_INVALID_ARG, "page_ids and valid_tokens must be 4-byte aligned");
    MetaArgs a;
    a.k_pool = k_pool;
    a.page_ids = page_ids;
    a.valid_tokens = valid_tokens;
    a.meta = centroids;
    a.flags = static_cast<uint32_t *>(workspace);
    a.n_list = n_pages;
    a.num_kv_heads = shape->num_kv_heads;
    a.page_size = shape->page_size;
    a.num_pool_pages = shape->num_pool_pages;
    return launched(launch_centroid_build(a, kv_dtype, shape->head_dim, static_cast<cudaStream_t>(stream)),
                    "kv_centroid_build launch");
}

qskv_status qskv_page_select_centroid(const void *q, qskv_dtype q_dtype, const float *centroids,
                                      const int32_t *page_table, const int32_t *seq_lens, const qskv_shape *shape,
                                      int32_t top_k, int32_t *selected, int32_t *n_selected, float *scores,
                                      void *workspace, size_t workspace_bytes, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(q_dtype, "q"));
    if (top_k < 1) return fail(QSKV_ERR_INVALID_ARG, "top_k must be >= 1 (got %d)", top_k);
    if (!q || !centroids || !page_table || !seq_lens || !selected || !n_selected)
        return fail(QSKV_ERR_INVALID_ARG,
                    "q, centroids, page_table, seq_lens, selected and n_selected must be non-NULL");
    if (!aligned(q, 16) || !aligned(centroids, 16))
        return fail(QSKV_ERR_INVALID_ARG, "q and centroids must be 16-byte aligned");
    if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(selected, 4) || !aligned(n_selected, 4) ||
        !aligned(scores, 4))
        return fail(QSKV_ERR_INVALID_ARG, "index and score arrays must be 4-byte aligned");
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) return fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const WorkspaceLayout L = workspace_layout(rows, G, shape->head_dim, shape->max_pages, sms);
    QSKV_TRY(check_workspace(workspace, workspace_bytes, L.total));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    SelectArgs a;
    a.k_pool = nullptr;
    a.meta_w = nullptr;
    a.q = q;
    a.meta = centroids;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.selected = selected;
    a.n_selected = n_selected;
    a.scores = scores ? scores : reinterpret_cast<float *>(ws + L.scores);
    a.flags = reinterpret_cast<uint32_t *>(ws + L.flags);
    a.batch = shape->batch;
    a.num_q_heads = shape->num_q_heads;
    a.num_kv_heads = shape->num_kv_heads;
    a.group = G;
    a.page_size = shape->page_size;
    a.max_pages = shape->max_pages;
    a.num_pool_pages = shape->num_pool_pages;
    a.top_k = top_k;
    a.need_max = 0;
    a.seed = 0;
    a.meta_evict_first = 0;
    a.head_quads = 0;
    return launched(launch_page_select_centroid(a, q_dtype, shape->head_dim, static_cast<cudaStream_t>(stream),
                                                scores != nullptr),
                    "page_select_centroid launch");
}

qskv_status qskv_page_select_approx(qskv_scorer scorer, const void *q, qskv_dtype q_dtype, const void *meta,
                                    qskv_dtype meta_dtype, const int32_t *page_table, const int32_t *seq_lens,
                                    const qskv_shape *shape, int32_t top_k, double epsilon, uint64_t seed,
                                    int32_t *selected, int32_t *n_selected, float *scores, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(q_dtype, "q"));
    QSKV_TRY(check_dtype(meta_dtype, "meta"));
    if (scorer != QSKV_SCORE_BOUND && scorer != QSKV_SCORE_CENTROID)
        return fail(QSKV_ERR_INVALID_ARG, "unknown scorer %d", int(scorer));
    if (scorer == QSKV_SCORE_CENTROID && meta_dtype != QSKV_F32)
        return fail(QSKV_ERR_INVALID_ARG, "centroid metadata is fp32");
    if (!(epsilon >= 0.0 && epsilon < 1.0)) return fail(QSKV_ERR_INVALID_ARG, "epsilon must be in [0, 1)");
    if (top_k < 1) return fail(QSKV_ERR_INVALID_ARG, "top_k must be >= 1 (got %d)", top_k);
    if (!q || !meta || !page_table || !seq_lens || !selected || !n_selected)
        return fail(QSKV_ERR_INVALID_ARG, "q, meta, page_table, seq_lens, selected and n_selected must be non-NULL");
    if (!aligned(q, 16) || !aligned(meta, 16)) return fail(QSKV_ERR_INVALID_ARG, "q and meta must be 16-byte aligned");
    if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(selected, 4) || !aligned(n_selected, 4) ||
        !aligned(scores, 4))
        return fail(QSKV_ERR_INVALID_ARG, "index and score arrays must be 4-byte aligned");
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) return fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const WorkspaceLayout L = workspace_layout(rows, G, shape->head_dim, shape->max_pages, sms);
    QSKV_TRY(check_workspace(workspace, workspace_bytes, L.total));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    SelectArgs a;
    a.k_pool = nullptr;
    a.meta_w = nullptr;
    a.q = q;
    a.meta = meta;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.selected = selected;
    a.n_selected = n_selected;
    a.scores = scores ? scores : reinterpret_cast<float *>(ws + L.scores);
    a.flags = reinterpret_cast<uint32_t *>(ws + L.flags);
    a.batch = shape->batch;
    a.num_q_heads = shape->num_q_heads;
    a.num_kv_heads = shape->num_kv_heads;
    a.group = G;
    a.page_size = shape->page_size;
    a.max_pages = shape->max_pages;
    a.num_pool_pages = shape->num_pool_pages;
    a.top_k = top_k;
    a.need_max = int32_t(floor(epsilon * double(top_k)));
    a.seed = seed;
    a.meta_evict_first = 0;
    a.head_quads = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = scorer == QSKV_SCORE_CENTROID
                              ? launch_page_select_centroid(a, q_dtype, shape->head_dim, st, scores != nullptr)
                              : launch_page_select(a, q_dtype, meta_dtype, shape->head_dim, st, scores != nullptr);
    return launched(e, "page_select_approx launch");
}

qskv_status qskv_select_decode(const void *q, qskv_dtype q_dtype, const void *k_pool, const void *v_pool, void *meta,
                               qskv_dtype kv_dtype, const int32_t *page_table, const int32_t *seq_lens,
                               const qskv_shape *shape, int32_t top_k, float sm_scale, int32_t *selected,
                               int32_t *n_selected, float *scores, float *out, float *lse, void *workspace,
                               size_t workspace_bytes, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(q_dtype, "q"));
    QSKV_TRY(check_dtype(kv_dtype, "kv"));
    if (kv_dtype != QSKV_BF16)
        return fail(QSKV_ERR_UNSUPPORTED, "qskv_select_decode needs a bf16 KV cache (use the separate calls)");
    if (top_k < 1) return fail(QSKV_ERR_INVALID_ARG, "top_k must be >= 1 (got %d)", top_k);
    if (!q || !k_pool || !v_pool || !meta || !page_table || !seq_lens || !selected || !n_selected || !out)
        return fail(QSKV_ERR_INVALID_ARG,
                    "q, k_pool, v_pool, meta, page_table, seq_lens, selected, n_selected and out must be non-NULL");
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(meta, 16) || !aligned(out, 16))
        return fail(QSKV_ERR_INVALID_ARG, "q, k_pool, v_pool, meta and out must be 16-byte aligned");
    if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(selected, 4) || !aligned(n_selected, 4) ||
        !aligned(scores, 4) || !aligned(lse, 4))
        return fail(QSKV_ERR_INVALID_ARG, "index, score and lse arrays must be 4-byte aligned");
    if (!(sm_scale >= 0.f) || isinf(sm_scale)) return fail(QSKV_ERR_INVALID_ARG, "sm_scale must be finite and >= 0");
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) return fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const WorkspaceLayout L = workspace_layout(rows, G, shape->head_dim, shape->max_pages, sms);
    QSKV_TRY(check_workspace(workspace, workspace_bytes, L.total));
    const DecodeGrid grid = decode_grid(sms, shape->head_dim);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *sc = scores ? scores : reinterpret_cast<float *>(ws + L.scores);
    uint32_t *tickets = reinterpret_cast<uint32_t *>(ws + L.tickets);
    // The decode ranks its own rows when they go one row per k CTAs.  With
    // k >= 2, when each CTA's share of a full row's pages (max_pages / k)
    // fits its staging memory at once, it also scores them (the k CTAs of a
    // row one cluster) and the step is that one launch; longer shares would
    // be staged in serial rounds, slower than the scoring grid (measured).
    const int rk = row_blocks_for(rows, top_k, grid.ctas, true, true);
    const bool fused = rk > 0;
    const bool fused_score = rk >= kFusedScoreMinBlocks &&
                             (int64_t(shape->max_pages) + rk - 1) / rk <= fused_score_pages_per_round(shape->head_dim);

    SelectArgs sa;
    sa.k_pool = k_pool;
    sa.meta_w = meta;
    sa.q = q;
    sa.meta = meta;
    sa.page_table = page_table;
    sa.seq_lens = seq_lens;
    sa.selected = selected;
    sa.n_selected = n_selected;
    sa.scores = sc;
    sa.flags = reinterpret_cast<uint32_t *>(ws + L.flags);
    sa.batch = shape->batch;
    sa.num_q_heads = shape->num_q_heads;
    sa.num_kv_heads = shape->num_kv_heads;
    sa.group = G;
    sa.page_size = shape->page_size;
    sa.max_pages = shape->max_pages;
    sa.num_pool_pages = shape->num_pool_pages;
    sa.top_k = top_k;
    sa.need_max = 0;
    sa.seed = 0;
    sa.meta_evict_first = 0;
    sa.head_quads = 0;

    DecodeArgs a;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.selected = selected;
    a.n_selected = n_selected;
    a.out = out;
    a.lse = lse;
    a.part_o = reinterpret_cast<float *>(ws + L.part_o);
    a.part_lse = reinterpret_cast<float *>(ws + L.part_lse);
    a.flags = reinterpret_cast<uint32_t *>(ws + L.flags);
    a.batch = shape->batch;
    a.num_q_heads = shape->num_q_heads;
    a.num_kv_heads = shape->num_kv_heads;
    a.group = G;
    a.page_size = shape->page_size;
    a.max_pages = shape->max_pages;
    a.num_pool_pages = shape->num_pool_pages;
    a.top_k = top_k;
    a.slots_per_row = top_k;
    a.page_begin = 0;
    a.extra_pieces = 0;
    a.extra_slot0 = 0;
    a.wait_at_exit = 0;
    a.kv_evict_first = 0;
    a.stages = decode_stages(shape->head_dim);
    a.tickets = tickets;
    a.fold = 0;
    a.total_units = rows * a.slots_per_row;
    a.units_per_warp = (a.total_units + grid.total_warps - 1) / grid.total_warps;
    const float scale = sm_scale > 0.f ? sm_scale : 1.f / sqrtf(float(shape->head_dim));
    a.scale_log2 = scale * 1.4426950408889634f;
    if (fused) {
        a.scores = sc;
        a.selected_out = selected;
        a.n_selected_out = n_selected;
    }
    CUtensorMap tk, tv;
    QSKV_TRY(make_pool_map(&tk, k_pool, shape));
    QSKV_TRY(make_pool_map(&tv, v_pool, shape));
    if (fused_score) {
        DecodeArgs af = a;
        af.meta = meta;
        af.meta_w = meta;
        af.refresh = 1;
        af.score_all = scores != nullptr ? 1 : 0;
        const cudaError_t e = launch_decode(af, &tk, &tv, q_dtype, kv_dtype, shape->head_dim, grid, st);
        // cudaErrorNotSupported: no cluster of rk such CTAs fits this device
        // (nothing was launched); the two-launch form below serves instead
        if (e != cudaErrorNotSupported) return launched(e, "select_decode launch");
    }
    QSKV_TRY(launched(launch_page_select(sa, q_dtype, QSKV_BF16, shape->head_dim, st, scores != nullptr, 1,
                                         fused ? 0 : 1),
                      "select_decode scoring launch"));
    return launched(launch_decode(a, &tk, &tv, q_dtype, kv_dtype, shape->head_dim, grid, st),
                    "select_decode decode launch");
}

qskv_status qskv_sparse_paged_decode(const void *q, qskv_dtype q_dtype, const void *k_pool, const void *v_pool,
                                     qskv_dtype kv_dtype, const int32_t *page_table, const int32_t *seq_lens,
                                     const qskv_shape *shape, const int32_t *selected, const int32_t *n_selected,
                                     int32_t top_k, float sm_scale, float *out, float *lse, void *workspace,
                                     size_t workspace_bytes, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(q_dtype, "q"));
    QSKV_TRY(check_dtype(kv_dtype, "kv"));
    if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !out)
        return fail(QSKV_ERR_INVALID_ARG, "q, k_pool, v_pool, page_table, seq_lens and out must be non-NULL");
    if (selected && (!n_selected || top_k < 1))
        return fail(QSKV_ERR_INVALID_ARG, "with a selected list, n_selected must be non-NULL and top_k >= 1");
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16))
        return fail(QSKV_ERR_INVALID_ARG, "q, k_pool, v_pool and out must be 16-byte aligned");
    if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(selected, 4) || !aligned(n_selected, 4) ||
        !aligned(lse, 4))
        return fail(QSKV_ERR_INVALID_ARG, "index and lse arrays must be 4-byte aligned");
    if (!(sm_scale >= 0.f) || isinf(sm_scale)) return fail(QSKV_ERR_INVALID_ARG, "sm_scale must be finite and >= 0");
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) return fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const WorkspaceLayout L = workspace_layout(rows, G, shape->head_dim, shape->max_pages, sms);
    QSKV_TRY(check_workspace(workspace, workspace_bytes, L.total));
    const DecodeGrid grid = decode_grid(sms, shape->head_dim);
    uint8_t *ws = static_cast<uint8_t *>(workspace);

    DecodeArgs a;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.selected = selected;
    a.n_selected = n_selected;
    a.out = out;
    a.lse = lse;
    a.part_o = reinterpret_cast<float *>(ws + L.part_o);
    a.part_lse = reinterpret_cast<float *>(ws + L.part_lse);
    a.flags = reinterpret_cast<uint32_t *>(ws + L.flags);
    a.batch = shape->batch;
    a.num_q_heads = shape->num_q_heads;
    a.num_kv_heads = shape->num_kv_heads;
    a.group = G;
    a.page_size = shape->page_size;
    a.max_pages = shape->max_pages;
    a.num_pool_pages = shape->num_pool_pages;
    a.top_k = selected ? top_k : 0;
    a.slots_per_row = selected ? top_k : shape->max_pages;
    a.page_begin = 0;
    a.extra_pieces = 0;
    a.extra_slot0 = 0;
    a.wait_at_exit = 0;
    a.kv_evict_first = 0;
    a.stages = decode_stages(shape->head_dim);
    a.tickets = reinterpret_cast<uint32_t *>(ws + L.tickets);
    a.fold = 0;
    a.total_units = rows * a.slots_per_row;
    a.units_per_warp = (a.total_units + grid.total_warps - 1) / grid.total_warps;
    const float scale = sm_scale > 0.f ? sm_scale : 1.f / sqrtf(float(shape->head_dim));
    a.scale_log2 = scale * 1.4426950408889634f;

    CUtensorMap tk, tv;
    memset(&tk, 0, sizeof tk);
    memset(&tv, 0, sizeof tv);
    if (kv_dtype == QSKV_BF16) {
        QSKV_TRY(make_pool_map(&tk, k_pool, shape));
        QSKV_TRY(make_pool_map(&tv, v_pool, shape));
    }
    return launched(launch_decode(a, &tk, &tv, q_dtype, kv_dtype, shape->head_dim, grid, static_cast<cudaStream_t>(stream)),
                    "sparse_paged_decode launch");
}

qskv_status qskv_sparse_paged_decode_noalloc(const void *q, qskv_dtype q_dtype, const void *k_pool,
                                             const void *v_pool, qskv_dtype kv_dtype, const int32_t *page_table,
                                             const int32_t *seq_lens, const qskv_shape *shape,
                                             const int32_t *selected, const int32_t *n_selected, int32_t top_k,
                                             float sm_scale, float *out, float *lse, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(q_dtype, "q"));
    QSKV_TRY(check_dtype(kv_dtype, "kv"));
    if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !out)
        return fail(QSKV_ERR_INVALID_ARG, "q, k_pool, v_pool, page_table, seq_lens and out must be non-NULL");
    if (selected && (!n_selected || top_k < 1))
        return fail(QSKV_ERR_INVALID_ARG, "with a selected list, n_selected must be non-NULL and top_k >= 1");
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16))
        return fail(QSKV_ERR_INVALID_ARG, "q, k_pool, v_pool and out must be 16-byte aligned");
    if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(selected, 4) || !aligned(n_selected, 4) ||
        !aligned(lse, 4))
        return fail(QSKV_ERR_INVALID_ARG, "index and lse arrays must be 4-byte aligned");
    if (!(sm_scale >= 0.f) || isinf(sm_scale)) return fail(QSKV_ERR_INVALID_ARG, "sm_scale must be finite and >= 0");
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) return fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const DecodeGrid grid = decode_grid(sms, shape->head_dim);

    // Layout inside the static scratch: error word, per-row counters, then the partials.
    const int64_t slots = rows + grid.total_warps;
    const size_t off_tickets = 256;
    const size_t off_part_o = align256(off_tickets + size_t(rows) * 4);
    const size_t off_part_lse = align256(off_part_o + size_t(slots) * G * shape->head_dim * 4);
    const size_t need = align256(off_part_lse + size_t(slots) * G * 4);
    if (need > kNoallocScratchBytes)
        return fail(QSKV_ERR_WORKSPACE,
                    "this shape needs %zu bytes of decode scratch but the built-in buffer holds %zu; "
                    "call qskv_sparse_paged_decode with a caller-allocated workspace instead",
                    need, kNoallocScratchBytes);
    void *scratch = nullptr;
    cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return fail(QSKV_ERR_CUDA, "cudaGetSymbolAddress of the decode scratch: %s", cudaGetErrorString(e));
    uint8_t *ws = static_cast<uint8_t *>(scratch);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the error word and the row counters start at zero on every call
    e = cudaMemsetAsync(ws, 0, off_part_o, st);
    if (e != cudaSuccess) return fail(QSKV_ERR_CUDA, "clearing the decode scratch: %s", cudaGetErrorString(e));

    DecodeArgs a;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.selected = selected;
    a.n_selected = n_selected;
    a.out = out;
    a.lse = lse;
    a.part_o = reinterpret_cast<float *>(ws + off_part_o);
    a.part_lse = reinterpret_cast<float *>(ws + off_part_lse);
    a.flags = reinterpret_cast<uint32_t *>(ws);
    a.batch = shape->batch;
    a.num_q_heads = shape->num_q_heads;
    a.num_kv_heads = shape->num_kv_heads;
    a.group = G;
    a.page_size = shape->page_size;
    a.max_pages = shape->max_pages;
    a.num_pool_pages = shape->num_pool_pages;
    a.top_k = selected ? top_k : 0;
    a.slots_per_row = selected ? top_k : shape->max_pages;
    a.page_begin = 0;
    a.extra_pieces = 0;
    a.extra_slot0 = 0;
    a.wait_at_exit = 0;
    a.kv_evict_first = 0;
    a.stages = decode_stages(shape->head_dim);
    a.tickets = reinterpret_cast<uint32_t *>(ws + off_tickets);
    a.fold = 0;
    a.total_units = rows * a.slots_per_row;
    a.units_per_warp = (a.total_units + grid.total_warps - 1) / grid.total_warps;
    const float scale = sm_scale > 0.f ? sm_scale : 1.f / sqrtf(float(shape->head_dim));
    a.scale_log2 = scale * 1.4426950408889634f;

    CUtensorMap tk, tv;
    memset(&tk, 0, sizeof tk);
    memset(&tv, 0, sizeof tv);
    if (kv_dtype == QSKV_BF16) {
        QSKV_TRY(make_pool_map(&tk, k_pool, shape));
        QSKV_TRY(make_pool_map(&tv, v_pool, shape));
    }
    return launched(launch_decode(a, &tk, &tv, q_dtype, kv_dtype, shape->head_dim, grid, st),
                    "sparse_paged_decode_noalloc launch");
}

size_t qskv_cascade_workspace_size(const qskv_shape *shape, int32_t prefix_pages) {
    if (check_shape(shape) != QSKV_OK) return 0;
    if (prefix_pages < 0 || prefix_pages > shape->max_pages) {
        fail(QSKV_ERR_INVALID_ARG, "prefix_pages must be in [0, max_pages] (got %d)", prefix_pages);
        return 0;
    }
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) {
        fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
        return 0;
    }
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const int E = prefix_splits(shape->batch, G, shape->num_kv_heads, shape->page_size, prefix_pages, sms);
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    return workspace_layout(rows, G, shape->head_dim, shape->max_pages, sms, E).total;
}

qskv_status qskv_cascade_paged_decode(const void *q, qskv_dtype q_dtype, const void *k_pool, const void *v_pool,
                                      qskv_dtype kv_dtype, const int32_t *page_table, const int32_t *seq_lens,
                                      const qskv_shape *shape, int32_t prefix_pages, float sm_scale, float *out,
                                      float *lse, void *workspace, size_t workspace_bytes, void *stream) {
    QSKV_TRY(check_shape(shape));
    QSKV_TRY(check_dtype(q_dtype, "q"));
    QSKV_TRY(check_dtype(kv_dtype, "kv"));
    if (kv_dtype != QSKV_BF16) return fail(QSKV_ERR_UNSUPPORTED, "the cascade decode needs a bf16 KV cache");
    if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !out)
        return fail(QSKV_ERR_INVALID_ARG, "q, k_pool, v_pool, page_table, seq_lens and out must be non-NULL");
    if (prefix_pages < 0 || prefix_pages > shape->max_pages)
        return fail(QSKV_ERR_INVALID_ARG, "prefix_pages must be in [0, max_pages] (got %d)", prefix_pages);
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16))
        return fail(QSKV_ERR_INVALID_ARG, "q, k_pool, v_pool and out must be 16-byte aligned");
    if (!aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(lse, 4))
        return fail(QSKV_ERR_INVALID_ARG, "index and lse arrays must be 4-byte aligned");
    if (!(sm_scale >= 0.f) || isinf(sm_scale)) return fail(QSKV_ERR_INVALID_ARG, "sm_scale must be finite and >= 0");
    const int sms = current_sm_count(nullptr);
    if (sms <= 0) return fail(QSKV_ERR_CUDA, "cannot query the current CUDA device");
    const int64_t rows = int64_t(shape->batch) * shape->num_kv_heads;
    const int G = shape->num_q_heads / shape->num_kv_heads;
    const int E = prefix_splits(shape->batch, G, shape->num_kv_heads, shape->page_size, prefix_pages, sms);
    const WorkspaceLayout L = workspace_layout(rows, G, shape->head_dim, shape->max_pages, sms, E);
    QSKV_TRY(check_workspace(workspace, workspace_bytes, L.total));
    // The prefix runs as a persistent grid on a share of the SMs and the
    // paged decode of the rows' own pages on the others, side by side.  The
    // partial slots keep the full grid's layout (prefix pieces after every
    // decode warp's slot).
    const DecodeGrid full = decode_grid(sms, shape->head_dim);
    const int prefix_items = E > 0 ? prefix_tiles(shape->batch, G) * shape->num_kv_heads * E : 0;
    const int pctas = prefix_ctas(prefix_items, sms);
    const DecodeGrid grid = decode_grid(sms - pctas > 0 ? sms - pctas : 1, shape->head_dim);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const float scale = sm_scale > 0.f ? sm_scale : 1.f / sqrtf(float(shape->head_dim));

    DecodeArgs a;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.page_table = page_table;
    a.seq_lens = seq_lens;
    a.selected = nullptr;
    a.n_selected = nullptr;
    a.out = out;
    a.lse = lse;
    a.part_o = reinterpret_cast<float *>(ws + L.part_o);
    a.part_lse = reinterpret_cast<float *>(ws + L.part_lse);
    a.flags = reinterpret_cast<uint32_t *>(ws + L.flags);
    a.batch = shape->batch;
    a.num_q_heads = shape->num_q_heads;
    a.num_kv_heads = shape->num_kv_heads;
    a.group = G;
    a.page_size = shape->page_size;
    a.max_pages = shape->max_pages;
    a.num_pool_pages = shape->num_pool_pages;
    a.top_k = 0;
    a.page_begin = E > 0 ? prefix_pages : 0;
    a.slots_per_row = shape->max_pages - a.page_begin;
    a.extra_pieces = E;
    a.extra_slot0 = rows + full.total_warps;
    a.wait_at_exit = 0;
    a.kv_evict_first = 0;
    a.stages = decode_stages(shape->head_dim);
    a.tickets = reinterpret_cast<uint32_t *>(ws + L.tickets);
    a.fold = 0;
    a.total_units = rows * a.slots_per_row;
    a.units_per_warp = (a.total_units + grid.total_warps - 1) / grid.total_warps;
    a.scale_log2 = scale * 1.4426950408889634f;

    PrefixArgs p;
    p.q = q;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.part_o = a.part_o;
    p.part_lse = a.part_lse;
    p.flags = a.flags;
    p.batch = shape->batch;
    p.num_q_heads = shape->num_q_heads;
    p.num_kv_heads = shape->num_kv_heads;
    p.group = G;
    p.page_size = shape->page_size;
    p.max_pages = shape->max_pages;
    p.num_pool_pages = shape->num_pool_pages;
    p.prefix_pages = prefix_pages;
    p.splits = E;
    p.ctas = pctas;
    p.slot0 = a.extra_slot0;
    p.scale_log2 = a.scale_log2;

    CUtensorMap tk, tv;
    memset(&tk, 0, sizeof tk);
    memset(&tv, 0, sizeof tv);
    QSKV_TRY(make_pool_map(&tk, k_pool, shape));
    QSKV_TRY(make_pool_map(&tv, v_pool, shape));
    return launched(launch_decode(a, &tk, &tv, q_dtype, kv_dtype, shape->head_dim, grid,
                                  static_cast<cudaStream_t>(stream), E > 0 ? &p : nullptr),
                    "cascade_paged_decode launch");
}

qskv_status qskv_get_error(void *workspace, void *stream) {
    if (!workspace) return fail(QSKV_ERR_WORKSPACE, "workspace is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t flags = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&flags, workspace, sizeof flags, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof flags, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(QSKV_ERR_CUDA, "qskv_get_error: %s", cudaGetErrorString(e));
    if (flags == 0) return ok();
    std::string what;
    if (flags & kErrPageId) what += " page-id-out-of-range";
    if (flags & kErrSelected) what += " selected-index-out-of-range";
    if (flags & kErrSeqLen) what += " seq_len-out-of-range";
    if (flags & kErrValid) what += " valid-tokens-out-of-range";
    if (flags & kErrTimeout) what += " wait-timeout";
    if (flags & kErrPrefix) what += " shared-prefix-contract-broken";
    if (flags & kErrTimeout) return fail(QSKV_ERR_DEVICE_TIMEOUT, "device flags:%s", what.c_str());
    return fail(QSKV_ERR_DEVICE_INDEX, "device flags:%s", what.c_str());
}

const char *qskv_status_string(qskv_status status) {
    switch (status) {
        case QSKV_OK: return "QSKV_OK";
        case QSKV_ERR_INVALID_ARG: return "QSKV_ERR_INVALID_ARG";
        case QSKV_ERR_UNSUPPORTED: return "QSKV_ERR_UNSUPPORTED";
        case QSKV_ERR_WORKSPACE: return "QSKV_ERR_WORKSPACE";
        case QSKV_ERR_CUDA: return "QSKV_ERR_CUDA";
        case QSKV_ERR_DEVICE_INDEX: return "QSKV_ERR_DEVICE_INDEX";
        case QSKV_ERR_DEVICE_TIMEOUT: return "QSKV_ERR_DEVICE_TIMEOUT";
    }
    return "QSKV_UNKNOWN_STATUS";
}

const char *qskv_last_error_message(void) { return g_last_error.c_str(); }

}  // extern "C"

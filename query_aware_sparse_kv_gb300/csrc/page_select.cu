// Page selection: bound score of every page, then the top-K pages per
// (sequence, KV head) row.
//
// TinyServe query-aware page selection, s2.2: for query q and page j with
// metadata (m_j, M_j), score_j = sum_i q[i] * (q[i] > 0 ? M_j[i] : m_j[i]),
// an upper bound of the page's largest q.k.  s2.3: all pages are scored in
// parallel ("metadata parallel scan"), then the K best are picked by a radix
// pass in shared memory.  With grouped-query attention the row score is the
// maximum of the G query heads' bounds (one selection per KV head).
//
// Scoring, bf16 metadata.  With q- = min(q, 0) and q+ = max(q, 0), the bound
// is the dot product  [m_j | M_j] . [q- | q+]  (exact rewrite: for q > 0 the
// first term is 0 and the second q M; for q < 0 the reverse; for q = 0 both
// vanish).  So the scores of 16 pages for the G <= 8 heads of a group form a
// (16 pages x 2d) . (2d x 8 heads) product: each warp runs it as m16n8k16
// bf16 mma.sync with fp32 accumulation, the 16 metadata rows being the A
// operand read straight from global memory in 16-byte vectors.  A and B use
// the same permutation of the 2d-long k axis (each lane's 16-byte chunk feeds
// two k-steps), which the dot product does not see.  bf16 products are exact
// in fp32; fp32 queries are split as hi + lo bf16 pairs (two mma per step).
// The same identity runs on CUDA cores (fp32 FMA) for fp32 metadata.
//
// Selection.  A second kernel (launched with programmatic dependent launch,
// so it is resident when scoring drains) ranks each row in one CTA.  Scores
// map to order-preserving 32-bit keys; an MSB-first radix select over 8-bit
// digits, starting at the highest bit where the row's keys differ, finds the
// K-th key; a stable compaction in page order keeps every key above it and
// the lowest-index keys equal to it.  The selected list comes out in
// ascending page order.
#include <type_traits>

#include "qskv_device.cuh"
#include "qskv_internal.h"
#include "qskv_select.cuh"

namespace qskv {
namespace {

// Row bookkeeping shared by both score kernels.
struct RowInfo {
    int row, b, g, n_b, seq;
};

__device__ __forceinline__ RowInfo row_info(const SelectArgs &a) {
    // No early trigger here: the scoring grid runs several waves, and ranking
    // CTAs made resident early would take thread slots and shared memory
    // from its later waves (measured: up to 20 % slower steps).  The ranking
    // grid launches when scoring completes.
    pdl_wait();
    RowInfo r;
    r.row = blockIdx.y;
    r.b = r.row / a.num_kv_heads;
    r.g = r.row % a.num_kv_heads;
    int seq = a.seq_lens[r.b];
    const int cap = a.max_pages * a.page_size;
    if (seq < 0 || seq > cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(a.flags, kErrSeqLen);
        seq = seq < 0 ? 0 : cap;
    }
    r.seq = seq;
    r.n_b = (seq + a.page_size - 1) / a.page_size;
    return r;
}

// One CTA per row: rank the row's scores.
__global__ void __launch_bounds__(kSelectThreads) select_kernel(SelectArgs a) {
    pdl_trigger();
    pdl_wait();
    const int row = blockIdx.x;
    const int b = row / a.num_kv_heads;
    int seq = a.seq_lens[b];
    const int cap = a.max_pages * a.page_size;
    seq = seq < 0 ? 0 : (seq > cap ? cap : seq);  // flagged by the scoring kernel
    const int n_b = (seq + a.page_size - 1) / a.page_size;
    __shared__ uint32_t s_keys[kSelectKeyCap];
    __shared__ uint32_t s_hist[256];
    __shared__ int s_tmp[2 * kSelectThreads / 32];
    __shared__ uint32_t s_mm[2 * kSelectThreads / 32];
    __shared__ int s_pick[3];
    const SelectSmem sm{s_keys, s_hist, s_mm, s_tmp, s_pick};
    select_row<kSelectThreads>(a, row, n_b, a.scores + int64_t(row) * a.max_pages, sm, nullptr, true);
}

// ---------------------------------------------- scores on tensor cores --
// One warp scores 32 pages of a row: two groups of 16 pages, each a
// (16 pages x 2D) . (2D x 8 heads) mma.sync product (bound_group_scores).

// Query chunks of head `gid` of KV head g's group (zero past the group).
template <int D, bool QF32>
__device__ __forceinline__ void bound_load_q(const SelectArgs &a, int b, int g, uint4 (&qraw)[2 * D / 32][QF32 ? 2 : 1]) {
    constexpr int NKP = BoundScanRegs<D>::NKP;
    const int lane = threadIdx.x & 31, t = lane & 3, gid = lane >> 2;
    const bool head_ok = gid < a.group;
    const int64_t qoff = (int64_t(b) * a.num_q_heads + int64_t(g) * a.group + (head_ok ? gid : 0)) * D;
#pragma unroll
    for (int kp = 0; kp < NKP; kp++) {
        const int col = bound_q_col<D>(4 * kp + t);
        if (QF32) {
            const uint4 *qp = reinterpret_cast<const uint4 *>(static_cast<const float *>(a.q) + qoff + col);
            qraw[kp][0] = qp[0];
            qraw[kp][QF32 ? 1 : 0] = qp[1];
        } else {
            qraw[kp][0] = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.q) + qoff + col);
        }
    }
}

// Logical pages (jj) and physical ids (pp) of this lane's four metadata rows
// among the warp's 32 pages from w_page0: rows gid, gid + 8 of group 0,
// then of group 1; vv: j < n_b.  The table row holds max_pages entries, so
// the ids can be read with n_b = max_pages before the sequence length is
// known (vv is then recomputed and the ids past the length are not used).
__device__ __forceinline__ void bound_page_ids(const SelectArgs &a, int b, int w_page0, int n_b, int (&jj)[4],
                                               int (&pp)[4], bool (&vv)[4]) {
    const int gid = (threadIdx.x & 31) >> 2;
    const int32_t *trow = a.page_table + int64_t(b) * a.max_pages;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        jj[i] = w_page0 + (i >> 1) * 16 + gid + (i & 1) * 8;
        vv[i] = jj[i] < n_b;
        pp[i] = vv[i] ? trow[jj[i]] : 0;
    }
}

// The lane's metadata chunks of its four rows (zero for absent or bad pages).
// The row of logical page fresh_j, just rewritten by this warp, is read
// through L2 (the read-only path may hold its previous contents).
template <int D, bool HINT>
__device__ __forceinline__ void bound_load_meta(const SelectArgs &a, int g, const int (&pp)[4], const bool (&vv)[4],
                                                bool (&bad)[4], uint4 (&av)[4][2 * D / 32], uint64_t policy,
                                                const int (&jj)[4], int fresh_j = -1) {
    constexpr int NKP = BoundScanRegs<D>::NKP;
    const int t = threadIdx.x & 3;
    const char *meta = static_cast<const char *>(a.meta);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        bad[i] = vv[i] && (pp[i] < 0 || pp[i] >= a.num_pool_pages);
        const char *rowp = meta + (int64_t(bad[i] ? 0 : pp[i]) * a.num_kv_heads + g) * (2 * D * 2);
        const bool fresh = jj[i] == fresh_j;
#pragma unroll
        for (int kp = 0; kp < NKP; kp++)
            av[i][kp] = !(vv[i] && !bad[i]) ? make_uint4(0, 0, 0, 0)
                        : fresh ? __ldcg(reinterpret_cast<const uint4 *>(rowp + (4 * kp + t) * 16))
                        : HINT  ? ldg_stream_v4_hint(rowp + (4 * kp + t) * 16, policy)
                                : ldg_stream_v4(rowp + (4 * kp + t) * 16);
    }
    if ((bad[0] || bad[1] || bad[2] || bad[3]) && t == 0) raise_error(a.flags, kErrPageId);
}

// Row scores of the warp's 32 pages: the bound of every head of the group as
// [m | M] . [q- | q+] on the tensor cores, the best head per page, stored to
// srow[j] (-inf for a bad page id).
template <int D, bool QF32>
__device__ __forceinline__ void bound_score_store(const SelectArgs &a, const uint4 (&qraw)[2 * D / 32][QF32 ? 2 : 1],
                                                  const uint4 (&av)[4][2 * D / 32], const int (&jj)[4],
                                                  const bool (&vv)[4], const bool (&bad)[4], int w_page0, int n_b,
                                                  float *srow) {
    constexpr int NKP = BoundScanRegs<D>::NKP;
    const int lane = threadIdx.x & 31, t = lane & 3, gid = lane >> 2;
    uint32_t bh[NKP][4], bl[NKP][4];
    bound_q_operand<D, QF32>(qraw, gid < a.group, bh, bl);
    const float NEG = -INFINITY;
#pragma unroll
    for (int grp = 0; grp < 2; grp++) {
        const int ia = 2 * grp, ib = 2 * grp + 1;
        if (w_page0 + grp * 16 >= n_b) break;  // warp-uniform: the group holds no page
        float sa, sb;
        bound_group_scores<D, QF32>(av[ia], av[ib], bh, bl, a.group, sa, sb);
        if (t == 0) {
            if (vv[ia]) srow[jj[ia]] = bad[ia] ? NEG : sa;
            if (vv[ib]) srow[jj[ib]] = bad[ib] ? NEG : sb;
        }
    }
}

// One CTA per (row, 128 pages) -- or, head-major (num_kv_heads a multiple of
// 4), per (sequence, 32 pages, 4 KV heads): warp w takes KV head 4 (x % Q) + w
// (Q = num_kv_heads / 4), so neighbouring CTAs read a page's metadata rows
// for all heads (contiguous in the [page][head] layout) at about the same
// time -- then the separate ranking kernel.  Three CTAs per SM (168
// registers): more metadata rows in flight per SM than at two, measured
// faster on GB300 despite a small spill.
// HINT: the metadata scan is larger than L2 and is read evict-first.
// REFRESH: first recompute the metadata of each row's last page from its
// valid key rows (TinyServe s5.3: the page the new token went into), with the
// warp that scores that page, which then scores it with the new rows.  The
// CTAs take a sequence's pages from the last one backwards, so the refreshing
// CTAs are among the first to run.
template <int D, bool QF32, bool HINT, bool REFRESH>
__global__ void __launch_bounds__(kScoreThreads, 3) score_mma_kernel(SelectArgs a, int score_all) {
    constexpr int NKP = BoundScanRegs<D>::NKP;
    const int warp = threadIdx.x >> 5;
    // The warp's row and pages follow from the block index alone, so the
    // sequence length, the query and the page ids (the table row holds
    // max_pages entries whatever the length) are requested together, and the
    // metadata right after: two dependent round trips per CTA.  REFRESH
    // counts the chunks back from max_pages, so a sequence's last chunk is its
    // first CTA with pages.
    int b, g, w_page0;  // w_page0: this warp's 32 pages (2 groups of 16)
    if (a.head_quads > 0) {
        b = blockIdx.y;
        g = (int(blockIdx.x) % a.head_quads) * 4 + warp;
        const int k = int(blockIdx.x) / a.head_quads, nk = int(gridDim.x) / a.head_quads;
        w_page0 = (REFRESH ? nk - 1 - k : k) * 32;
    } else {
        b = int(blockIdx.y) / a.num_kv_heads;
        g = int(blockIdx.y) % a.num_kv_heads;
        w_page0 = (REFRESH ? int(gridDim.x) - 1 - int(blockIdx.x) : int(blockIdx.x)) * kScoreThreads + warp * 32;
    }
    const int row = b * a.num_kv_heads + g;
    pdl_wait();
    int seq = a.seq_lens[b];
    uint4 qraw[NKP][QF32 ? 2 : 1];
    bound_load_q<D, QF32>(a, b, g, qraw);
    int jj[4], pp[4];
    bool vv[4], bad[4];
    bound_page_ids(a, b, w_page0, a.max_pages, jj, pp, vv);
    const int cap = a.max_pages * a.page_size;
    if (seq < 0 || seq > cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(a.flags, kErrSeqLen);
        seq = seq < 0 ? 0 : cap;
    }
    const int n_b = (seq + a.page_size - 1) / a.page_size;
#pragma unroll
    for (int i = 0; i < 4; i++) vv[i] = jj[i] < n_b;

    int fresh_j = -1;
    if (REFRESH && n_b > 0 && n_b - 1 >= w_page0 && n_b - 1 < w_page0 + 32) {
        fresh_j = n_b - 1;
        const int p = a.page_table[int64_t(b) * a.max_pages + fresh_j];
        if (p >= 0 && p < a.num_pool_pages)  // a bad id is flagged by the scan below
            meta_tile_warp<Bf16Ops, D * 2>(a.k_pool, a.meta_w, p, g, seq - fresh_j * a.page_size, a.num_kv_heads,
                                            a.page_size);
        __syncwarp();
    }
    float *srow = a.scores + int64_t(row) * a.max_pages;
    if (w_page0 >= n_b || (a.top_k >= n_b && !score_all)) return;

    uint4 av[4][NKP];
    bound_load_meta<D, HINT>(a, g, pp, vv, bad, av, HINT ? l2_evict_first_policy() : 0, jj, fresh_j);
    bound_score_store<D, QF32>(a, qraw, av, jj, vv, bad, w_page0, n_b, srow);
}

// -------------------------------------------------- scores on CUDA cores --
template <typename MT, bool QF32>
__global__ void __launch_bounds__(kScoreThreads) score_simt_kernel(SelectArgs a, int D, int score_all) {
    __shared__ float s_qp[8][128];
    __shared__ float s_qn[8][128];
    const RowInfo r = row_info(a);
    float *srow = a.scores + int64_t(r.row) * a.max_pages;
    const int j = blockIdx.x * kScoreThreads + threadIdx.x;
    const bool work = int(blockIdx.x) * kScoreThreads < r.n_b && (a.top_k < r.n_b || score_all);
    if (work) {
        for (int e = threadIdx.x; e < a.group * D; e += blockDim.x) {
            const int h = e / D, c = e % D;
            const int64_t qi = (int64_t(r.b) * a.num_q_heads + int64_t(r.g) * a.group + h) * D + c;
            const float v = QF32 ? static_cast<const float *>(a.q)[qi]
                                 : __bfloat162float(static_cast<const __nv_bfloat16 *>(a.q)[qi]);
            s_qp[h][c] = fmaxf(v, 0.f);
            s_qn[h][c] = fminf(v, 0.f);
        }
    }
    __syncthreads();
    if (work && j < r.n_b) {
        const int p = a.page_table[int64_t(r.b) * a.max_pages + j];
        if (p < 0 || p >= a.num_pool_pages) {
            raise_error(a.flags, kErrPageId);
            srow[j] = -INFINITY;
        } else {
            const MT *m = static_cast<const MT *>(a.meta) + (int64_t(p) * a.num_kv_heads + r.g) * 2 * D;
            const MT *M = m + D;
            float s[8];
#pragma unroll
            for (int h = 0; h < 8; h++) s[h] = 0.f;
            for (int c = 0; c < D; c++) {
                const float lo = float(m[c]), hi = float(M[c]);
#pragma unroll
                for (int h = 0; h < 8; h++)
                    if (h < a.group) s[h] = fmaf(s_qp[h][c], hi, fmaf(s_qn[h][c], lo, s[h]));
            }
            float best = -INFINITY;
#pragma unroll
            for (int h = 0; h < 8; h++)
                if (h < a.group) best = fmaxf(best, s[h]);
            srow[j] = best;
        }
    }
}

// ------------------------------------- Block Top-K scores (CUDA cores) --
// Vortex sparse-attention digest, method overview item 1: a page's score is
// q . centroid, the centroid being the page's mean key (fp32); with G query
// heads per KV head the row score is the best head's.  HBM-bound like the
// bound scorer (D fp32 per page, the same bytes as the bf16 [m | M] rows),
// so it runs on the CUDA cores.  Lanes span the D dims of one page row
// (coalesced), a warp takes 32 / G pages at a time so that the 32 (page,
// head) partial dot products of a batch are reduced with one butterfly
// reduce-scatter (31 shuffles; lane l ends with the total of (page l / G,
// head l % G)), then a max over each group of G lanes.
// HINT: the centroid scan is larger than L2 and is read evict-first.
template <int D, bool QF32, int G, bool HINT>
__global__ void __launch_bounds__(kScoreThreads) score_centroid_kernel(SelectArgs a, int score_all) {
    constexpr int VEC = D / 32;  // dims per lane
    constexpr int NPG = 32 / G;  // pages per batch
    const RowInfo r = row_info(a);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *srow = a.scores + int64_t(r.row) * a.max_pages;
    const int w_page0 = blockIdx.x * kScoreThreads + warp * 32;  // this warp's 32 pages
    if (w_page0 >= r.n_b || (a.top_k >= r.n_b && !score_all)) return;

    // q of the group's heads, this lane's dims
    float q[G][VEC];
    const int64_t q0 = (int64_t(r.b) * a.num_q_heads + int64_t(r.g) * G) * D + lane * VEC;
#pragma unroll
    for (int h = 0; h < G; h++) {
#pragma unroll
        for (int k = 0; k < VEC; k++) {
            const int64_t qi = q0 + int64_t(h) * D + k;
            q[h][k] = QF32 ? static_cast<const float *>(a.q)[qi]
                           : __bfloat162float(static_cast<const __nv_bfloat16 *>(a.q)[qi]);
        }
    }
    // page id of page w_page0 + lane (-1 past n_b, -2 when out of the pool)
    int pid = -1;
    if (w_page0 + lane < r.n_b) {
        pid = a.page_table[int64_t(r.b) * a.max_pages + w_page0 + lane];
        if (pid < 0 || pid >= a.num_pool_pages) {
            raise_error(a.flags, kErrPageId);
            pid = -2;
        }
    }
    const float *cent = static_cast<const float *>(a.meta);
    const uint64_t policy = HINT ? l2_evict_first_policy() : 0;
    for (int p0 = 0; p0 < 32 && w_page0 + p0 < r.n_b; p0 += NPG) {
        // loads of the batch's pages first
        float c[NPG][VEC];
#pragma unroll
        for (int k = 0; k < NPG; k++) {
            const int pk = __shfl_sync(0xffffffffu, pid, p0 + k);
            const float *row = cent + (int64_t(pk < 0 ? 0 : pk) * a.num_kv_heads + r.g) * D + lane * VEC;
            if (VEC == 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (pk >= 0) {
                    if constexpr (HINT) {
                        const uint4 u = ldg_stream_v4_hint(row, policy);
                        x = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                        __uint_as_float(u.w));
                    } else {
                        x = __ldg(reinterpret_cast<const float4 *>(row));
                    }
                }
                c[k][0] = x.x;
                c[k][VEC > 1 ? 1 : 0] = x.y;
                c[k][VEC > 2 ? 2 : 0] = x.z;
                c[k][VEC > 3 ? 3 : 0] = x.w;
            } else {
                float2 x = make_float2(0.f, 0.f);
                if (pk >= 0) {
                    if constexpr (HINT) {
                        const uint2 u = ldg_stream_v2_hint(row, policy);
                        x = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
                    } else {
                        x = __ldg(reinterpret_cast<const float2 *>(row));
                    }
                }
                c[k][0] = x.x;
                c[k][VEC > 1 ? 1 : 0] = x.y;
            }
        }
        // 32 partial dots: slot k * G + h
        float v[32];
#pragma unroll
        for (int sl = 0; sl < 32; sl++) {
            const int k = sl / G, h = sl % G;
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; e++) acc = fmaf(q[h][e], c[k][e], acc);
            v[sl] = acc;
        }
#pragma unroll
        for (int s = 16; s >= 1; s >>= 1) {
            const bool up = lane & s;
#pragma unroll
            for (int i = 0; i < s; i++) {
                const float send = up ? v[i] : v[i + s];
                const float keep = up ? v[i + s] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
            }
        }
        float best = v[0];  // lane l: (page p0 + l / G, head l % G)
#pragma unroll
        for (int off = 1; off < G; off <<= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, off));
        const int k = lane / G;
        const int j = w_page0 + p0 + k;
        const int pk = __shfl_sync(0xffffffffu, pid, (p0 + k) & 31);
        if (lane % G == 0 && j < r.n_b) srow[j] = pk == -2 ? -INFINITY : best;
    }
}

}  // namespace

cudaError_t launch_page_select_centroid(const SelectArgs &a, int q_dtype, int head_dim, cudaStream_t stream,
                                        int score_all) {
    const int64_t rows = int64_t(a.batch) * a.num_kv_heads;
    const dim3 grid(unsigned((a.max_pages + kScoreThreads - 1) / kScoreThreads), unsigned(rows));
    const dim3 block(kScoreThreads);
    const bool qf = q_dtype == kDtypeF32;
    // a centroid scan larger than L2 is read evict-first (see launch_decode)
    const int l2 = l2_cache_bytes();
    const bool hint = l2 > 0 && double(rows) * a.max_pages * head_dim * 4.0 > double(l2);
    cudaError_t e = cudaErrorInvalidValue;
    auto go = [&](auto d_tag, auto q_tag, auto h_tag) {
        constexpr int D = decltype(d_tag)::value;
        constexpr bool QF = decltype(q_tag)::value;
        constexpr bool H = decltype(h_tag)::value;
        switch (a.group) {
            case 1: e = launch_pdl(score_centroid_kernel<D, QF, 1, H>, grid, block, 0, stream, a, score_all); break;
            case 2: e = launch_pdl(score_centroid_kernel<D, QF, 2, H>, grid, block, 0, stream, a, score_all); break;
            case 4: e = launch_pdl(score_centroid_kernel<D, QF, 4, H>, grid, block, 0, stream, a, score_all); break;
            case 8: e = launch_pdl(score_centroid_kernel<D, QF, 8, H>, grid, block, 0, stream, a, score_all); break;
        }
    };
    auto go_h = [&](auto d_tag, auto q_tag) {
        hint ? go(d_tag, q_tag, std::true_type()) : go(d_tag, q_tag, std::false_type());
    };
    using I64 = std::integral_constant<int, 64>;
    using I128 = std::integral_constant<int, 128>;
    if (head_dim == 128)
        qf ? go_h(I128(), std::true_type()) : go_h(I128(), std::false_type());
    else
        qf ? go_h(I64(), std::true_type()) : go_h(I64(), std::false_type());
    if (e != cudaSuccess) return e;
    return launch_pdl(select_kernel, dim3(unsigned(rows)), dim3(kSelectThreads), 0, stream, a);
}

cudaError_t launch_page_select(const SelectArgs &a_in, int q_dtype, int meta_dtype, int head_dim,
                               cudaStream_t stream, int score_all, int refresh, int rank) {
    const int64_t rows = int64_t(a_in.batch) * a_in.num_kv_heads;
    // a metadata scan larger than L2 is read evict-first (see launch_decode)
    SelectArgs a = a_in;
    const int l2 = l2_cache_bytes();
    const double meta_bytes = double(rows) * a.max_pages * 2.0 * head_dim * (meta_dtype == kDtypeBf16 ? 2.0 : 4.0);
    a.meta_evict_first = l2 > 0 && meta_bytes > double(l2) ? 1 : 0;
    a.head_quads = meta_dtype == kDtypeBf16 && a.num_kv_heads % 4 == 0 ? a.num_kv_heads / 4 : 0;
    const dim3 grid = a.head_quads > 0
                          ? dim3(unsigned((a.max_pages + 31) / 32 * a.head_quads), unsigned(a.batch))
                          : dim3(unsigned((a.max_pages + kScoreThreads - 1) / kScoreThreads), unsigned(rows));
    const dim3 block(kScoreThreads);
    const bool qf = q_dtype == kDtypeF32;
    cudaError_t e = cudaErrorInvalidValue;
    if (meta_dtype == kDtypeBf16) {
        auto go = [&](auto d_tag, auto q_tag, auto h_tag, auto r_tag) {
            e = launch_pdl(score_mma_kernel<decltype(d_tag)::value, decltype(q_tag)::value, decltype(h_tag)::value,
                                            decltype(r_tag)::value>,
                           grid, block, 0, stream, a, score_all);
        };
        auto go_r = [&](auto d_tag, auto q_tag, auto h_tag) {
            refresh ? go(d_tag, q_tag, h_tag, std::true_type()) : go(d_tag, q_tag, h_tag, std::false_type());
        };
        auto go_h = [&](auto d_tag, auto q_tag) {
            a.meta_evict_first ? go_r(d_tag, q_tag, std::true_type()) : go_r(d_tag, q_tag, std::false_type());
        };
        using I64 = std::integral_constant<int, 64>;
        using I128 = std::integral_constant<int, 128>;
        if (head_dim == 128)
            qf ? go_h(I128(), std::true_type()) : go_h(I128(), std::false_type());
        else
            qf ? go_h(I64(), std::true_type()) : go_h(I64(), std::false_type());
    } else {
        e = qf ? launch_pdl(score_simt_kernel<float, true>, grid, block, 0, stream, a, head_dim, score_all)
               : launch_pdl(score_simt_kernel<float, false>, grid, block, 0, stream, a, head_dim, score_all);
    }
    if (e != cudaSuccess || !rank) return e;
    return launch_pdl(select_kernel, dim3(unsigned(rows)), dim3(kSelectThreads), 0, stream, a);
}

}  // namespace qskv

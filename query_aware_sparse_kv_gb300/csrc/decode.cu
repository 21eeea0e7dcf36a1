// Split-K sparse paged decode attention (the merge of split rows is in merge.cu).
//
// TinyServe query-aware page selection, s2.3 stages 3-4: only the selected
// pages are loaded from HBM and attention runs while they stream in; s3.1:
// later pages are prefetched while the current one is processed.  The split
// over workers and the merge of their partial results by log-sum-exp
// rescaling follow the Quail AI-SQL engine article (partial attention
// combined as in flash decoding) and CS336 Lecture 10 s9.2 (fused paged
// reads, FlashDecoding).
//
// Work decomposition.  A "unit" is one slot of one (sequence, KV head) row:
// row r has `slots_per_row` units (top_k, or max_pages for dense decode),
// unit r*slots + s names the s-th selected page of the row (empty past
// n_selected).  The units are cut into equal contiguous ranges, one per warp
// of a persistent grid, so every warp streams about the same number of pages
// whatever the row lengths.  A warp keeps an online softmax per query head of
// the group; at the end of each row it owns a piece of, it either writes the
// final output (it owns the whole row) or a normalised partial output with
// its log-sum-exp into slot (row + warp) of the workspace.  A second, small
// kernel merges the partials of the split rows.  Both are launched with
// programmatic dependent launch, so the merge kernel is resident and waiting
// when the decode grid drains.  No warp ever waits for another.
//
// bf16 KV (tensor cores).  Each warp runs its own pipeline of `stages`
// shared-memory buffers filled by 2-D TMA tiled loads (16 tokens x 64 dims
// per box, 128-byte swizzle) that complete on one mbarrier per buffer; lane 0
// issues, the whole warp consumes, and the buffer is refilled as soon as the
// warp is done with it.  Per 16-token sub-tile:
//   S^T (16 tokens x 8 heads) = K_tile . Q^T       mma.sync m16n8k16, K via ldmatrix
//   online softmax per head column (exp2, scale folded with log2 e)
//   P^T as the B operand: bf16 pack + movmatrix.trans of the S^T fragment
//   O^T (d x 8 heads)    += V_tile^T . P^T         V via ldmatrix.trans
// Query heads sit on the n = 8 axis (G <= 8), so per-head state lines up
// with the accumulator columns.  Token rows past seq_len are masked to -inf
// before the softmax and the matching V rows are zeroed in shared memory
// (0 * NaN would poison the product).  fp32 queries are split into hi + lo
// bf16 halves (two mma per k-step).  Probabilities are rounded to bf16 for
// the P.V product and the same rounded values feed the softmax denominator.
//
// fp32 KV runs a CUDA-core kernel with the same decomposition and merge.
#include <mutex>
#include <type_traits>

#include "qskv_device.cuh"
#include "qskv_internal.h"
#include "qskv_select.cuh"

namespace qskv {
namespace {

constexpr float kLn2 = 0.6931471805599453f;

// (physical page << 6 | valid tokens) of slot `slot` of row `row`, or -1
// when the slot is empty or names an out-of-range page (flagged).  The
// index loads that do not depend on each other are issued together.
// pt_row: the sequence's page-table row (global memory, or a copy in shared
// memory).
__device__ __forceinline__ int unit_code(const DecodeArgs &a, int row, int slot, const int32_t *pt_row = nullptr) {
    const int b = row / a.num_kv_heads;
    int seq = __ldg(a.seq_lens + b);
    int ns = 0, j = slot + a.page_begin;
    if (a.selected) {
        ns = __ldg(a.n_selected + row);
        j = __ldg(a.selected + int64_t(row) * a.top_k + slot);
    }
    const int cap = a.max_pages * a.page_size;
    if (seq < 0 || seq > cap) {
        raise_error(a.flags, kErrSeqLen);
        seq = seq < 0 ? 0 : cap;
    }
    const int n_b = (seq + a.page_size - 1) / a.page_size;
    if (a.selected) {
        const int lim = min(a.top_k, n_b);
        if (ns < 0 || ns > lim) {
            raise_error(a.flags, kErrSelected);
            ns = max(0, min(ns, lim));
        }
        if (slot >= ns) return -1;
        if (j < 0 || j >= n_b) {
            raise_error(a.flags, kErrSelected);
            return -1;
        }
    } else if (j >= n_b) {
        return -1;
    }
    const int p = pt_row ? pt_row[j] : __ldg(a.page_table + int64_t(b) * a.max_pages + j);
    if (p < 0 || p >= a.num_pool_pages) {
        raise_error(a.flags, kErrPageId);
        return -1;
    }
    return (p << 6) | min(a.page_size, seq - j * a.page_size);
}

// Code of logical page j of row `row` (a selected index the caller did not
// pass: the fused rank + decode), with unit_code's checks; seq: the row's
// sequence length as read from seq_lens.
__device__ __forceinline__ int page_code(const DecodeArgs &a, int row, int j, const int32_t *pt_row, int seq) {
    const int b = row / a.num_kv_heads;
    const int cap = a.max_pages * a.page_size;
    seq = seq < 0 ? 0 : (seq > cap ? cap : seq);  // flagged by the scoring kernel
    const int n_b = (seq + a.page_size - 1) / a.page_size;
    if (j < 0 || j >= n_b) return -1;
    const int p = pt_row ? pt_row[j] : __ldg(a.page_table + int64_t(b) * a.max_pages + j);
    if (p < 0 || p >= a.num_pool_pages) {
        raise_error(a.flags, kErrPageId);
        return -1;
    }
    return (p << 6) | min(a.page_size, seq - j * a.page_size);
}

// Code of unit (row, slot) + lane offset `k` (0 <= k < 64), -1 past u_end.
__device__ __forceinline__ int unit_code_at(const DecodeArgs &a, int row, int slot, int k, int64_t u, int64_t u_end) {
    if (u + k >= u_end) return -1;
    const int s = slot + k;
    const int dr = s / a.slots_per_row;
    return unit_code(a, row + dr, s - dr * a.slots_per_row);
}

// ------------------------------------------------- bf16 KV, tensor cores --
// Pieces of rows a warp's range touches but that hold no sub-tile for it:
// an empty contribution (lse = -inf), or the final empty answer when the
// warp owns the row alone.
template <int D>
__device__ void write_empty_piece(const DecodeArgs &a, int row, int64_t gw) {
    const int lane = threadIdx.x & 31;
    const int G = a.group;
    int64_t w0, w1;
    row_warps(a, row, w0, w1);
    if (row_is_final(a, w0, w1)) {
        const int b = row / a.num_kv_heads, g = row % a.num_kv_heads;
        const int64_t qh0 = int64_t(b) * a.num_q_heads + int64_t(g) * G;
        for (int i = lane; i < G * D; i += 32) a.out[qh0 * D + i] = 0.f;
        if (a.lse && lane < G) a.lse[qh0 + lane] = -INFINITY;
    } else if (lane < G) {
        a.part_lse[(row + gw) * G + lane] = -INFINITY;
    }
}

// Folds the pieces of split row `row` (slots row + w0 .. row + w1) into its
// final output, with one warp (used when the pieces fit one round of loads,
// kFoldMaxLoads): out = sum_w 2^(lse_w - m) o_w / sum_w 2^(lse_w - m),
// m = max_w lse_w (log2 domain), exactly as the merge kernel.  Lane l folds
// columns l, l + 32, ... of the row's G x D/4 float4 columns (CPL per lane),
// BATCH pieces' loads in flight at a time.  Pieces are read from L2.
template <int D, int G>
__device__ void fold_row_warp(const DecodeArgs &a, int row, int64_t w0, int64_t w1) {
    constexpr int V4 = D / 4;
    constexpr int COLS = G * V4;
    constexpr int CPL = COLS >= 32 ? COLS / 32 : 1;
    constexpr int BATCH = 16 / CPL;
    const int lane = threadIdx.x & 31;
    if (COLS < 32 && lane >= COLS) return;
    // pieces: the decode warps' (slots row + w0 ..) then another kernel's
    // extra pieces (slots extra_slot0 + row * extra_pieces ..)
    const int nd = int(w1 - w0 + 1);
    const int n = nd + a.extra_pieces;
    const int64_t slot0 = row + w0, eslot0 = a.extra_slot0 + int64_t(row) * a.extra_pieces;
    const float4 *o_all = reinterpret_cast<const float4 *>(a.part_o);
    float mx[CPL], den[CPL];
    float4 acc[CPL];
#pragma unroll
    for (int j = 0; j < CPL; j++) {
        mx[j] = -INFINITY;
        den[j] = 0.f;
        acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int p0 = 0; p0 < n; p0 += BATCH) {
        float l[BATCH][CPL];
        float4 v[BATCH][CPL];
#pragma unroll
        for (int k = 0; k < BATCH; k++)
#pragma unroll
            for (int j = 0; j < CPL; j++) {
                const int c = lane + 32 * j;
                const bool ok = p0 + k < n;
                const int64_t s = p0 + k < nd ? slot0 + p0 + k : eslot0 + (p0 + k - nd);
                l[k][j] = ok ? __ldcg(a.part_lse + s * G + c / V4) : -INFINITY;
                v[k][j] = ok ? __ldcg(o_all + s * COLS + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
        for (int j = 0; j < CPL; j++) {
            float m = mx[j];
#pragma unroll
            for (int k = 0; k < BATCH; k++) m = fmaxf(m, l[k][j]);
            if (m == -INFINITY) continue;
            const float sc = exp2f(mx[j] - m);
            den[j] *= sc;
            acc[j].x *= sc;
            acc[j].y *= sc;
            acc[j].z *= sc;
            acc[j].w *= sc;
#pragma unroll
            for (int k = 0; k < BATCH; k++) {
                if (l[k][j] == -INFINITY) continue;  // an empty piece: its o holds no data
                const float w = exp2f(l[k][j] - m);
                den[j] += w;
                acc[j].x = fmaf(w, v[k][j].x, acc[j].x);
                acc[j].y = fmaf(w, v[k][j].y, acc[j].y);
                acc[j].z = fmaf(w, v[k][j].z, acc[j].z);
                acc[j].w = fmaf(w, v[k][j].w, acc[j].w);
            }
            mx[j] = m;
        }
    }
    const int b = row / a.num_kv_heads, g = row % a.num_kv_heads;
    const int64_t qh0 = int64_t(b) * a.num_q_heads + int64_t(g) * G;
#pragma unroll
    for (int j = 0; j < CPL; j++) {
        const int c = lane + 32 * j, h = c / V4, c4 = c % V4;
        const float inv = den[j] > 0.f ? 1.f / den[j] : 0.f;
        reinterpret_cast<float4 *>(a.out + (qh0 + h) * D)[c4] =
            make_float4(acc[j].x * inv, acc[j].y * inv, acc[j].z * inv, acc[j].w * inv);
        if (c4 == 0 && a.lse) a.lse[qh0 + h] = den[j] > 0.f ? (mx[j] + log2f(den[j])) * kLn2 : -INFINITY;
    }
}

// Ends a warp's work when the call folds split rows itself (no merge
// kernel): the warp's pieces are made visible device-wide, then the warp
// takes a ticket on each row it shares with other warps (only the first and
// the last row of its range can be shared); the warp drawing a row's last
// ticket has every other piece of the row visible and folds the row, then
// resets the row's counter for the next call.  No warp waits for another.
template <int D>
__device__ void fold_shared_rows(const DecodeArgs &a, int row_first, int row_last) {
    const int lane = threadIdx.x & 31;
    __threadfence();  // this lane's piece stores, before the tickets
    __syncwarp();
    for (int row = row_first; row <= row_last; row++) {
        int64_t w0, w1;
        row_warps(a, row, w0, w1);
        if (row_is_final(a, w0, w1)) continue;  // this warp wrote the row's output itself
        if (w0 < w1) {  // shared with other decode warps: the last ticket folds
            uint32_t last = 0;
            if (lane == 0) {
                last = atomicAdd(a.tickets + row, 1u) == uint32_t(w1 - w0) ? 1u : 0u;
                if (last) __threadfence();  // the other warps' pieces, before they are read
            }
            if (!__shfl_sync(0xffffffffu, last, 0)) continue;
        }
        switch (a.group) {
            case 1: fold_row_warp<D, 1>(a, row, w0, w1); break;
            case 2: fold_row_warp<D, 2>(a, row, w0, w1); break;
            case 4: fold_row_warp<D, 4>(a, row, w0, w1); break;
            default: fold_row_warp<D, 8>(a, row, w0, w1); break;
        }
        __syncwarp();
        if (lane == 0 && w0 < w1) a.tickets[row] = 0u;
    }
}

// Fused scoring (TinyServe query-aware page selection, s2.2-2.3: the bound
// score of every page from its metadata; s5.3: the last page's metadata is
// recomputed first).  Block `blk` of the k CTAs of row `row` scores the
// row's 16-page groups [blk ng / k, (blk + 1) ng / k).  `stage` (stage_bytes
// of shared memory) takes the page ids and metadata rows of as many groups
// at a time as fit (the host takes this path only when one round covers a
// CTA's share): the ids first (one coalesced pass, unless the table row is
// already in shared memory), then the rows by
// 16-byte copies through L2 (consecutive threads copy consecutive chunks of
// a row; chunk c of slot s sits at c ^ (s & 7), so the eight rows one
// fragment load touches fall in different banks); each warp then scores
// whole groups with bound_group_scores (the scoring kernel's product, in the
// same order: equal bits) and stores them to the row's scores.  The last
// page's metadata is recomputed by warp 0 of the CTA holding it while the
// other pages' copies are in flight, and written both to meta and straight
// into its staging slot (not copied).
template <int D, bool QF32, int WPC>
__device__ void score_row_share(const DecodeArgs &a, int row, int blk, int k, int seq, int n_b, uint8_t *stage,
                                size_t stage_bytes, const int32_t *pt_row, bool pt_in_smem, const void *s_q) {
    constexpr int NKP = BoundScanRegs<D>::NKP;
    constexpr int ROWB = 4 * D;        // bytes of one bf16 metadata row [m | M]
    constexpr int CPRW = ROWB / 16;    // its 16-byte chunks
    constexpr int NT = WPC * 32;
    const int cap_groups = int(stage_bytes / (16 * (ROWB + 4)));
    int32_t *s_ids = reinterpret_cast<int32_t *>(stage + size_t(cap_groups) * 16 * ROWB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = lane & 3, gid = lane >> 2;
    const int g = row % a.num_kv_heads;
    const int ng = (n_b + 15) >> 4;
    const int g0 = int(int64_t(blk) * ng / k), g1 = int(int64_t(blk + 1) * ng / k);
    const char *meta = static_cast<const char *>(a.meta);
    // the last page (its metadata recomputed here: the CTA holding the last group)
    const int fresh_j = a.refresh && n_b > 0 && blk == k - 1 ? n_b - 1 : -1;
    const int fresh_p = fresh_j >= 0 ? pt_row[fresh_j] : -1;
    const bool fresh_ok = fresh_p >= 0 && fresh_p < a.num_pool_pages;  // a bad id is flagged by the scan
    if (!(a.top_k < n_b || a.score_all)) {  // CTA-uniform: every page is kept, no score asked for
        if (fresh_ok && warp == 0)
            meta_tile_warp<Bf16Ops, D * 2>(a.k_pool, a.meta_w, fresh_p, g, seq - fresh_j * a.page_size,
                                            a.num_kv_heads, a.page_size);
        return;
    }

    uint32_t bh[NKP][4], bl[NKP][4];
    {
        uint4 qraw[NKP][QF32 ? 2 : 1];
        const bool head_ok = gid < a.group;
        const uint8_t *qh = static_cast<const uint8_t *>(s_q) + (head_ok ? gid : 0) * D * (QF32 ? 4 : 2);
#pragma unroll
        for (int kp = 0; kp < NKP; kp++) {
            const int col = bound_q_col<D>(4 * kp + t);
            if (QF32) {
                qraw[kp][0] = *reinterpret_cast<const uint4 *>(qh + col * 4);
                qraw[kp][QF32 ? 1 : 0] = *reinterpret_cast<const uint4 *>(qh + col * 4 + 16);
            } else {
                qraw[kp][0] = *reinterpret_cast<const uint4 *>(qh + col * 2);
            }
        }
        bound_q_operand<D, QF32>(qraw, head_ok, bh, bl);
    }
    float *srow = a.scores + int64_t(row) * a.max_pages;
    const float NEG = -INFINITY;
    for (int rg = g0; rg < g1; rg += cap_groups) {
        const int ngr = min(cap_groups, g1 - rg);
        const int j0 = rg * 16;
        // the round's page ids: the staged table row itself, else a copy
        const int32_t *ids = s_ids;
        if (pt_in_smem) {
            ids = pt_row + j0;
        } else {
            for (int sl = threadIdx.x; sl < ngr * 16; sl += NT) s_ids[sl] = j0 + sl < n_b ? pt_row[j0 + sl] : -1;
            __syncthreads();
        }
        for (int i = threadIdx.x; i < ngr * 16 * CPRW; i += NT) {
            const int sl = i / CPRW, c = i % CPRW;
            const int j = j0 + sl;
            if (j < n_b && j != fresh_j) {
                const int p = ids[sl];
                if (p >= 0 && p < a.num_pool_pages)
                    cp_async_cg16(stage + sl * ROWB + ((c ^ (sl & 7)) << 4),
                                  meta + (int64_t(p) * a.num_kv_heads + g) * ROWB + c * 16);
            }
        }
        if (fresh_ok && warp == 0 && fresh_j >= j0 && fresh_j < j0 + ngr * 16) {
            const int sl = fresh_j - j0;
            meta_tile_warp<Bf16Ops, D * 2, true>(a.k_pool, a.meta_w, fresh_p, g, seq - fresh_j * a.page_size,
                                                  a.num_kv_heads, a.page_size, stage + sl * ROWB, sl & 7);
        }
        cp_async_wait_all();
        __syncthreads();
        for (int gi = warp; gi < ngr; gi += WPC) {
            const int sa_ = gi * 16 + gid, sb_ = sa_ + 8;  // both = gid (mod 8)
            const int ja = j0 + sa_, jb = j0 + sb_;
            const bool va = ja < n_b, vb = jb < n_b;
            const int pa = va ? ids[sa_] : 0, pb = vb ? ids[sb_] : 0;
            const bool bada = va && (pa < 0 || pa >= a.num_pool_pages);
            const bool badb = vb && (pb < 0 || pb >= a.num_pool_pages);
            if ((bada || badb) && t == 0) raise_error(a.flags, kErrPageId);
            uint4 xa[NKP], xb[NKP];
#pragma unroll
            for (int kp = 0; kp < NKP; kp++) {
                const int c = 4 * kp + t;
                const uint4 z = make_uint4(0, 0, 0, 0);
                xa[kp] = va && !bada ? *reinterpret_cast<const uint4 *>(stage + sa_ * ROWB + ((c ^ gid) << 4)) : z;
                xb[kp] = vb && !badb ? *reinterpret_cast<const uint4 *>(stage + sb_ * ROWB + ((c ^ gid) << 4)) : z;
            }
            float sa, sb;
            bound_group_scores<D, QF32>(xa, xb, bh, bl, a.group, sa, sb);
            if (t == 0) {
                if (va) srow[ja] = bada ? NEG : sa;
                if (vb) srow[jb] = badb ? NEG : sb;
            }
        }
        // the stage is read before the next round reuses it (after the last
        // round, the caller's CTA or cluster barrier comes first)
        if (rg + cap_groups < g1) __syncthreads();
    }
}

// A stage holds up to HALVES 16-token sub-tiles ("halves") of one row: K
// then V, each half as D/64 boxes of 16 tokens x 64 dims (128-byte swizzle).
// HINT: the call streams more K/V than L2 holds; the loads carry an
// evict-first L2 policy.
// ROWCTA: the row_blocks (k <= kRowBlocksMax) CTAs c = k r .. k r + k - 1 decode row r alone
// (used when the rows fit one wave of CTAs: k = 1 with one or two rows per
// SM, k > 1 with fewer rows than SMs).  A CTA first reads the row's unit
// codes into shared memory; warp w of block j then takes units j + k (w + WPC
// n), n = 0, 1, ... (a fixed split, so repeated calls give bit-identical
// results; with k = 1 a shared counter handing units out in arrival order
// measured 1.3 % faster and is not deterministic).  Each warp leaves its
// piece in its own ring and, after a CTA barrier, the CTA folds the pieces:
// with k = 1 into the row's output (no global partials, no merge kernel);
// with k > 1 into one piece per block in the workspace, and the block that
// draws the row's last ticket (a per-row counter; no block waits for
// another) folds the k pieces with all its threads and resets the counter.
template <int D, bool QF32, int WPC, int HALVES, bool HINT, bool ROWCTA, bool RANK = false, bool SCORE = false>
__global__ void __launch_bounds__(WPC * 32, kDecodeCtasPerSm)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                       DecodeArgs a) {
    static_assert(HALVES == 1 || HALVES == 2, "a stage holds one or two 16-token halves");
    constexpr int NB = D / 64;            // 64-dim boxes per token row
    constexpr int BOX = 16 * 128;         // bytes of one box: 16 tokens x 128 B
    constexpr int HALF = NB * BOX;        // K (or V) bytes of one 16-token sub-tile
    constexpr int KVB = HALVES * HALF;    // K (or V) bytes of a stage
    constexpr int STAGE = 2 * KVB;
    constexpr int NKS = D / 16;           // k-steps of Q.K^T, m-tiles of P.V
    constexpr float kLazy = 8.f;          // rescale only when a head's max grows by > 2^8

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[WPC][kMaxStages];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = lane & 3, gid = lane >> 2;
    const int S = a.stages;
    const int G = a.group;
    const int64_t gw = int64_t(blockIdx.x) * WPC + warp;
    const int rc_k = ROWCTA ? a.row_blocks : 1;
    const int rc_row = ROWCTA ? int(blockIdx.x) / rc_k : 0, rc_blk = ROWCTA ? int(blockIdx.x) % rc_k : 0;
    const int64_t u_begin = ROWCTA ? int64_t(rc_row) * a.slots_per_row : gw * a.units_per_warp;
    const int64_t u_end = ROWCTA ? u_begin + a.slots_per_row : min(u_begin + a.units_per_warp, a.total_units);
    pdl_trigger();
    if (!ROWCTA && u_begin >= u_end) {
        if (a.wait_at_exit) pdl_wait();
        return;
    }

    uint8_t *ring0 = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = ring0 + size_t(warp) * S * STAGE;
    int *s_code = reinterpret_cast<int *>(ring0 + size_t(WPC) * S * STAGE);  // ROWCTA: [slots_per_row]
    int32_t *s_pt = s_code + ((a.slots_per_row + 3) & ~3);                   // ROWCTA: [max_pages] if staged
    uint4 *s_q = reinterpret_cast<uint4 *>(s_pt + (a.pt_in_smem ? ((a.max_pages + 3) & ~3) : 0));  // ROWCTA: [G][D]
    uint64_t *bar = bars[warp];
    if (lane == 0) {
        for (int s = 0; s < S; s++) mbar_init(bar + s, 1);
        mbar_fence_init();
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    __syncwarp();
    if constexpr (ROWCTA) {
        // The page table is an input no kernel of this library writes, so the
        // row's entries are staged before the wait for the previous kernel
        // (which ends the selection), leaving one dependent round trip
        // (selected -> code) after it.
        if (a.pt_in_smem) {
            const int32_t *pt = a.page_table + int64_t(rc_row / a.num_kv_heads) * a.max_pages;
            for (int j = threadIdx.x; j < a.max_pages; j += WPC * 32) s_pt[j] = __ldg(pt + j);
        }
        // the group's G query rows (contiguous), once per CTA in 16-byte
        // vectors (q may sit in host memory: few, whole-line requests)
        constexpr int QV = D * (QF32 ? 4 : 2) / 16;  // uint4 per query row
        const uint4 *qg = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(a.q) +
                          (int64_t(rc_row / a.num_kv_heads) * a.num_q_heads + int64_t(rc_row % a.num_kv_heads) * G) *
                              D * (QF32 ? 4 : 2));
        for (int i = threadIdx.x; i < G * QV; i += WPC * 32) s_q[i] = qg[i];
    }
    // the row's sequence length (an input too), for the fused rank / score
    const int rc_seq = ROWCTA && RANK ? __ldg(a.seq_lens + rc_row / a.num_kv_heads) : 0;
    if (!a.wait_at_exit) pdl_wait();
    if constexpr (ROWCTA) {
        __syncthreads();
        if constexpr (RANK) {
            // Fused rank + decode: the CTA ranks its row's scores first (the
            // ranking kernel's routine; keys in the ring's memory, the list in
            // s_code), then turns each selected page into its code in place.
            __shared__ uint32_t r_hist[256], r_mm[2 * WPC];
            __shared__ int r_tmp[2 * WPC], r_pick[3];
            const SelectSmem sm{reinterpret_cast<uint32_t *>(ring0), r_hist, r_mm, r_tmp, r_pick};
            SelectArgs sa{};
            sa.selected = a.selected_out;
            sa.n_selected = a.n_selected_out;
            sa.top_k = a.top_k;
            sa.need_max = 0;
            sa.seed = 0;
            const int b = rc_row / a.num_kv_heads;
            int seq = rc_seq;
            const int cap = a.max_pages * a.page_size;
            if (SCORE && (seq < 0 || seq > cap) && threadIdx.x == 0 && rc_blk == 0) raise_error(a.flags, kErrSeqLen);
            seq = seq < 0 ? 0 : (seq > cap ? cap : seq);  // flagged by the scoring kernel (or above)
            const int n_b = (seq + a.page_size - 1) / a.page_size;
            if constexpr (SCORE) {
                // the CTA's share of the row's scores, staged through the
                // rings' memory; then every CTA of the row (cluster) sees all
                score_row_share<D, QF32, WPC>(a, rc_row, rc_blk, rc_k, seq, n_b, ring0, size_t(WPC) * S * STAGE,
                                              a.pt_in_smem ? s_pt : a.page_table + int64_t(b) * a.max_pages,
                                              a.pt_in_smem != 0, s_q);
                if (rc_k > 1)
                    cluster_sync();
                else
                    __syncthreads();
            }
            const int nsel = select_row<WPC * 32>(sa, rc_row, n_b, a.scores + int64_t(rc_row) * a.max_pages, sm,
                                                  s_code, rc_blk == 0);
            fence_proxy_async_smem();  // the keys' stores, before TMA refills of the same memory
            __syncthreads();
            for (int i = threadIdx.x; i < a.slots_per_row; i += WPC * 32)
                s_code[i] = i < nsel ? page_code(a, rc_row, s_code[i], a.pt_in_smem ? s_pt : nullptr, rc_seq) : -1;
        } else {
            for (int i = threadIdx.x; i < a.slots_per_row; i += WPC * 32)
                s_code[i] = unit_code(a, rc_row, i, a.pt_in_smem ? s_pt : nullptr);
        }
        __syncthreads();
    }
    // K/V streams larger than L2 are read evict-first; smaller ones with no
    // hint (a hint with the normal policy, or a branch on the choice in the
    // issue path, measured slower than plain loads)
    const uint64_t kv_policy = HINT ? l2_evict_first_policy() : 0;
    auto load_kv = [&](void *dst, const CUtensorMap *map, int x, int y, uint64_t *b) {
        if constexpr (HINT)
            tma_load_2d_hint(dst, map, x, y, b, kv_policy);
        else
            tma_load_2d(dst, map, x, y, b);
    };

    // Units are walked with (row, slot) cursors, never by dividing the
    // 64-bit unit index in the loop.
    const int spr = a.slots_per_row;
    const int row_begin = int(u_begin / spr);
    const int slot_begin = int(u_begin - int64_t(row_begin) * spr);
    const int row_last = int((u_end - 1) / spr);

    // Codes of units [wbase, wbase + 64): lane i holds units wbase+i and
    // wbase+32+i; (wrow, wslot) are the coordinates of wbase.  Only the
    // producer reads them; it slides the window.
    int64_t wbase = u_begin;
    int wrow = row_begin, wslot = slot_begin;
    int code_cur = ROWCTA ? -1 : unit_code_at(a, wrow, wslot, lane, wbase, u_end);
    int code_nxt = ROWCTA ? -1 : unit_code_at(a, wrow, wslot, 32 + lane, wbase, u_end);
    auto code_of = [&](int64_t u) -> int {
        const int k = int(u - wbase);
        const int c0 = __shfl_sync(0xffffffffu, code_cur, k & 31);
        const int c1 = __shfl_sync(0xffffffffu, code_nxt, k & 31);
        return k < 32 ? c0 : c1;
    };

    // ---------------- producer: fills a stage with the next one or two
    // sub-tiles of one row; lane s remembers stage s's row and valid counts.
    int64_t pu = u_begin;
    int prow = row_begin, pslot = slot_begin, pg = row_begin % a.num_kv_heads;
    int psub = 0, ps = 0;
    uint32_t issued = 0, consumed = 0;
    int st_row = 0, st_valid = 0;  // lane s: stage s's row; valid tokens half0 | half1 << 8
    auto advance_sub = [&](int nsub) {
        if (++psub >= nsub) {
            psub = 0;
            pu++;
            if (++pslot == spr) {
                pslot = 0;
                prow++;
                if (++pg == a.num_kv_heads) pg = 0;
            }
        }
    };
    int rc_code = -1;       // ROWCTA: code of the unit being issued
    int rc_taken = 0;       // ROWCTA: units this warp has taken
    bool rc_done = false;   // ROWCTA: the warp's units are all issued
    auto produce = [&]() {
        while (int(issued - consumed) < S) {
            int nh = 0, srow = -1, v0 = 0, v1 = 0, y0 = 0, y1 = 0;
            if constexpr (ROWCTA) {
                while (nh < HALVES && !rc_done) {
                    if (psub == 0) {  // the warp's next unit: slots warp, warp + WPC, ...
                        const int idx = rc_blk + rc_k * (rc_taken * WPC + warp);
                        rc_taken++;
                        if (idx >= spr) {
                            rc_done = true;
                            break;
                        }
                        rc_code = s_code[idx];
                        if (rc_code < 0) continue;  // an empty slot
                    }
                    srow = prow;
                    const int valid = rc_code & 63, phys = rc_code >> 6;
                    const int v = min(16, valid - psub * 16);
                    const int y = (phys * a.num_kv_heads + pg) * a.page_size + psub * 16;
                    if (nh == 0) {
                        v0 = v;
                        y0 = y;
                    } else {
                        v1 = v;
                        y1 = y;
                    }
                    nh++;
                    if (++psub >= ((valid + 15) >> 4)) psub = 0;
                }
            }
            while (!ROWCTA && nh < HALVES && pu < u_end) {
                if (pu - wbase >= 32) {  // slide the code window by 32 units
                    wbase += 32;
                    wslot += 32;
                    while (wslot >= spr) {
                        wslot -= spr;
                        wrow++;
                    }
                    code_cur = code_nxt;
                    code_nxt = unit_code_at(a, wrow, wslot, 32 + lane, wbase, u_end);
                }
                const int code = code_of(pu);
                if (code < 0) {
                    advance_sub(0);
                    continue;
                }
                if (nh > 0 && prow != srow) break;  // a stage never spans two rows
                srow = prow;
                const int valid = code & 63, phys = code >> 6;
                const int v = min(16, valid - psub * 16);
                const int y = (phys * a.num_kv_heads + pg) * a.page_size + psub * 16;
                if (nh == 0) {
                    v0 = v;
                    y0 = y;
                } else {
                    v1 = v;
                    y1 = y;
                }
                nh++;
                advance_sub((valid + 15) >> 4);
            }
            if (nh == 0) break;
            if (lane == 0) {
                uint8_t *st = ring + size_t(ps) * STAGE;
                mbar_arrive_expect_tx(bar + ps, uint32_t(nh) * 2 * HALF);
#pragma unroll
                for (int nb = 0; nb < NB; nb++) {
                    load_kv(st + nb * BOX, &tmap_k, nb * 64, y0, bar + ps);
                    load_kv(st + KVB + nb * BOX, &tmap_v, nb * 64, y0, bar + ps);
                }
                if (HALVES == 2 && nh == 2) {
#pragma unroll
                    for (int nb = 0; nb < NB; nb++) {
                        load_kv(st + HALF + nb * BOX, &tmap_k, nb * 64, y1, bar + ps);
                        load_kv(st + KVB + HALF + nb * BOX, &tmap_v, nb * 64, y1, bar + ps);
                    }
                }
            }
            if (lane == ps) {
                st_row = srow;
                st_valid = v0 | (v1 << 8);
            }
            issued++;
            ps = ps + 1 == S ? 0 : ps + 1;
        }
    };

    // ---------------- consumer state (per row)
    int cur_row = -1;
    float o[NKS][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2t, 2t+1
    uint32_t qb[NKS][2], ql[NKS][2];

    auto start_row = [&](int row) {
        const int b = row / a.num_kv_heads, g = row % a.num_kv_heads;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
#pragma unroll
        for (int i = 0; i < NKS; i++) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        const bool ok = gid < G;
        // ROWCTA: the group's queries were staged in shared memory (s_q)
        const void *qbase = ROWCTA ? static_cast<const void *>(s_q) : a.q;
        const int64_t qoff = ROWCTA ? int64_t(ok ? gid : 0) * D
                                    : (int64_t(b) * a.num_q_heads + int64_t(g) * G + (ok ? gid : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < NKS; ks++) {
            const int k0 = ks * 16 + 2 * t;
            if (QF32) {
                const float *q = static_cast<const float *>(qbase) + qoff;
                const float2 x0 = *reinterpret_cast<const float2 *>(q + k0);
                const float2 x1 = *reinterpret_cast<const float2 *>(q + k0 + 8);
                const uint32_t h0 = pack_bf16x2(x0.x, x0.y), h1 = pack_bf16x2(x1.x, x1.y);
                qb[ks][0] = ok ? h0 : 0u;
                qb[ks][1] = ok ? h1 : 0u;
                ql[ks][0] = ok ? pack_bf16x2(x0.x - bf16_lo_to_float(h0), x0.y - bf16_hi_to_float(h0)) : 0u;
                ql[ks][1] = ok ? pack_bf16x2(x1.x - bf16_lo_to_float(h1), x1.y - bf16_hi_to_float(h1)) : 0u;
            } else {
                const uint32_t *q = reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(qbase) + qoff);
                qb[ks][0] = ok ? q[k0 / 2] : 0u;
                qb[ks][1] = ok ? q[(k0 + 8) / 2] : 0u;
            }
        }
    };

    auto finish_row = [&](int row) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
        const float e0 = l0 > 0.f ? m0 + log2f(l0) : -INFINITY, e1 = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
        const int h0 = 2 * t, h1 = 2 * t + 1;
        int64_t w0, w1;
        row_warps(a, row, w0, w1);
        float *dst;
        if (row_is_final(a, w0, w1)) {
            const int b = row / a.num_kv_heads, g = row % a.num_kv_heads;
            const int64_t qh = int64_t(b) * a.num_q_heads + int64_t(g) * G;
            dst = a.out + qh * D;
            if (a.lse && gid == 0) {
                if (h0 < G) a.lse[qh + h0] = e0 * kLn2;
                if (h1 < G) a.lse[qh + h1] = e1 * kLn2;
            }
        } else {
            const int64_t slot = row + gw;
            dst = a.part_o + slot * G * D;
            if (gid == 0) {
                if (h0 < G) a.part_lse[slot * G + h0] = e0;
                if (h1 < G) a.part_lse[slot * G + h1] = e1;
            }
        }
#pragma unroll
        for (int mt = 0; mt < NKS; mt++) {
            const int d0 = mt * 16 + gid;
            if (h0 < G) {
                dst[h0 * D + d0] = o[mt][0] * i0;
                dst[h0 * D + d0 + 8] = o[mt][2] * i0;
            }
            if (h1 < G) {
                dst[h1 * D + d0] = o[mt][1] * i1;
                dst[h1 * D + d0 + 8] = o[mt][3] * i1;
            }
        }
    };

    // Q.K^T of NH halves (tokens gid / gid+8 x heads 2t / 2t+1), masked.
    // Every ldmatrix of a half is issued before its first mma, and the
    // mma land on four accumulators in turn (short dependency chains).
    constexpr int NCH = 4;
    auto mask_scale = [&](const float (&sa)[NCH][4], int valid, float (&s)[4]) {
        const float sc = a.scale_log2;
        float x[4];
#pragma unroll
        for (int i = 0; i < 4; i++) x[i] = (sa[0][i] + sa[1][i]) + (sa[2][i] + sa[3][i]);
        s[0] = gid < valid ? x[0] * sc : -INFINITY;
        s[1] = gid < valid ? x[1] * sc : -INFINITY;
        s[2] = gid + 8 < valid ? x[2] * sc : -INFINITY;
        s[3] = gid + 8 < valid ? x[3] * sc : -INFINITY;
    };
    auto qk = [&](auto nh_tag, uint32_t kb, int v0, int v1, float (&s0)[4], float (&s1)[4]) {
        constexpr int NH = decltype(nh_tag)::value;
        float sa[NH][NCH][4];
#pragma unroll
        for (int h = 0; h < NH; h++)
#pragma unroll
            for (int c = 0; c < NCH; c++)
#pragma unroll
                for (int i = 0; i < 4; i++) sa[h][c][i] = 0.f;
        const int mat = lane >> 3;
        const int r = (lane & 7) + ((mat & 1) << 3);
        uint32_t af[NH][NKS][4];
#pragma unroll
        for (int ks = 0; ks < NKS; ks++) {
            const int c = (ks & 3) * 2 + (mat >> 1);
            const uint32_t off = (ks >> 2) * BOX + r * 128 + ((c ^ (r & 7)) << 4);
#pragma unroll
            for (int h = 0; h < NH; h++) ldmatrix_x4(af[h][ks], kb + h * HALF + off);
        }
#pragma unroll
        for (int ks = 0; ks < NKS; ks++)
#pragma unroll
            for (int h = 0; h < NH; h++) {
                mma_bf16_16816(sa[h][(QF32 ? 2 * ks : ks) % NCH], af[h][ks], qb[ks][0], qb[ks][1]);
                if (QF32) mma_bf16_16816(sa[h][(2 * ks + 1) % NCH], af[h][ks], ql[ks][0], ql[ks][1]);
            }
        mask_scale(sa[0], v0, s0);
        if (NH == 2) mask_scale(sa[NH - 1], v1, s1);
    };
    // O^T += V^T . P^T for one half (the V fragments all loaded first).
    auto pv_half = [&](uint32_t vb, uint32_t pb0, uint32_t pb1) {
        const int mat = lane >> 3;
        const int r = (lane & 7) + ((mat >> 1) << 3);
        uint32_t af[NKS][4];
#pragma unroll
        for (int mt = 0; mt < NKS; mt++) {
            const int c = (mt & 3) * 2 + (mat & 1);
            ldmatrix_x4_trans(af[mt], vb + (mt >> 2) * BOX + r * 128 + ((c ^ (r & 7)) << 4));
        }
#pragma unroll
        for (int mt = 0; mt < NKS; mt++) mma_bf16_16816(o[mt], af[mt], pb0, pb1);
    };
    // Zero the V rows of a half past its valid tokens (they may hold NaN).
    // The stores are ordered before the stage's next TMA refill by a proxy
    // fence (a refill only overwrites data the warp has read, which needs
    // none).
    auto zero_v_tail = [&](uint8_t *vhalf, int valid) {
        uint4 *vrow = reinterpret_cast<uint4 *>(vhalf);
        const int n = (16 - valid) * 8;
        for (int i = lane; i < NB * n; i += 32) {
            const int nb = i / n, r = valid + (i % n) / 8, c = i % 8;
            vrow[(nb * BOX + r * 128) / 16 + c] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    };

    // ---------------- main loop: one stage (up to 32 tokens of one row) per pass
    int cs = 0;
    uint32_t cphase = 0;
    int empty_from = row_begin;  // first row not yet given a piece
    produce();
    while (consumed != issued) {
        if (!mbar_wait_bounded(bar + cs, cphase, kWaitLimitNs)) {
            if (lane == 0) raise_error(a.flags, kErrTimeout);
            // let the copies already issued land before the CTA's memory is released
            while (consumed != issued) {
                mbar_wait_bounded(bar + cs, cphase, kWaitLimitNs);
                consumed++;
                if (++cs == S) {
                    cs = 0;
                    cphase ^= 1u;
                }
            }
            if constexpr (ROWCTA) {  // the CTA barrier below is still met; this piece counts as empty
                cur_row = -1;
                break;
            }
            // keep the row counters consistent (the outputs are flagged as invalid)
            if (a.wait_at_exit) pdl_wait();
            if (a.fold) fold_shared_rows<D>(a, row_begin, row_last);
            return;
        }
        const int row = __shfl_sync(0xffffffffu, st_row, cs);
        const int vv = __shfl_sync(0xffffffffu, st_valid, cs);
        const int v0 = vv & 255, v1 = vv >> 8;
        if (row != cur_row) {
            if (cur_row >= 0) finish_row(cur_row);
            for (int r = empty_from; r < row; r++)
                if (r != cur_row) write_empty_piece<D>(a, r, gw);
            empty_from = row + 1;
            cur_row = row;
            start_row(row);
        }
        uint8_t *st = ring + size_t(cs) * STAGE;
        if (v0 < 16) zero_v_tail(st + KVB, v0);
        if (v1 > 0 && v1 < 16) zero_v_tail(st + KVB + HALF, v1);
        if (v0 < 16 || (v1 > 0 && v1 < 16)) __syncwarp();
        const uint32_t kb = smem_u32(st), vb = kb + KVB;

        float s0[4], s1[4];
        if (HALVES == 2 && v1 > 0) {
            qk(std::integral_constant<int, 2>(), kb, v0, v1, s0, s1);
        } else {
            qk(std::integral_constant<int, 1>(), kb, v0, v1, s0, s1);
            s1[0] = s1[1] = s1[2] = s1[3] = -INFINITY;
        }
        // s*[0], s*[2]: head 2t; s*[1], s*[3]: head 2t+1.  Lazy rescale: the
        // running max moves only when some head's new max exceeds it by more
        // than kLazy (then probabilities stay <= 2^kLazy); the per-lane maxima
        // are tested first, so the cross-lane reduction runs only then.
        float mx0 = fmaxf(fmaxf(s0[0], s0[2]), fmaxf(s1[0], s1[2]));
        float mx1 = fmaxf(fmaxf(s0[1], s0[3]), fmaxf(s1[1], s1[3]));
        if (__any_sync(0xffffffffu, mx0 > m0 + kLazy || mx1 > m1 + kLazy)) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
            const float al0 = exp2f(m0 - n0), al1 = exp2f(m1 - n1);
            m0 = n0;
            m1 = n1;
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int mt = 0; mt < NKS; mt++) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
        }
        const uint32_t x00 = pack_bf16x2(exp2f(s0[0] - m0), exp2f(s0[1] - m1));
        const uint32_t x01 = pack_bf16x2(exp2f(s0[2] - m0), exp2f(s0[3] - m1));
        l0 += bf16_lo_to_float(x00) + bf16_lo_to_float(x01);
        l1 += bf16_hi_to_float(x00) + bf16_hi_to_float(x01);
        pv_half(vb, movmatrix_trans(x00), movmatrix_trans(x01));
        if (HALVES == 2 && v1 > 0) {
            const uint32_t x10 = pack_bf16x2(exp2f(s1[0] - m0), exp2f(s1[1] - m1));
            const uint32_t x11 = pack_bf16x2(exp2f(s1[2] - m0), exp2f(s1[3] - m1));
            l0 += bf16_lo_to_float(x10) + bf16_lo_to_float(x11);
            l1 += bf16_hi_to_float(x10) + bf16_hi_to_float(x11);
            pv_half(vb + HALF, movmatrix_trans(x10), movmatrix_trans(x11));
        }
        __syncwarp();
        consumed++;
        if (++cs == S) {
            cs = 0;
            cphase ^= 1u;
        }
        produce();
    }
    if constexpr (ROWCTA) {
        // this warp's piece (normalised o, log2-LSE) at the head of its own ring
        float *piece = reinterpret_cast<float *>(ring);
        float *plse = piece + G * D;
        if (cur_row >= 0) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
            const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
            const int h0 = 2 * t, h1 = 2 * t + 1;
#pragma unroll
            for (int mt = 0; mt < NKS; mt++) {
                const int d0 = mt * 16 + gid;
                if (h0 < G) {
                    piece[h0 * D + d0] = o[mt][0] * i0;
                    piece[h0 * D + d0 + 8] = o[mt][2] * i0;
                }
                if (h1 < G) {
                    piece[h1 * D + d0] = o[mt][1] * i1;
                    piece[h1 * D + d0 + 8] = o[mt][3] * i1;
                }
            }
            if (gid == 0) {
                if (h0 < G) plse[h0] = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
                if (h1 < G) plse[h1] = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
            }
        } else if (lane < G) {
            plse[lane] = -INFINITY;
        }
        __syncthreads();
        // out = sum_w 2^(lse_w - m) o_w / sum_w 2^(lse_w - m), m = max_w lse_w
        const int row = rc_row, b = row / a.num_kv_heads, g = row % a.num_kv_heads;
        const int64_t qh0 = int64_t(b) * a.num_q_heads + int64_t(g) * G;
        const int64_t slot = int64_t(row) * rc_k + rc_blk;  // k > 1: this block's piece
        constexpr int V4 = D / 4;
        for (int c = threadIdx.x; c < G * V4; c += WPC * 32) {  // float4 columns (vector stores)
            const int h = c / V4;
            float m = -INFINITY;
#pragma unroll
            for (int w = 0; w < WPC; w++)
                m = fmaxf(m, reinterpret_cast<const float *>(ring0 + size_t(w) * S * STAGE)[G * D + h]);
            float den = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m != -INFINITY) {
#pragma unroll
                for (int w = 0; w < WPC; w++) {
                    const float *pw = reinterpret_cast<const float *>(ring0 + size_t(w) * S * STAGE);
                    const float l = pw[G * D + h];
                    if (l == -INFINITY) continue;  // a warp without units: no data
                    const float wt = exp2f(l - m);
                    const float4 v = reinterpret_cast<const float4 *>(pw)[c];
                    den += wt;
                    acc.x = fmaf(wt, v.x, acc.x);
                    acc.y = fmaf(wt, v.y, acc.y);
                    acc.z = fmaf(wt, v.z, acc.z);
                    acc.w = fmaf(wt, v.w, acc.w);
                }
            }
            const float inv = den > 0.f ? 1.f / den : 0.f;
            const float4 r4 = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (rc_k == 1) {
                reinterpret_cast<float4 *>(a.out + qh0 * D)[c] = r4;
                if (a.lse && c % V4 == 0) a.lse[qh0 + h] = den > 0.f ? (m + log2f(den)) * kLn2 : -INFINITY;
            } else {
                reinterpret_cast<float4 *>(a.part_o + slot * G * D)[c] = r4;
                if (c % V4 == 0) a.part_lse[slot * G + h] = den > 0.f ? m + log2f(den) : -INFINITY;
            }
        }
        if (rc_k == 1) return;
        // k > 1: the block drawing the row's last ticket folds the k pieces
        __shared__ uint32_t s_last;
        __threadfence();  // this thread's piece stores, before the ticket
        __syncthreads();
        if (threadIdx.x == 0) {
            s_last = atomicAdd(a.tickets + row, 1u) == uint32_t(rc_k - 1) ? 1u : 0u;
            if (s_last) __threadfence();  // the other blocks' pieces, before they are read
        }
        __syncthreads();
        if (!s_last) return;
        // the k x G log-sum-exps into shared memory, then per float4 column
        // the k pieces' loads issued together (one round for G x D <= 768)
        __shared__ float s_plse[kRowBlocksMax * 8];
        const int64_t s0 = int64_t(row) * rc_k;
        for (int i = threadIdx.x; i < rc_k * G; i += WPC * 32) s_plse[i] = __ldcg(a.part_lse + s0 * G + i);
        __syncthreads();
        for (int c = threadIdx.x; c < G * V4; c += WPC * 32) {
            const float4 *po = reinterpret_cast<const float4 *>(a.part_o) + s0 * G * V4 + c;
            float4 v[kRowBlocksMax];
#pragma unroll
            for (int j = 0; j < kRowBlocksMax; j++)
                v[j] = j < rc_k ? __ldcg(po + int64_t(j) * G * V4) : make_float4(0.f, 0.f, 0.f, 0.f);
            const int h = c / V4;
            float m = -INFINITY;
            for (int j = 0; j < rc_k; j++) m = fmaxf(m, s_plse[j * G + h]);
            float den = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m != -INFINITY) {
#pragma unroll
                for (int j = 0; j < kRowBlocksMax; j++) {
                    if (j >= rc_k) break;
                    const float l = s_plse[j * G + h];
                    if (l == -INFINITY) continue;  // an empty piece: its o holds no data
                    const float wt = exp2f(l - m);
                    den += wt;
                    acc.x = fmaf(wt, v[j].x, acc.x);
                    acc.y = fmaf(wt, v[j].y, acc.y);
                    acc.z = fmaf(wt, v[j].z, acc.z);
                    acc.w = fmaf(wt, v[j].w, acc.w);
                }
            }
            const float inv = den > 0.f ? 1.f / den : 0.f;
            reinterpret_cast<float4 *>(a.out + qh0 * D)[c] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (a.lse && c % V4 == 0) a.lse[qh0 + h] = den > 0.f ? (m + log2f(den)) * kLn2 : -INFINITY;
        }
        if (threadIdx.x == 0) a.tickets[row] = 0u;
        return;
    }
    if (cur_row >= 0) finish_row(cur_row);
    for (int r = empty_from; r <= row_last; r++)
        if (r != cur_row) write_empty_piece<D>(a, r, gw);
    if (a.wait_at_exit) pdl_wait();  // a cascade: the prefix kernel's pieces are complete
    if (a.fold) fold_shared_rows<D>(a, row_begin, row_last);
}

// --------------------------------------------------- fp32 KV, CUDA cores --
template <int D, bool QF32>
__global__ void __launch_bounds__(256) decode_simt_kernel(DecodeArgs a) {
    constexpr int PL = D / 32;  // dims per lane: lane + 32 * i
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group;
    const int64_t gw = int64_t(blockIdx.x) * (blockDim.x >> 5) + warp;
    const int64_t u_begin = gw * a.units_per_warp;
    const int64_t u_end = min(u_begin + a.units_per_warp, a.total_units);
    pdl_trigger();
    pdl_wait();
    if (u_begin >= u_end) return;
    float q[8][PL], o[8][PL], m[8], l[8];
    int cur_row = -1;

    auto start_row = [&](int row) {
        const int b = row / a.num_kv_heads, g = row % a.num_kv_heads;
#pragma unroll
        for (int h = 0; h < 8; h++) {
            m[h] = -INFINITY;
            l[h] = 0.f;
            const int64_t qh = int64_t(b) * a.num_q_heads + int64_t(g) * G + (h < G ? h : 0);
#pragma unroll
            for (int i = 0; i < PL; i++) {
                o[h][i] = 0.f;
                const int64_t qi = qh * D + lane + 32 * i;
                q[h][i] = QF32 ? static_cast<const float *>(a.q)[qi]
                               : __bfloat162float(static_cast<const __nv_bfloat16 *>(a.q)[qi]);
            }
        }
    };
    auto finish_row = [&](int row) {
        int64_t w0, w1;
        row_warps(a, row, w0, w1);
        const bool fin = row_is_final(a, w0, w1);
        const int b = row / a.num_kv_heads, g = row % a.num_kv_heads;
        const int64_t qh = int64_t(b) * a.num_q_heads + int64_t(g) * G;
        const int64_t slot = row + gw;
#pragma unroll
        for (int h = 0; h < 8; h++) {
            if (h >= G) break;
            const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
            const float e = l[h] > 0.f ? m[h] + log2f(l[h]) : -INFINITY;
            float *dst = fin ? a.out + (qh + h) * D : a.part_o + (slot * G + h) * D;
#pragma unroll
            for (int i = 0; i < PL; i++) dst[lane + 32 * i] = o[h][i] * inv;
            if (lane == 0) {
                if (fin) {
                    if (a.lse) a.lse[qh + h] = e * kLn2;
                } else {
                    a.part_lse[slot * G + h] = e;
                }
            }
        }
    };

    for (int64_t u = u_begin; u < u_end; u++) {
        const int row = int(u / a.slots_per_row);
        if (row != cur_row) {
            if (cur_row >= 0) finish_row(cur_row);
            cur_row = row;
            start_row(row);
        }
        const int code = unit_code(a, row, int(u - int64_t(row) * a.slots_per_row));
        if (code < 0) continue;
        const int valid = code & 63, phys = code >> 6;
        const int g = row % a.num_kv_heads;
        const int64_t tile = (int64_t(phys) * a.num_kv_heads + g) * a.page_size * D;
        const float *kt = static_cast<const float *>(a.k_pool) + tile;
        const float *vt = static_cast<const float *>(a.v_pool) + tile;
        for (int tok = 0; tok < valid; tok++) {
            float kv[PL], vv[PL];
#pragma unroll
            for (int i = 0; i < PL; i++) {
                kv[i] = kt[tok * D + lane + 32 * i];
                vv[i] = vt[tok * D + lane + 32 * i];
            }
#pragma unroll
            for (int h = 0; h < 8; h++) {
                if (h >= G) break;
                float dot = 0.f;
#pragma unroll
                for (int i = 0; i < PL; i++) dot = fmaf(q[h][i], kv[i], dot);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
                const float s = dot * a.scale_log2;
                const float mn = fmaxf(m[h], s);
                const float al = exp2f(m[h] - mn), p = exp2f(s - mn);
                m[h] = mn;
                l[h] = l[h] * al + p;
#pragma unroll
                for (int i = 0; i < PL; i++) o[h][i] = fmaf(p, vv[i], o[h][i] * al);
            }
        }
    }
    if (cur_row >= 0) finish_row(cur_row);
}

template <int D, bool QF32, bool HINT, bool ROWCTA, bool RANK = false, bool SCORE = false>
cudaError_t launch_bf16_hint(const DecodeArgs &a, const CUtensorMap *tk, const CUtensorMap *tv,
                             const DecodeGrid &grid, cudaStream_t stream) {
    constexpr int WPC = D == 128 ? kDecodeWarpsD128 : kDecodeWarpsD64;
    constexpr int HALVES = D == 128 ? kDecodeHalvesD128 : kDecodeHalvesD64;
    if (grid.warps_per_cta != WPC) return cudaErrorInvalidConfiguration;
    // ROWCTA: the row's unit codes after the rings, then its page-table row if staged
    const size_t smem = decode_smem_bytes(D, a.stages) + (ROWCTA ? rowcta_extra_smem(a, D * (QF32 ? 4 : 2)) : 0);
    const unsigned ctas = ROWCTA ? unsigned(int64_t(a.batch) * a.num_kv_heads * a.row_blocks) : unsigned(grid.ctas);
    auto kernel = decode_bf16_kernel<D, QF32, WPC, HALVES, HINT, ROWCTA, RANK, SCORE>;
    static size_t configured[64] = {0};  // dynamic smem limit already set, per device
    static std::mutex mu;                // calls may come from several host threads
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || configured[dev] < smem) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) configured[dev] = smem;
        }
    }
    // the fused scoring shares a row's scores among its k CTAs: one cluster
    const unsigned cluster = SCORE && ROWCTA ? unsigned(a.row_blocks) : 1u;
    if (cluster > unsigned(kRowBlocksMax)) return cudaErrorInvalidConfiguration;
    if (cluster > 1) {
        // whether one cluster of these CTAs fits an SM group of this device
        // (cached per device and cluster size for the last smem size asked)
        static size_t fit_smem[64][kRowBlocksMax + 1] = {};
        static int fit[64][kRowBlocksMax + 1] = {};
        if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
        std::lock_guard<std::mutex> lock(mu);
        if (fit_smem[dev][cluster] != smem) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(cluster);
            cfg.blockDim = dim3(WPC * 32);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = cluster;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
            if (e != cudaSuccess) (void)cudaGetLastError();  // an answer of "no": not an error of the call
            fit[dev][cluster] = e == cudaSuccess && n >= 1 ? 1 : 0;
            fit_smem[dev][cluster] = smem;
        }
        if (!fit[dev][cluster]) return cudaErrorNotSupported;
    }
    return launch_pdl_cluster(kernel, dim3(ctas), dim3(WPC * 32), smem, stream, cluster, *tk, *tv, a);
}

template <int D, bool QF32>
cudaError_t launch_bf16(const DecodeArgs &a, const CUtensorMap *tk, const CUtensorMap *tv, const DecodeGrid &grid,
                        cudaStream_t stream, bool rowcta = false) {
    if (rowcta && a.scores && a.meta)  // fused score + rank + decode
        return a.kv_evict_first ? launch_bf16_hint<D, QF32, true, true, true, true>(a, tk, tv, grid, stream)
                                : launch_bf16_hint<D, QF32, false, true, true, true>(a, tk, tv, grid, stream);
    if (rowcta && a.scores)  // fused rank + decode
        return a.kv_evict_first ? launch_bf16_hint<D, QF32, true, true, true>(a, tk, tv, grid, stream)
                                : launch_bf16_hint<D, QF32, false, true, true>(a, tk, tv, grid, stream);
    if (rowcta)
        return a.kv_evict_first ? launch_bf16_hint<D, QF32, true, true>(a, tk, tv, grid, stream)
                                : launch_bf16_hint<D, QF32, false, true>(a, tk, tv, grid, stream);
    return a.kv_evict_first ? launch_bf16_hint<D, QF32, true, false>(a, tk, tv, grid, stream)
                            : launch_bf16_hint<D, QF32, false, false>(a, tk, tv, grid, stream);
}

}  // namespace

// Scratch of qskv_sparse_paged_decode_noalloc: the error word and the split
// partial outputs live here instead of in a caller-allocated workspace.  Every device that loads the library holds
// these bytes until the process exits.  All calls share them.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

cudaError_t noalloc_scratch_address(void **ptr) {
    // Resolved once per device, with that device current.
    static void *addr[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

int fused_score_pages_per_round(int head_dim) {
    // the rings' memory holds the page ids and bf16 metadata rows (4 d bytes)
    // of whole 16-page groups (score_row_share)
    const size_t ring = decode_smem_bytes(head_dim, decode_stages(head_dim)) - 1024;
    return int(ring / (16 * (size_t(4) * head_dim + 4))) * 16;
}

size_t rowcta_extra_smem(const DecodeArgs &a, int q_bytes) {
    return size_t((a.slots_per_row + 3) & ~3) * 4 + (a.pt_in_smem ? size_t((a.max_pages + 3) & ~3) * 4 : 0) +
           size_t(a.group) * q_bytes;
}

int row_blocks_for(int64_t rows, int slots_per_row, int ctas, bool no_extra_pieces, bool have_tickets) {
    if (!no_extra_pieces || rows <= 0 || rows > ctas || slots_per_row > kRowCtaMaxSlots) return 0;
    const int64_t sms = ctas / kDecodeCtasPerSm;
    if (rows >= sms) return 1;
    if (!have_tickets) return 0;
    int64_t k = ctas / rows;
    k = k < kRowBlocksMax ? k : kRowBlocksMax;
    k = k < slots_per_row / 4 ? k : slots_per_row / 4;
    return k >= 2 && rows * k >= sms ? int(k) : 0;
}

size_t rowcta_smem_budget() {
    // dynamic shared memory per CTA with kDecodeCtasPerSm CTAs per SM (less
    // a margin for the kernel's static shared memory, about 2 KB), cached per device
    static size_t budget[64] = {0};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!budget[dev]) {
        int per_sm = 0, reserved = 0;
        if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
            return 0;
        const int64_t b = int64_t(per_sm) / kDecodeCtasPerSm - reserved - 3072;
        budget[dev] = b > 0 ? size_t(b) : 1;
    }
    return budget[dev];
}

int decode_stages(int head_dim) { return head_dim == 128 ? kDecodeStagesD128 : kDecodeStagesD64; }

int decode_warps_per_cta(int head_dim) { return head_dim == 128 ? kDecodeWarpsD128 : kDecodeWarpsD64; }

size_t decode_smem_bytes(int head_dim, int stages) {
    const int halves = head_dim == 128 ? kDecodeHalvesD128 : kDecodeHalvesD64;
    const size_t stage = size_t(head_dim / 64) * 16 * 128 * 2 * size_t(halves);  // K and V
    return stage * size_t(stages) * size_t(decode_warps_per_cta(head_dim)) + 1024;
}


cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap *tmap_k, const CUtensorMap *tmap_v, int q_dtype,
                          int kv_dtype, int head_dim, const DecodeGrid &grid, cudaStream_t stream,
                          const PrefixArgs *prefix) {
    const bool qf = q_dtype == kDtypeF32;
    // K/V this call may stream: when it exceeds L2 it is read evict-first, so
    // it does not push the split partials, scores and tables out of L2; a
    // smaller selection is left to stay in L2 for the next step.  A plain
    // dense decode keeps the normal policy: its rows may alias pages (a
    // shared prefix in the block table), which L2 then serves to every row.
    DecodeArgs da = a;
    const int l2 = l2_cache_bytes();
    const double kv_bytes =
        double(a.total_units) * a.page_size * head_dim * 2.0 * (kv_dtype == kDtypeBf16 ? 2.0 : 4.0);
    const bool private_pages = a.selected != nullptr || a.page_begin > 0;
    da.kv_evict_first = private_pages && l2 > 0 && kv_bytes > double(l2) ? 1 : 0;
    if (prefix) {
        // cascade: the shared prefix first, as a persistent grid on a share
        // of the SMs; it waits for the previous kernel and then releases the
        // decode of the rows' own pages, whose grid (sized by the caller to
        // the other SMs) runs beside it.  The decode waits for the prefix
        // grid only at its exit, so the merge behind it sees both.
        if (kv_dtype != kDtypeBf16) return cudaErrorInvalidValue;
        cudaError_t e = launch_prefix(*prefix, tmap_k, tmap_v, q_dtype, head_dim, stream);
        if (e != cudaSuccess) return e;
        // a row's decode pieces and the prefix kernel's are folded by the
        // decode warp that finishes the row last (after its wait for the
        // prefix grid) when one warp can load them in one round; otherwise
        // by the merge kernel
        const int64_t upw_c = a.units_per_warp > 0 ? a.units_per_warp : 1;
        const int64_t pieces_c = (a.slots_per_row + upw_c - 1) / upw_c + 1 + a.extra_pieces;
        const int64_t per_lane_c = a.group * head_dim / 128 > 1 ? a.group * head_dim / 128 : 1;
        const bool fold_c = a.total_units > 0 && a.tickets != nullptr && pieces_c * per_lane_c <= kFoldMaxLoads;
        if (a.total_units > 0) {
            DecodeArgs d = da;
            d.wait_at_exit = 1;
            d.fold = fold_c ? 1 : 0;
            if (head_dim == 128)
                e = qf ? launch_bf16<128, true>(d, tmap_k, tmap_v, grid, stream)
                       : launch_bf16<128, false>(d, tmap_k, tmap_v, grid, stream);
            else
                e = qf ? launch_bf16<64, true>(d, tmap_k, tmap_v, grid, stream)
                       : launch_bf16<64, false>(d, tmap_k, tmap_v, grid, stream);
            if (e != cudaSuccess) return e;
        }
        return fold_c ? cudaSuccess : launch_merge(a, head_dim, stream);
    }
    if (a.total_units == 0) return cudaSuccess;
    if (kv_dtype == kDtypeBf16) {
        // Rows that fit one wave of CTAs are decoded one row per k CTAs (the
        // pieces folded in the CTA, then across the k CTAs by the last one):
        // k = 1 with one or two rows per SM, k > 1 with fewer rows than SMs
        // (up to kRowBlocksMax, at least 4 units per CTA, and then at least
        // one CTA per SM; the fold across CTAs needs the per-row counters).
        const int k = row_blocks_for(int64_t(a.batch) * a.num_kv_heads, a.slots_per_row, grid.ctas,
                                     a.extra_pieces == 0, a.tickets != nullptr);
        if (k > 0) {
            DecodeArgs d = da;
            d.fold = 0;
            d.row_blocks = k;
            // stage the page-table row when two CTAs per SM still fit
            d.pt_in_smem = 1;
            const size_t need = decode_smem_bytes(head_dim, d.stages) + rowcta_extra_smem(d, head_dim * (qf ? 4 : 2));
            if (need > rowcta_smem_budget()) d.pt_in_smem = 0;
            if (head_dim == 128)
                return qf ? launch_bf16<128, true>(d, tmap_k, tmap_v, grid, stream, true)
                          : launch_bf16<128, false>(d, tmap_k, tmap_v, grid, stream, true);
            return qf ? launch_bf16<64, true>(d, tmap_k, tmap_v, grid, stream, true)
                      : launch_bf16<64, false>(d, tmap_k, tmap_v, grid, stream, true);
        }
        const int64_t upw = a.units_per_warp > 0 ? a.units_per_warp : 1;
        const int64_t pieces = (a.slots_per_row + upw - 1) / upw + 1;
        const int64_t per_lane = a.group * head_dim / 128 > 1 ? a.group * head_dim / 128 : 1;
        da.fold = a.tickets != nullptr && pieces * per_lane <= kFoldMaxLoads ? 1 : 0;
        cudaError_t e;
        if (head_dim == 128)
            e = qf ? launch_bf16<128, true>(da, tmap_k, tmap_v, grid, stream)
                   : launch_bf16<128, false>(da, tmap_k, tmap_v, grid, stream);
        else
            e = qf ? launch_bf16<64, true>(da, tmap_k, tmap_v, grid, stream)
                   : launch_bf16<64, false>(da, tmap_k, tmap_v, grid, stream);
        if (e != cudaSuccess) return e;
        return da.fold ? cudaSuccess : launch_merge(a, head_dim, stream);
    }
    const dim3 g(grid.ctas), b(grid.warps_per_cta * 32);
    cudaError_t e;
    if (head_dim == 128)
        e = qf ? launch_pdl(decode_simt_kernel<128, true>, g, b, 0, stream, a)
               : launch_pdl(decode_simt_kernel<128, false>, g, b, 0, stream, a);
    else
        e = qf ? launch_pdl(decode_simt_kernel<64, true>, g, b, 0, stream, a)
               : launch_pdl(decode_simt_kernel<64, false>, g, b, 0, stream, a);
    if (e != cudaSuccess) return e;
    return launch_merge(a, head_dim, stream);
}

}  // namespace qskv

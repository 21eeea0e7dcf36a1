// Shared-prefix cascade decode: the prefix half, on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// When every sequence of a batch starts with the same physical pages (prefix
// sharing of PagedAttention, CS336 Lecture 10 s9.2; the anchor + suffix
// recursion of the Quail AI-SQL engine article, merged by log-sum-exp as in
// flash decoding), the attention of each (sequence, query head) row splits
// into a part over the shared prefix and a part over the row's own pages.
// The prefix part is one dense product per KV head: the B x G query rows of
// the head against the T prefix keys.  This kernel computes it once for all
// rows instead of streaming the prefix pages once per sequence; the paged
// decode kernel covers each row's own pages and the merge kernel combines
// the two by log-sum-exp.
//
// A work item is one tile of 128 query rows (row = sequence-major, query
// head of the group minor), one KV head and one contiguous range of 128-key
// blocks of the prefix (a key split).  The grid is persistent and small
// (about 40 % of the SMs, each CTA taking items in turn): the paged decode of
// the rows' own pages is launched right behind it on the other SMs, so the
// two run side by side instead of the decode waiting for SMs the prefix
// holds.  Roles within an item:
//   TMA warps:     one for K, one for V.  Each gathers its blocks' pages
//                  (16-token x 64-dim boxes, 128-byte swizzle) into its own
//                  ring, deep enough to cover the load latency (a K stage is
//                  refilled as soon as its Q . K^T has run, a V stage once
//                  its P . V has); page ids are read one ring-round ahead.
//   MMA warp:      one lane issues S = Q . K^T into tensor memory (two S
//                  buffers, so S of block j+1 is computed while block j's
//                  softmax runs), then O += P . V into a TMEM accumulator,
//                  with P (and, for bf16 queries, Q) read from tensor memory.
//   softmax warps: two threads per query row (TMEM lane), each owning 64 of
//                  a block's keys and half of the output dims.  A thread
//                  reads its S columns, takes its partial maximum and keeps
//                  the online-softmax state (exp2 with the scale folded into
//                  log2 e, a partial denominator summing the same bf16 values
//                  P . V uses).  The running maximum only moves when a
//                  block's maximum exceeds it by more than 2^8 (one barrier
//                  vote per block; the partial maxima are exchanged only then,
//                  or for the first block), and O is then rescaled in TMEM.
//                  The bf16 P pairs go to a TMEM region of their own once the
//                  previous block's P . V has completed.  At the end each
//                  thread normalises its part of the O row into the workspace
//                  slot of (row, split); the log2-domain log-sum-exp goes with it.
// fp32 queries are split into bf16 hi + lo tiles kept in shared memory (two
// MMAs per k-step).  Between items every role meets at a CTA barrier and the
// mbarriers are invalidated and armed afresh (no copy or MMA is pending by
// then); tensor memory stays allocated until the last item.  Every wait is
// bounded; a wait that gives up flags a timeout, stops the CTA's other
// roles, lets issued copies and MMAs complete and frees the tensor memory
// before the CTA exits.
#include <mutex>

#include "qskv_device.cuh"
#include "qskv_internal.h"

namespace qskv {
namespace {

constexpr int kPrefixMaxStages = 6;

template <int D, bool QF32>
struct PrefixCfg {
    static constexpr int NB = D / 64;                 // 64-dim (128-byte) column groups
    static constexpr int ATOM = 128 * 128;            // 128 rows x 128 bytes
    static constexpr bool Q_TMEM = !QF32;             // bf16 Q: A operand from tensor memory
    static constexpr int QB = NB * ATOM;              // one 128-row Q tile in shared memory
    static constexpr int QSMEM = QF32 ? 2 * QB : 0;   // fp32 Q: hi + lo tiles
    static constexpr int KVB = NB * ATOM;             // K (or V) of one 128-key block
    // ring depths: the K and V rings fill what shared memory is left
    static constexpr int NK = QF32 ? (D == 128 ? 2 : 5) : (D == 128 ? 4 : 6);
    static constexpr int NV = QF32 ? (D == 128 ? 2 : 5) : (D == 128 ? 3 : 6);
    static constexpr int SMEM = QSMEM + (NK + NV) * KVB + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0;              // S buffers: columns [0, 256)
    static constexpr uint32_t O_COL = 256;            // O: [256, 256 + D)
    static constexpr uint32_t P_COL = 384;            // P as bf16 pairs: [384, 448)
    static constexpr uint32_t Q_COL = 448;            // bf16 Q pairs: [448, 448 + D/2)
    static_assert(NK <= kPrefixMaxStages && NV <= kPrefixMaxStages, "ring depth");
    static_assert(SMEM + 2048 <= 227 * 1024, "shared memory budget (dynamic + static)");
};

// Bounded wait that also gives up when another role of the CTA has.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile uint32_t *abort,
                                           uint32_t *flags) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1u;
            raise_error(flags, kErrTimeout);
            return false;
        }
    }
    return true;
}

// The cascade's contract for the sequences of tile `mt`: their first
// prefix_pages table entries equal row 0's and they hold the whole prefix.
__device__ void check_prefix_contract(const PrefixArgs &a, int mt, int t, int nthreads, int T) {
    const int G = a.group;
    const int b_first = mt * (kPrefixRows / G);
    const int b_end = min(a.batch, b_first + kPrefixRows / G);
    const int nseq = b_end - b_first;
    bool bad = false;
    for (int idx = t; idx < nseq * a.prefix_pages; idx += nthreads) {
        const int bb = b_first + idx / a.prefix_pages, jj = idx % a.prefix_pages;
        bad |= __ldg(a.page_table + int64_t(bb) * a.max_pages + jj) != __ldg(a.page_table + jj);
    }
    for (int bb = b_first + t; bb < b_end; bb += nthreads) bad |= __ldg(a.seq_lens + bb) < T;
    if (bad) raise_error(a.flags, kErrPrefix);
}

// Page id of lane `lane`'s page in block `blk` (lanes >= pages in the block,
// and invalid ids, give -1; invalid ids are flagged).
__device__ __forceinline__ int block_page_id(const PrefixArgs &a, int blk, int ppb, int lane) {
    const int pg = blk * ppb + lane;
    if (lane >= ppb || pg >= a.prefix_pages) return -1;
    const int pid = __ldg(a.page_table + pg);  // row 0's entries name the shared pages
    if (pid < 0 || pid >= a.num_pool_pages) {
        raise_error(a.flags, kErrPageId);
        return -1;
    }
    return pid;
}

template <int D, bool QF32>
__global__ void __launch_bounds__(kPrefixThreads, 1)
    prefix_attend_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                         PrefixArgs a) {
    using C = PrefixCfg<D, QF32>;
    constexpr int ATOM = C::ATOM;
    constexpr int KEYS = kPrefixKeys;
    constexpr int TPR = kPrefixRowThreads;
    constexpr int SW = 4 * TPR;           // softmax warps
    constexpr int NSM = 32 * SW;          // softmax threads
    constexpr int KP = KEYS / TPR;        // keys of a block per softmax thread
    constexpr int DP = D / TPR;           // output dims per softmax thread
    constexpr int MMA_WARP = SW, K_WARP = SW + 1, V_WARP = SW + 2;
    constexpr uint32_t kBarRows = 1;      // named barrier of the softmax threads
    constexpr float kLazy = 8.f;
    static_assert(KP % 32 == 0 && DP % 32 == 0, "a thread moves whole 32-column TMEM groups");

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_q, bar_k_full[kPrefixMaxStages], bar_k_empty[kPrefixMaxStages],
        bar_v_full[kPrefixMaxStages], bar_v_empty[kPrefixMaxStages], bar_s_full[2], bar_s_free[2], bar_p_full,
        bar_pv_done, bar_o_full, bar_drain;
    __shared__ float red[TPR][kPrefixRows];
    __shared__ uint32_t s_tmem;
    __shared__ volatile uint32_t s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group, P = a.page_size;
    const int T = a.prefix_pages * P;
    const int nblk = (T + KEYS - 1) / KEYS;
    const int n_items = (a.batch * G + kPrefixRows - 1) / kPrefixRows * a.num_kv_heads * a.splits;
    // Everything before this grid in the stream has completed before the
    // dependents (the decode of the rows' own pages) are released: they
    // skip their own wait until exit.
    pdl_wait();
    pdl_trigger();

    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = base;                        // fp32 Q: [2][NB][128 rows][128 B]
    uint8_t *k_s = base + C::QSMEM;             // [NK][NB][128 keys][128 B]
    uint8_t *v_s = k_s + C::NK * C::KVB;        // [NV][NB][128 keys][128 B]

    // every mbarrier of an item (thread 0); `inval` first when re-arming
    // barriers an earlier item used (none of them has a pending arrival then)
    auto arm_barriers = [&](bool inval) {
        uint64_t *all[] = {&bar_q, &bar_s_full[0], &bar_s_full[1], &bar_s_free[0], &bar_s_free[1], &bar_p_full,
                           &bar_pv_done, &bar_o_full, &bar_drain};
        if (inval) {
            for (uint64_t *b : all) mbar_inval(b);
            for (int i = 0; i < kPrefixMaxStages; i++) {
                mbar_inval(&bar_k_full[i]);
                mbar_inval(&bar_k_empty[i]);
                mbar_inval(&bar_v_full[i]);
                mbar_inval(&bar_v_empty[i]);
            }
        }
        mbar_init(&bar_q, NSM);
        for (int i = 0; i < kPrefixMaxStages; i++) {
            mbar_init(&bar_k_full[i], 1);
            mbar_init(&bar_k_empty[i], 1);
            mbar_init(&bar_v_full[i], 1);
            mbar_init(&bar_v_empty[i], 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar_s_full[i], 1);
            mbar_init(&bar_s_free[i], NSM);
        }
        mbar_init(&bar_p_full, NSM);
        mbar_init(&bar_pv_done, 1);
        mbar_init(&bar_o_full, 1);
        mbar_init(&bar_drain, 1);
        mbar_fence_init();
    };
    if (threadIdx.x == 0) {
        s_abort = 0u;
        arm_barriers(false);
    }
    if (warp == MMA_WARP) tmem_alloc(&s_tmem, C::TMEM_COLS);
    if (warp == K_WARP && lane == 0) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // Persistent grid: CTA x takes items x, x + gridDim.x, ... (an item is a
    // (query tile, KV head, key split)).  Every role meets the barrier at an
    // item's end; the mbarriers are then armed afresh for the next item, and
    // tensor memory stays allocated throughout.
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        if (item != int(blockIdx.x)) {
            if (threadIdx.x == 0) arm_barriers(true);
            __syncthreads();
        }
        int c = item;
        const int split = c % a.splits;
        c /= a.splits;
        const int g = c % a.num_kv_heads;
        const int mt = c / a.num_kv_heads;
        const int blk0 = int(int64_t(split) * nblk / a.splits);
        const int nloc = int(int64_t(split + 1) * nblk / a.splits) - blk0;  // >= 1: splits <= nblk

        if (warp < SW) {
            // ------------------------------------------------ softmax rows
            const int quarter = warp & 3, part = warp >> 2;
            const int r = quarter * 32 + lane;  // tile row = TMEM lane
            const int tr = mt * kPrefixRows + r;
            const int b = tr / G, hq = tr % G;
            const bool row_ok = b < a.batch;
            const uint32_t lane_base = uint32_t(quarter * 32) << 16;
            {
                const int64_t qoff = (int64_t(row_ok ? b : 0) * a.num_q_heads + int64_t(g) * G + hq) * D;
                if (C::Q_TMEM) {
                    // bf16 pairs of the row into TMEM lane r; with d = 64 one
                    // thread of the row stores all 32 columns
                    constexpr int QC = D / 2;                    // columns of a Q row
                    constexpr int QT = QC / TPR >= 32 ? QC / TPR : QC;
                    if (QT == QC / TPR || part == 0) {
                        const int c0 = QT == QC ? 0 : part * QT;
                        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.q) + qoff);
    #pragma unroll
                        for (int cb = 0; cb < QT / 32; cb++) {
                            uint32_t rr[32];
    #pragma unroll
                            for (int k = 0; k < 8; k++) {
                                const uint4 v = row_ok ? __ldg(src + (c0 + cb * 32) / 4 + k) : make_uint4(0, 0, 0, 0);
                                rr[4 * k] = v.x;
                                rr[4 * k + 1] = v.y;
                                rr[4 * k + 2] = v.z;
                                rr[4 * k + 3] = v.w;
                            }
                            tmem_st32(tmem + lane_base + C::Q_COL + c0 + cb * 32, rr);
                        }
                    }
                    tc_fence_before();
                } else {
                    constexpr int CH = D / 8 / TPR;  // 16-byte chunks of 8 dims per thread
    #pragma unroll
                    for (int ch = part * CH; ch < (part + 1) * CH; ch++) {
                        uint4 hv = make_uint4(0, 0, 0, 0), lv = make_uint4(0, 0, 0, 0);
                        if (row_ok) {
                            const float4 *src =
                                reinterpret_cast<const float4 *>(static_cast<const float *>(a.q) + qoff) + 2 * ch;
                            const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
                            hv = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w), pack_bf16x2(x1.x, x1.y),
                                            pack_bf16x2(x1.z, x1.w));
                            lv = make_uint4(pack_bf16x2(x0.x - bf16_lo_to_float(hv.x), x0.y - bf16_hi_to_float(hv.x)),
                                            pack_bf16x2(x0.z - bf16_lo_to_float(hv.y), x0.w - bf16_hi_to_float(hv.y)),
                                            pack_bf16x2(x1.x - bf16_lo_to_float(hv.z), x1.y - bf16_hi_to_float(hv.z)),
                                            pack_bf16x2(x1.z - bf16_lo_to_float(hv.w), x1.w - bf16_hi_to_float(hv.w)));
                        }
                        const uint32_t off = (ch >> 3) * ATOM + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
                        *reinterpret_cast<uint4 *>(q_s + off) = hv;
                        *reinterpret_cast<uint4 *>(q_s + C::QB + off) = lv;
                    }
                    fence_proxy_async_smem();
                }
                mbar_arrive(&bar_q);
            }
            if (g == 0 && split == 0) check_prefix_contract(a, mt, threadIdx.x, NSM, T);

            const float sc = a.scale_log2;
            float m = -INFINITY;  // running maximum of the scaled logits (log2 domain)
            float l4[4] = {0.f, 0.f, 0.f, 0.f};  // partial denominator over this thread's keys
            bool ok = true;       // warp-uniform; after a failed wait the warp only keeps
                                  // visiting the named barriers (they have no time limit)
            for (int i = 0; i < nloc; i++) {
                const int ntok = min(KEYS, T - (blk0 + i) * KEYS);
                const int sb = i & 1;
                float sv[KP];
                float lmax = -INFINITY;
                if (ok) ok = __all_sync(0xffffffffu, wait_phase(&bar_s_full[sb], (i >> 1) & 1, &s_abort, a.flags));
                if (ok) {
                    tc_fence_after();
    #pragma unroll
                    for (int cb = 0; cb < KP / 32; cb++) {
                        uint32_t rr[32];
                        tmem_ld32(tmem + lane_base + C::S_COL + sb * KEYS + part * KP + cb * 32, rr);
    #pragma unroll
                        for (int k = 0; k < 32; k++) sv[cb * 32 + k] = __uint_as_float(rr[k]);
                    }
                    tc_fence_before();
                    mbar_arrive(&bar_s_free[sb]);
                    if (ntok < KEYS) {
    #pragma unroll
                        for (int k = 0; k < KP; k++)
                            if (part * KP + k >= ntok) sv[k] = -INFINITY;
                    }
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    #pragma unroll
                    for (int k = 0; k < KP; k++) mx[k & 3] = fmaxf(mx[k & 3], sv[k]);
                    lmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                }
                // the row's maximum is needed on the first block, and later only
                // when some row's block maximum leaves the 2^8 band
                float mn = m;
                if (i == 0 || named_bar_any(kBarRows, NSM, ok && lmax * sc > m + kLazy)) {
                    red[part][r] = lmax;
                    named_bar_sync(kBarRows, NSM);
                    float rm = red[0][r];
    #pragma unroll
                    for (int pp = 1; pp < TPR; pp++) rm = fmaxf(rm, red[pp][r]);
                    const float cand = rm * sc;
                    mn = (i == 0 || cand > m + kLazy) ? cand : m;
                    named_bar_sync(kBarRows, NSM);  // everyone has read `red` before it is reused
                }
                if (!ok) continue;
                uint32_t pk[KP / 2];
    #pragma unroll
                for (int k = 0; k < KP / 2; k++) {
                    pk[k] = pack_bf16x2(exp2f(fmaf(sv[2 * k], sc, -mn)), exp2f(fmaf(sv[2 * k + 1], sc, -mn)));
                }
                const float al = exp2f(m - mn);  // 1 for rows that keep their maximum
    #pragma unroll
                for (int k = 0; k < 4; k++) l4[k] *= al;
    #pragma unroll
                for (int k = 0; k < KP / 2; k++)
                    l4[k & 3] += bf16_lo_to_float(pk[k]) + bf16_hi_to_float(pk[k]);
                if (i > 0) {
                    // P . V of the previous block must be complete: it read the
                    // P region and accumulated into O
                    ok = __all_sync(0xffffffffu, wait_phase(&bar_pv_done, (i - 1) & 1, &s_abort, a.flags));
                    if (!ok) continue;
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, mn != m)) {
    #pragma unroll 1
                        for (int cb = 0; cb < DP / 32; cb++) {
                            uint32_t rr[32];
                            const uint32_t ta = tmem + lane_base + C::O_COL + part * DP + cb * 32;
                            tmem_ld32(ta, rr);
    #pragma unroll
                            for (int k = 0; k < 32; k++) rr[k] = __float_as_uint(__uint_as_float(rr[k]) * al);
                            tmem_st32(ta, rr);
                        }
                    }
                }
                m = mn;
    #pragma unroll
                for (int cb = 0; cb < KP / 64; cb++) {
                    uint32_t rr[32];
    #pragma unroll
                    for (int k = 0; k < 32; k++) rr[k] = pk[cb * 32 + k];
                    tmem_st32(tmem + lane_base + C::P_COL + part * (KP / 2) + cb * 32, rr);
                }
                tc_fence_before();
                mbar_arrive(&bar_p_full);
            }
            // the row's denominator: the parts' partial sums (all softmax threads
            // take part, whatever happened above)
            red[part][r] = (l4[0] + l4[1]) + (l4[2] + l4[3]);
            named_bar_sync(kBarRows, NSM);
            float l = 0.f;
    #pragma unroll
            for (int pp = 0; pp < TPR; pp++) l += red[pp][r];
            if (ok) ok = __all_sync(0xffffffffu, wait_phase(&bar_o_full, 0, &s_abort, a.flags));
            if (ok) {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int64_t slot = a.slot0 + (int64_t(row_ok ? b : 0) * a.num_kv_heads + g) * a.splits + split;
                float4 *dst = reinterpret_cast<float4 *>(a.part_o + (slot * G + hq) * D + part * DP);
    #pragma unroll 1
                for (int cb = 0; cb < DP / 32; cb++) {
                    uint32_t rr[32];
                    tmem_ld32(tmem + lane_base + C::O_COL + part * DP + cb * 32, rr);
                    if (row_ok) {
    #pragma unroll
                        for (int k = 0; k < 8; k++)
                            dst[cb * 8 + k] = make_float4(__uint_as_float(rr[4 * k]) * inv, __uint_as_float(rr[4 * k + 1]) * inv,
                                                          __uint_as_float(rr[4 * k + 2]) * inv,
                                                          __uint_as_float(rr[4 * k + 3]) * inv);
                    }
                }
                if (row_ok && part == 0) a.part_lse[slot * G + hq] = l > 0.f ? m + log2f(l) : -INFINITY;
            }
        } else if (warp == K_WARP || warp == V_WARP) {
            // ------------------------------------------------ TMA producers
            const bool is_k = warp == K_WARP;
            const int NS = is_k ? C::NK : C::NV;
            const CUtensorMap *map = is_k ? &tmap_k : &tmap_v;
            const uint8_t *pool = static_cast<const uint8_t *>(is_k ? a.k_pool : a.v_pool);
            uint8_t *ring = is_k ? k_s : v_s;
            uint64_t *full = is_k ? bar_k_full : bar_v_full;
            uint64_t *empty = is_k ? bar_k_empty : bar_v_empty;
            const int ppb = KEYS / P;  // pages per block
            const uint32_t tile_bytes = uint32_t(P) * D * 2;
            // every page tile of this key range, requested from L2 up front (by
            // the first query tile's CTA only: the others read the same pages)
            for (int idx = lane; mt == 0 && idx < nloc * ppb; idx += 32) {
                const int pg = blk0 * ppb + idx;
                if (pg < a.prefix_pages) {
                    const int pid = __ldg(a.page_table + pg);
                    if (pid >= 0 && pid < a.num_pool_pages)
                        prefetch_l2_bulk(pool + (int64_t(pid) * a.num_kv_heads + g) * tile_bytes, tile_bytes);
                }
            }
            // page ids of the next ring-round of blocks, lane j holding page j
            int ids[kPrefixMaxStages];
    #pragma unroll
            for (int s = 0; s < kPrefixMaxStages; s++)
                ids[s] = s < NS && s < nloc ? block_page_id(a, blk0 + s, ppb, lane) : -1;
            int nissued = 0;
            bool ok = true;
            for (int i = 0; i < nloc; i++) {
                const int st = i % NS;
                int pid = -1;
    #pragma unroll
                for (int s = 0; s < kPrefixMaxStages; s++)
                    if (s == st) pid = ids[s];
                if (i >= NS) {
                    ok = __all_sync(0xffffffffu, wait_phase(&empty[st], ((i / NS) - 1) & 1, &s_abort, a.flags));
                    if (!ok) break;
                }
                uint8_t *buf = ring + st * C::KVB;
                const uint32_t good = __ballot_sync(0xffffffffu, pid >= 0);
                if (good != (1u << ppb) - 1u) {
                    // token rows without data (past the prefix, or an invalid
                    // page) are zeroed so the masked columns stay finite
                    for (int idx = lane; idx < KEYS * C::NB * 8; idx += 32) {
                        const int row = idx / (C::NB * 8), rest = idx % (C::NB * 8);
                        if ((good >> (row / P)) & 1u) continue;
                        *reinterpret_cast<uint4 *>(buf + (rest >> 3) * ATOM + row * 128 + (rest & 7) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(&full[st], uint32_t(__popc(good)) * tile_bytes);
                __syncwarp();
                if (pid >= 0) {
                    for (int sub = 0; sub < P / 16; sub++) {
                        const int y = (pid * a.num_kv_heads + g) * P + sub * 16;
                        const int row = lane * P + sub * 16;
    #pragma unroll
                        for (int nb = 0; nb < C::NB; nb++) tma_load_2d(buf + nb * ATOM + row * 128, map, nb * 64, y, &full[st]);
                    }
                }
                nissued++;
                // this stage's next block: its ids are read now, a ring-round ahead
                const int nxt = i + NS < nloc ? block_page_id(a, blk0 + i + NS, ppb, lane) : -1;
    #pragma unroll
                for (int s = 0; s < kPrefixMaxStages; s++)
                    if (s == st) ids[s] = nxt;
            }
            if (!ok) {  // copies already issued land before the CTA's memory is released
                for (int i = max(0, nissued - NS); i < nissued; i++)
                    mbar_wait_bounded(&full[i % NS], (i / NS) & 1, kWaitLimitNs);
            }
        } else {
            // ------------------------------------------------ MMA issuer
            if (lane == 0) {
                constexpr uint32_t idS = tc_idesc_bf16(128, KEYS, false, false);
                constexpr uint32_t idO = tc_idesc_bf16(128, D, false, true);
                const uint32_t qa = smem_u32(q_s), ka0 = smem_u32(k_s), va0 = smem_u32(v_s);
                bool issued = false;
                auto pv = [&](int i) -> bool {
                    const int st = i % C::NV;
                    if (!wait_phase(&bar_p_full, i & 1, &s_abort, a.flags)) return false;
                    if (!wait_phase(&bar_v_full[st], (i / C::NV) & 1, &s_abort, a.flags)) return false;
                    tc_fence_after();
                    const uint32_t va = va0 + st * C::KVB;
    #pragma unroll
                    for (int ks = 0; ks < KEYS / 16; ks++) {
                        // A = P from TMEM (8 columns = 16 keys); B = V, MN-major (dims contiguous)
                        tc_mma_bf16_ts(tmem + C::O_COL, tmem + C::P_COL + ks * 8,
                                       tc_sdesc_sw128(va + ks * 16 * 128, ATOM, 1024), idO, i > 0 || ks > 0);
                    }
                    tc_commit(&bar_v_empty[st]);
                    tc_commit(&bar_pv_done);
                    return true;
                };
                bool ok = wait_phase(&bar_q, 0, &s_abort, a.flags);
                for (int i = 0; i < nloc && ok; i++) {
                    const int st = i % C::NK, sb = i & 1;
                    ok = wait_phase(&bar_k_full[st], (i / C::NK) & 1, &s_abort, a.flags);
                    if (ok && i >= 2) ok = wait_phase(&bar_s_free[sb], ((i - 2) >> 1) & 1, &s_abort, a.flags);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t ka = ka0 + st * C::KVB;
    #pragma unroll
                    for (int kk = 0; kk < D / 16; kk++) {
                        // A = Q (TMEM, or K-major in shared memory), B = K, K-major
                        const uint32_t koff = (kk >> 2) * ATOM + (kk & 3) * 32;
                        const uint64_t bd = tc_sdesc_sw128(ka + koff, 16, 1024);
                        if (C::Q_TMEM) {
                            tc_mma_bf16_ts(tmem + C::S_COL + sb * KEYS, tmem + C::Q_COL + kk * 8, bd, idS, kk > 0);
                        } else {
                            tc_mma_bf16(tmem + C::S_COL + sb * KEYS, tc_sdesc_sw128(qa + koff, 16, 1024), bd, idS,
                                        kk > 0);
                            tc_mma_bf16(tmem + C::S_COL + sb * KEYS, tc_sdesc_sw128(qa + C::QB + koff, 16, 1024), bd,
                                        idS, true);
                        }
                    }
                    tc_commit(&bar_k_empty[st]);
                    tc_commit(&bar_s_full[sb]);
                    issued = true;
                    if (i >= 1) ok = pv(i - 1);
                }
                if (ok) ok = pv(nloc - 1);
                if (ok) tc_commit(&bar_o_full);
                if (issued) {  // every MMA has completed before the tensor memory is freed
                    tc_commit(&bar_drain);
                    mbar_wait_bounded(&bar_drain, 0, kWaitLimitNs);
                }
            }
            __syncwarp();
        }

        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (warp == MMA_WARP) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, bool QF32>
cudaError_t launch_prefix_t(const PrefixArgs &a, const CUtensorMap *tk, const CUtensorMap *tv, int ctas,
                            cudaStream_t stream) {
    using C = PrefixCfg<D, QF32>;
    auto kernel = prefix_attend_kernel<D, QF32>;
    static bool configured[64] = {false};  // dynamic smem limit set, per device
    static std::mutex mu;                  // calls may come from several host threads
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || !configured[dev]) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) configured[dev] = true;
        }
    }
    return launch_pdl(kernel, dim3(ctas), dim3(kPrefixThreads), size_t(C::SMEM), stream, *tk, *tv, a);
}

}  // namespace

int prefix_splits(int batch, int group, int num_kv_heads, int page_size, int prefix_pages, int num_sms) {
    const int64_t T = int64_t(prefix_pages) * page_size;
    const int nblk = int((T + kPrefixKeys - 1) / kPrefixKeys);
    if (nblk == 0) return 0;
    const int64_t tiles = prefix_tiles(batch, group) * int64_t(num_kv_heads);
    int64_t e = num_sms / tiles;
    if (e < 1) e = 1;
    if (e > nblk) e = nblk;
    if (e > kMaxPrefixSplits) e = kMaxPrefixSplits;
    return int(e);
}

int prefix_tiles(int batch, int group) {
    return int((int64_t(batch) * group + kPrefixRows - 1) / kPrefixRows);
}

// Persistent prefix CTAs for `items` work items: about kPrefixSmShare of the
// SMs, each taking an equal number of items, so that the paged decode of the
// rows' own pages runs beside them on the other SMs from the start.
int prefix_ctas(int items, int num_sms) {
    if (items <= 0) return 0;
    int share = int(float(num_sms) * kPrefixSmShare);
    share = share < 1 ? 1 : share;
    const int rounds = (items + share - 1) / share;
    return (items + rounds - 1) / rounds;
}

cudaError_t launch_prefix(const PrefixArgs &a, const CUtensorMap *tmap_k, const CUtensorMap *tmap_v, int q_dtype,
                          int head_dim, cudaStream_t stream) {
    const int items = prefix_tiles(a.batch, a.group) * a.num_kv_heads * a.splits;
    if (items == 0) return cudaSuccess;
    const int ctas = a.ctas > 0 && a.ctas < items ? a.ctas : items;
    const bool qf = q_dtype == kDtypeF32;
    if (head_dim == 128)
        return qf ? launch_prefix_t<128, true>(a, tmap_k, tmap_v, ctas, stream)
                  : launch_prefix_t<128, false>(a, tmap_k, tmap_v, ctas, stream);
    return qf ? launch_prefix_t<64, true>(a, tmap_k, tmap_v, ctas, stream)
              : launch_prefix_t<64, false>(a, tmap_k, tmap_v, ctas, stream);
}

}  // namespace qskv

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
// A CTA owns one tile of 128 query rows (row = sequence-major, query head of
// the group minor), one KV head and one contiguous range of 128-key blocks
// of the prefix (a key split).  Roles:
//   warp 4, TMA:   gathers each block's pages (K and V, 16-token x 64-dim
//                  boxes, 128-byte swizzle) into a two-stage ring;
//   warp 5, MMA:   one lane issues S = Q . K^T into tensor memory (two S
//                  buffers, so S of block j+1 is computed while block j's
//                  softmax runs) and O += P . V into a TMEM accumulator;
//   warps 0-3:     thread r owns query row r (TMEM lane r): it reads its S
//                  row, keeps the online-softmax state (exp2 with the scale
//                  folded into log2 e; the running maximum is only moved, and
//                  O rescaled in TMEM, when a block's maximum exceeds it by
//                  more than 2^8), writes its bf16 P row into shared memory
//                  for the next MMA, and at the end normalises its O row into
//                  the workspace slot of (row, split) with its log2-domain
//                  log-sum-exp.
// fp32 queries are split into bf16 hi + lo tiles (two MMAs per k-step).  The
// softmax denominator sums the same bf16-rounded probabilities the P . V
// product uses.  Every wait is bounded; a wait that gives up flags a timeout,
// stops the CTA's other roles, lets issued copies and MMAs complete and frees
// the tensor memory before the CTA exits.
#include "qskv_device.cuh"
#include "qskv_internal.h"

namespace qskv {
namespace {

template <int D, bool QF32>
struct PrefixCfg {
    static constexpr int NB = D / 64;                 // 64-dim (128-byte) column groups
    static constexpr int ATOM = 128 * 128;            // 128 rows x 128 bytes
    static constexpr int QB = NB * ATOM;              // one 128-row Q tile
    static constexpr int NQ = QF32 ? 2 : 1;           // hi (+ lo) tiles
    static constexpr int KVB = NB * ATOM;             // K (or V) of one 128-key block
    static constexpr int NSTAGE = 2;
    static constexpr int NP = (QF32 && D == 128) ? 1 : 2;  // P buffers
    static constexpr int PB = 2 * ATOM;               // 128 rows x 128 keys
    static constexpr int SMEM = NQ * QB + NSTAGE * 2 * KVB + NP * PB + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0;              // S buffers: columns [0, 256)
    static constexpr uint32_t O_COL = 256;            // O: columns [256, 256 + D)
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
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
__device__ void check_prefix_contract(const PrefixArgs &a, int mt, int r, int T) {
    const int G = a.group;
    const int b_first = mt * (kPrefixRows / G);
    const int b_end = min(a.batch, b_first + kPrefixRows / G);
    const int nseq = b_end - b_first;
    bool bad = false;
    for (int idx = r; idx < nseq * a.prefix_pages; idx += kPrefixRows) {
        const int bb = b_first + idx / a.prefix_pages, jj = idx % a.prefix_pages;
        bad |= __ldg(a.page_table + int64_t(bb) * a.max_pages + jj) != __ldg(a.page_table + jj);
    }
    for (int bb = b_first + r; bb < b_end; bb += kPrefixRows) bad |= __ldg(a.seq_lens + bb) < T;
    if (bad) raise_error(a.flags, kErrPrefix);
}

template <int D, bool QF32>
__global__ void __launch_bounds__(kPrefixThreads, 1)
    prefix_attend_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                         PrefixArgs a) {
    using C = PrefixCfg<D, QF32>;
    constexpr int ATOM = C::ATOM;
    constexpr int KEYS = kPrefixKeys;
    constexpr float kLazy = 8.f;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_q, bar_kv_full[2], bar_kv_empty[2], bar_s_full[2], bar_s_free[2],
        bar_p_full[2], bar_p_free[2], bar_o_full, bar_drain;
    __shared__ uint32_t s_tmem;
    __shared__ volatile uint32_t s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group, P = a.page_size;
    int c = blockIdx.x;
    const int split = c % a.splits;
    c /= a.splits;
    const int g = c % a.num_kv_heads;
    const int mt = c / a.num_kv_heads;
    const int T = a.prefix_pages * P;
    const int nblk = (T + KEYS - 1) / KEYS;
    const int blk0 = int(int64_t(split) * nblk / a.splits);
    const int nloc = int(int64_t(split + 1) * nblk / a.splits) - blk0;  // >= 1: splits <= nblk
    pdl_trigger();

    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = base;                           // [NQ][NB][128 rows][128 B]
    uint8_t *kv_s = base + C::NQ * C::QB;          // stage st: K at + st*2*KVB, V at + KVB
    uint8_t *p_s = kv_s + C::NSTAGE * 2 * C::KVB;  // [NP][2][128 rows][128 B]

    if (threadIdx.x == 0) {
        mbar_init(&bar_q, 128);
        for (int i = 0; i < 2; i++) {
            mbar_init(&bar_kv_full[i], 1);
            mbar_init(&bar_kv_empty[i], 1);
            mbar_init(&bar_s_full[i], 1);
            mbar_init(&bar_s_free[i], 128);
            mbar_init(&bar_p_full[i], 128);
            mbar_init(&bar_p_free[i], 1);
        }
        mbar_init(&bar_o_full, 1);
        mbar_init(&bar_drain, 1);
        s_abort = 0u;
        mbar_fence_init();
    }
    if (warp == 5) tmem_alloc(&s_tmem, C::TMEM_COLS);
    if (warp == 4 && lane == 0) {
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp < 4) {
        // ------------------------------------------------ softmax rows
        const int r = threadIdx.x;
        const int tr = mt * kPrefixRows + r;
        const int b = tr / G, hq = tr % G;
        const bool row_ok = b < a.batch;
        const uint32_t lane_base = uint32_t(warp * 32) << 16;
        {
            const int64_t qoff = (int64_t(row_ok ? b : 0) * a.num_q_heads + int64_t(g) * G + hq) * D;
#pragma unroll 4
            for (int ch = 0; ch < D / 8; ch++) {  // 16-byte chunks of 8 dims
                uint4 hv = make_uint4(0, 0, 0, 0), lv = make_uint4(0, 0, 0, 0);
                if (row_ok) {
                    if (QF32) {
                        const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(a.q) + qoff) + 2 * ch;
                        const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
                        hv = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w), pack_bf16x2(x1.x, x1.y),
                                        pack_bf16x2(x1.z, x1.w));
                        lv = make_uint4(pack_bf16x2(x0.x - bf16_lo_to_float(hv.x), x0.y - bf16_hi_to_float(hv.x)),
                                        pack_bf16x2(x0.z - bf16_lo_to_float(hv.y), x0.w - bf16_hi_to_float(hv.y)),
                                        pack_bf16x2(x1.x - bf16_lo_to_float(hv.z), x1.y - bf16_hi_to_float(hv.z)),
                                        pack_bf16x2(x1.z - bf16_lo_to_float(hv.w), x1.w - bf16_hi_to_float(hv.w)));
                    } else {
                        hv = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.q) + qoff) + ch);
                    }
                }
                const uint32_t off = (ch >> 3) * ATOM + r * 128 + (((ch & 7) ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(q_s + off) = hv;
                if (QF32) *reinterpret_cast<uint4 *>(q_s + C::QB + off) = lv;
            }
            fence_proxy_async_smem();
            mbar_arrive(&bar_q);
        }
        if (g == 0 && split == 0) check_prefix_contract(a, mt, r, T);

        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < nloc; i++) {
            const int ntok = min(KEYS, T - (blk0 + i) * KEYS);
            const int sb = i & 1, pb = i % C::NP;
            ok = __all_sync(0xffffffffu, wait_phase(&bar_s_full[sb], (i >> 1) & 1, &s_abort, a.flags));
            if (!ok) break;
            tc_fence_after();
            float sv[KEYS];
#pragma unroll
            for (int cb = 0; cb < KEYS / 32; cb++) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_base + C::S_COL + sb * KEYS + cb * 32, rr);
#pragma unroll
                for (int k = 0; k < 32; k++) sv[cb * 32 + k] = __uint_as_float(rr[k]);
            }
            tc_fence_before();
            mbar_arrive(&bar_s_free[sb]);
            float bm = -INFINITY;
#pragma unroll
            for (int k = 0; k < KEYS; k++) {
                const float x = k < ntok ? sv[k] * a.scale_log2 : -INFINITY;
                sv[k] = x;
                bm = fmaxf(bm, x);
            }
            if (i == 0) {
                m = bm;  // O is written (not accumulated) by the first P . V
            } else {
                const bool resc = bm > m + kLazy;
                if (__any_sync(0xffffffffu, resc)) {
                    // P . V of the previous block must have landed in O first
                    const int pp = i - 1;
                    ok = __all_sync(0xffffffffu,
                                    wait_phase(&bar_p_free[pp % C::NP], (pp / C::NP) & 1, &s_abort, a.flags));
                    if (!ok) break;
                    tc_fence_after();
                    const float mn = resc ? bm : m;
                    const float al = exp2f(m - mn);
#pragma unroll 1
                    for (int cb = 0; cb < D / 32; cb++) {
                        uint32_t rr[32];
                        const uint32_t ta = tmem + lane_base + C::O_COL + cb * 32;
                        tmem_ld32(ta, rr);
#pragma unroll
                        for (int k = 0; k < 32; k++) rr[k] = __float_as_uint(__uint_as_float(rr[k]) * al);
                        tmem_st32(ta, rr);
                    }
                    l *= al;
                    m = mn;
                }
            }
            if (i >= C::NP) {  // P buffer pb is free once P . V of block i - NP completed
                ok = __all_sync(0xffffffffu,
                                wait_phase(&bar_p_free[pb], ((i - C::NP) / C::NP) & 1, &s_abort, a.flags));
                if (!ok) break;
            }
            uint8_t *prow = p_s + pb * C::PB + r * 128;
#pragma unroll
            for (int ch = 0; ch < KEYS / 8; ch++) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    w[k] = pack_bf16x2(exp2f(sv[ch * 8 + 2 * k] - m), exp2f(sv[ch * 8 + 2 * k + 1] - m));
                    l += bf16_lo_to_float(w[k]) + bf16_hi_to_float(w[k]);
                }
                *reinterpret_cast<uint4 *>(prow + (ch >> 3) * ATOM + (((ch & 7) ^ (r & 7)) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar_p_full[pb]);
        }
        if (ok) ok = __all_sync(0xffffffffu, wait_phase(&bar_o_full, 0, &s_abort, a.flags));
        if (ok) {
            tc_fence_after();
            pdl_wait();  // the previous user of the workspace slots has finished
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t slot = a.slot0 + (int64_t(row_ok ? b : 0) * a.num_kv_heads + g) * a.splits + split;
            float4 *dst = reinterpret_cast<float4 *>(a.part_o + (slot * G + hq) * D);
#pragma unroll 1
            for (int cb = 0; cb < D / 32; cb++) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_base + C::O_COL + cb * 32, rr);
                if (row_ok) {
#pragma unroll
                    for (int k = 0; k < 8; k++)
                        dst[cb * 8 + k] = make_float4(__uint_as_float(rr[4 * k]) * inv, __uint_as_float(rr[4 * k + 1]) * inv,
                                                      __uint_as_float(rr[4 * k + 2]) * inv,
                                                      __uint_as_float(rr[4 * k + 3]) * inv);
                }
            }
            if (row_ok) a.part_lse[slot * G + hq] = l > 0.f ? m + log2f(l) : -INFINITY;
        }
    } else if (warp == 4) {
        // ------------------------------------------------ TMA producer
        const int ppb = KEYS / P;  // pages per block
        int nissued = 0;
        bool ok = true;
        for (int i = 0; i < nloc; i++) {
            const int st = i % C::NSTAGE;
            if (i >= C::NSTAGE) {
                ok = __all_sync(0xffffffffu,
                                wait_phase(&bar_kv_empty[st], ((i / C::NSTAGE) - 1) & 1, &s_abort, a.flags));
                if (!ok) break;
            }
            uint8_t *ks = kv_s + st * 2 * C::KVB, *vs = ks + C::KVB;
            const int pg0 = (blk0 + i) * ppb;
            const int npg = min(ppb, a.prefix_pages - pg0);
            int pid = -1;
            if (lane < npg) {
                pid = __ldg(a.page_table + pg0 + lane);  // row 0's entries name the shared pages
                if (pid < 0 || pid >= a.num_pool_pages) {
                    raise_error(a.flags, kErrPageId);
                    pid = -1;
                }
            }
            const uint32_t good = __ballot_sync(0xffffffffu, pid >= 0);
            if (good != (1u << ppb) - 1u) {
                // token rows without data (past the prefix, or an invalid
                // page): zero K and V so the masked columns stay finite
                for (int idx = lane; idx < KEYS * C::NB * 8; idx += 32) {
                    const int row = idx / (C::NB * 8), rest = idx % (C::NB * 8);
                    if ((good >> (row / P)) & 1u) continue;
                    const uint32_t off = (rest >> 3) * ATOM + row * 128 + (rest & 7) * 16;
                    *reinterpret_cast<uint4 *>(ks + off) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(vs + off) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&bar_kv_full[st], uint32_t(__popc(good)) * P * D * 2 * 2);
            __syncwarp();
            if (pid >= 0) {
                for (int sub = 0; sub < P / 16; sub++) {
                    const int y = (pid * a.num_kv_heads + g) * P + sub * 16;
                    const int row = lane * P + sub * 16;
#pragma unroll
                    for (int nb = 0; nb < C::NB; nb++) {
                        tma_load_2d(ks + nb * ATOM + row * 128, &tmap_k, nb * 64, y, &bar_kv_full[st]);
                        tma_load_2d(vs + nb * ATOM + row * 128, &tmap_v, nb * 64, y, &bar_kv_full[st]);
                    }
                }
            }
            nissued++;
        }
        if (!ok) {  // copies already issued land before the CTA's memory is released
            for (int i = max(0, nissued - C::NSTAGE); i < nissued; i++)
                mbar_wait_bounded(&bar_kv_full[i % C::NSTAGE], (i / C::NSTAGE) & 1, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = tc_idesc_bf16(128, KEYS, false, false);
            constexpr uint32_t idO = tc_idesc_bf16(128, D, false, true);
            const uint32_t qa = smem_u32(q_s), kva = smem_u32(kv_s), pa0 = smem_u32(p_s);
            bool issued = false;
            auto pv = [&](int i) -> bool {
                const int pb = i % C::NP, st = i % C::NSTAGE;
                if (!wait_phase(&bar_p_full[pb], (i / C::NP) & 1, &s_abort, a.flags)) return false;
                tc_fence_after();
                const uint32_t pa = pa0 + pb * C::PB, va = kva + st * 2 * C::KVB + C::KVB;
#pragma unroll
                for (int ks = 0; ks < KEYS / 16; ks++) {
                    // A = P (K-major, keys along K); B = V (MN-major: dims contiguous)
                    const uint64_t ad = tc_sdesc_sw128(pa + (ks >> 2) * ATOM + (ks & 3) * 32, 16, 1024);
                    const uint64_t bd = tc_sdesc_sw128(va + ks * 16 * 128, ATOM, 1024);
                    tc_mma_bf16(tmem + C::O_COL, ad, bd, idO, i > 0 || ks > 0);
                }
                tc_commit(&bar_kv_empty[st]);
                tc_commit(&bar_p_free[pb]);
                return true;
            };
            bool ok = wait_phase(&bar_q, 0, &s_abort, a.flags);
            for (int i = 0; i < nloc && ok; i++) {
                const int st = i % C::NSTAGE, sb = i & 1;
                ok = wait_phase(&bar_kv_full[st], (i / C::NSTAGE) & 1, &s_abort, a.flags);
                if (ok && i >= 2) ok = wait_phase(&bar_s_free[sb], ((i - 2) >> 1) & 1, &s_abort, a.flags);
                if (!ok) break;
                tc_fence_after();
                const uint32_t ka = kva + st * 2 * C::KVB;
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) {
                    // A = Q, B = K, both K-major (dims contiguous)
                    const uint32_t koff = (kk >> 2) * ATOM + (kk & 3) * 32;
                    const uint64_t bd = tc_sdesc_sw128(ka + koff, 16, 1024);
                    tc_mma_bf16(tmem + C::S_COL + sb * KEYS, tc_sdesc_sw128(qa + koff, 16, 1024), bd, idS, kk > 0);
                    if (QF32)
                        tc_mma_bf16(tmem + C::S_COL + sb * KEYS, tc_sdesc_sw128(qa + C::QB + koff, 16, 1024), bd, idS,
                                    true);
                }
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
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, bool QF32>
cudaError_t launch_prefix_t(const PrefixArgs &a, const CUtensorMap *tk, const CUtensorMap *tv, int ctas,
                            cudaStream_t stream) {
    using C = PrefixCfg<D, QF32>;
    auto kernel = prefix_attend_kernel<D, QF32>;
    static bool configured[64] = {false};  // dynamic smem limit set, per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
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

cudaError_t launch_prefix(const PrefixArgs &a, const CUtensorMap *tmap_k, const CUtensorMap *tmap_v, int q_dtype,
                          int head_dim, cudaStream_t stream) {
    const int ctas = prefix_tiles(a.batch, a.group) * a.num_kv_heads * a.splits;
    if (ctas == 0) return cudaSuccess;
    const bool qf = q_dtype == kDtypeF32;
    if (head_dim == 128)
        return qf ? launch_prefix_t<128, true>(a, tmap_k, tmap_v, ctas, stream)
                  : launch_prefix_t<128, false>(a, tmap_k, tmap_v, ctas, stream);
    return qf ? launch_prefix_t<64, true>(a, tmap_k, tmap_v, ctas, stream)
              : launch_prefix_t<64, false>(a, tmap_k, tmap_v, ctas, stream);
}

}  // namespace qskv

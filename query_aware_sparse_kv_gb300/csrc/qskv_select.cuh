// Ranking of one row's page scores by one CTA (the top-K select of
// TinyServe query-aware page selection, s2.3: radix sort in shared memory),
// shared by the ranking kernel (page_select.cu) and the fused rank + decode
// launch (decode.cu); and the bound product of s2.2 on the tensor cores,
// shared by the scoring kernel and the decode launch that scores its own
// rows.  MSB-first radix select over 8-bit digits of
// order-preserving 32-bit keys, stopping early when a bucket is taken whole;
// stable compaction in page order (ties to the lower page index); the lossy
// variant of the Vortex digest (method overview item 3) when a.need_max > 0.
#pragma once

#include "qskv_device.cuh"

namespace qskv {

// fp32 -> unsigned key with the same order; -0 and +0 map to one key.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t shr32(uint32_t x, int s) { return s >= 32 ? 0u : (x >> s); }

// ---------------------------------------------------------- bound score --
// With q- = min(q, 0) and q+ = max(q, 0) the bound of page j is the dot
// product [m_j | M_j] . [q- | q+].  The scores of 16 pages for the G <= 8
// heads of a group are a (16 pages x 2D) . (2D x 8 heads) m16n8k16 bf16
// product with fp32 accumulation.  Lane (gid, t) holds the 16-byte chunks
// 4 kp + t (kp < NKP) of the metadata rows of pages gid and gid + 8 (the A
// operand) and the same chunks of head gid's [q- | q+] column (the B
// operand): A and B use one permutation of the 2D-long k axis, which the dot
// product does not see.  bf16 products are exact in fp32; fp32 queries are
// split into hi + lo bf16 halves (two mma per k-step).
template <int D>
struct BoundScanRegs {
    static constexpr int NKP = 2 * D / 32;  // 16-byte chunks per lane per metadata row
};

// Column of the 2D-long k axis where this lane's chunk c starts in q: the
// first D columns pair m with q-, the next D pair M with q+.
template <int D>
__device__ __forceinline__ int bound_q_col(int c) { return 8 * c - (8 * c >= D ? D : 0); }

// B operand (bh, and the lo halves bl for fp32 q) from the lane's raw query
// chunks qraw[kp] (chunk 4 kp + t of head gid; 8 floats or 8 bf16).
template <int D, bool QF32>
__device__ __forceinline__ void bound_q_operand(const uint4 (&qraw)[2 * D / 32][QF32 ? 2 : 1], bool head_ok,
                                                uint32_t (&bh)[2 * D / 32][4], uint32_t (&bl)[2 * D / 32][4]) {
    constexpr int NKP = BoundScanRegs<D>::NKP;
    const int t = threadIdx.x & 3;
#pragma unroll
    for (int kp = 0; kp < NKP; kp++) {
        const bool upper = 8 * (4 * kp + t) >= D;  // chunk of the M half: pairs with q+
        float v[8];
        if (QF32) {
            const uint4 x0 = qraw[kp][0], x1 = qraw[kp][QF32 ? 1 : 0];
            v[0] = __uint_as_float(x0.x); v[1] = __uint_as_float(x0.y);
            v[2] = __uint_as_float(x0.z); v[3] = __uint_as_float(x0.w);
            v[4] = __uint_as_float(x1.x); v[5] = __uint_as_float(x1.y);
            v[6] = __uint_as_float(x1.z); v[7] = __uint_as_float(x1.w);
        } else {
            const uint4 x = qraw[kp][0];
            v[0] = bf16_lo_to_float(x.x); v[1] = bf16_hi_to_float(x.x);
            v[2] = bf16_lo_to_float(x.y); v[3] = bf16_hi_to_float(x.y);
            v[4] = bf16_lo_to_float(x.z); v[5] = bf16_hi_to_float(x.z);
            v[6] = bf16_lo_to_float(x.w); v[7] = bf16_hi_to_float(x.w);
        }
#pragma unroll
        for (int i = 0; i < 8; i++) {
            v[i] = upper ? fmaxf(v[i], 0.f) : fminf(v[i], 0.f);
            if (!head_ok) v[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 4; i++) {
            bh[kp][i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
            if (QF32) {
                const float r0 = v[2 * i] - bf16_lo_to_float(bh[kp][i]);
                const float r1 = v[2 * i + 1] - bf16_hi_to_float(bh[kp][i]);
                bl[kp][i] = pack_bf16x2(r0, r1);
            }
        }
    }
}

// Row scores of one 16-page group: xa / xb are the lane's chunks of the
// metadata rows of pages gid and gid + 8.  Returns in sa / sb the best head's
// bound of those two pages (valid in the lanes with t = 0).  The k axis is
// summed in four independent accumulator chains (kp even / odd x the two
// halves of a chunk), issued round-robin so consecutive mma do not wait on
// each other, then added pairwise.  Every caller accumulates in this one
// order, so the two scoring paths give equal bits.
template <int D, bool QF32>
__device__ __forceinline__ void bound_group_scores(const uint4 (&xa)[2 * D / 32], const uint4 (&xb)[2 * D / 32],
                                                   const uint32_t (&bh)[2 * D / 32][4],
                                                   const uint32_t (&bl)[2 * D / 32][4], int group, float &sa,
                                                   float &sb) {
    constexpr int NKP = BoundScanRegs<D>::NKP;
    static_assert(NKP % 2 == 0, "chunks come in pairs");
    const int t = threadIdx.x & 3;
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
    float c2[4] = {0.f, 0.f, 0.f, 0.f}, c3[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kp = 0; kp < NKP; kp += 2) {
        const uint32_t a0[4] = {xa[kp].x, xb[kp].x, xa[kp].y, xb[kp].y};
        const uint32_t a1[4] = {xa[kp].z, xb[kp].z, xa[kp].w, xb[kp].w};
        const uint32_t a2[4] = {xa[kp + 1].x, xb[kp + 1].x, xa[kp + 1].y, xb[kp + 1].y};
        const uint32_t a3[4] = {xa[kp + 1].z, xb[kp + 1].z, xa[kp + 1].w, xb[kp + 1].w};
        mma_bf16_16816(c0, a0, bh[kp][0], bh[kp][1]);
        mma_bf16_16816(c1, a1, bh[kp][2], bh[kp][3]);
        mma_bf16_16816(c2, a2, bh[kp + 1][0], bh[kp + 1][1]);
        mma_bf16_16816(c3, a3, bh[kp + 1][2], bh[kp + 1][3]);
        if (QF32) {
            mma_bf16_16816(c0, a0, bl[kp][0], bl[kp][1]);
            mma_bf16_16816(c1, a1, bl[kp][2], bl[kp][3]);
            mma_bf16_16816(c2, a2, bl[kp + 1][0], bl[kp + 1][1]);
            mma_bf16_16816(c3, a3, bl[kp + 1][2], bl[kp + 1][3]);
        }
    }
    float acc[4];
#pragma unroll
    for (int i = 0; i < 4; i++) acc[i] = (c0[i] + c2[i]) + (c1[i] + c3[i]);
    // acc: [page gid][head 2t], [gid][2t+1], [gid+8][2t], [gid+8][2t+1]
    const float NEG = -INFINITY;
    const bool h0 = 2 * t < group, h1 = 2 * t + 1 < group;
    sa = fmaxf(h0 ? acc[0] : NEG, h1 ? acc[1] : NEG);
    sb = fmaxf(h0 ? acc[2] : NEG, h1 ? acc[3] : NEG);
    sa = fmaxf(sa, __shfl_xor_sync(0xffffffffu, sa, 1));
    sa = fmaxf(sa, __shfl_xor_sync(0xffffffffu, sa, 2));
    sb = fmaxf(sb, __shfl_xor_sync(0xffffffffu, sb, 1));
    sb = fmaxf(sb, __shfl_xor_sync(0xffffffffu, sb, 2));
}

// --------------------------------------------------------------- select --
// Exclusive block scans of x and y; total_y gets the sum of y over the block.
template <int NT>
__device__ __forceinline__ void block_exclusive_scan2(int &x, int &y, int &total_y, int *s_tmp /* 2*NT/32 */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int ix = x, iy = y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int tx = __shfl_up_sync(0xffffffffu, ix, o);
        const int ty = __shfl_up_sync(0xffffffffu, iy, o);
        if (lane >= o) {
            ix += tx;
            iy += ty;
        }
    }
    if (lane == 31) {
        s_tmp[warp] = ix;
        s_tmp[NT / 32 + warp] = iy;
    }
    __syncthreads();
    int ox = 0, oy = 0, ty = 0;
    for (int w = 0; w < NT / 32; w++) {
        if (w < warp) {
            ox += s_tmp[w];
            oy += s_tmp[NT / 32 + w];
        }
        ty += s_tmp[NT / 32 + w];
    }
    x = ox + ix - x;
    y = oy + iy - y;
    total_y = ty;
    __syncthreads();
}

// Output i (i >= 1) of SplitMix64 started at `seed` (Steele, Lea and Flood,
// "Fast splittable pseudorandom number generators", 2014), used as a
// counter-based generator: the random start of a row's sample.
__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t i) {
    uint64_t z = seed + i * 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

// Shared memory of select_row: keys[kSelectKeyCap], hist[256], tmp[2 NT/32],
// mm[2 NT/32], pick[3].
struct SelectSmem {
    uint32_t *keys, *hist, *mm;
    int *tmp, *pick;
};

// Ranks one row's scores (all NT threads of the CTA take part) and returns
// how many pages are kept.  The ascending list goes to a.selected (and the
// count to a.n_selected) when write_global, and to s_sel[0 .. top_k) in
// shared memory when s_sel is not null (-1 past the count in both).
template <int NT>
__device__ int select_row(const SelectArgs &a, int row, int n_b, const float *srow, const SelectSmem &sm,
                          int *s_sel, bool write_global) {
    static_assert(NT % 32 == 0 && NT <= 256, "ranking CTAs have at most 256 threads, whole warps");
    constexpr int NW = NT / 32;
    uint32_t *s_keys = sm.keys, *s_hist = sm.hist, *s_mm = sm.mm;
    int *s_tmp = sm.tmp, *s_pick = sm.pick;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.top_k;
    int32_t *sel = a.selected + int64_t(row) * K;
    auto put = [&](int pos, int v) {
        if (write_global) sel[pos] = v;
        if (s_sel) s_sel[pos] = v;
    };

    if (K >= n_b) {  // every page is kept
        for (int i = tid; i < K; i += NT) put(i, i < n_b ? i : -1);
        if (tid == 0 && write_global) a.n_selected[row] = n_b;
        return n_b;
    }
    const bool in_smem = n_b <= kSelectKeyCap;
    auto key_at = [&](int i) -> uint32_t { return in_smem ? s_keys[i] : order_key(__ldcg(srow + i)); };

    uint32_t kmin = 0xffffffffu, kmax = 0u;
    if (in_smem) {
        // all of this thread's scores are requested before any is used
        constexpr int PER = (kSelectKeyCap + NT - 1) / NT;
        float v[PER];
#pragma unroll
        for (int j = 0; j < PER; j++) {
            const int i = tid + j * NT;
            v[j] = i < n_b ? __ldcg(srow + i) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < PER; j++) {
            const int i = tid + j * NT;
            if (i < n_b) {
                const uint32_t k = order_key(v[j]);
                s_keys[i] = k;
                kmin = min(kmin, k);
                kmax = max(kmax, k);
            }
        }
    } else {
        for (int i = tid; i < n_b; i += NT) {
            const uint32_t k = order_key(__ldcg(srow + i));
            kmin = min(kmin, k);
            kmax = max(kmax, k);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
        kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    if (lane == 0) {
        s_mm[warp] = kmin;
        s_mm[NT / 32 + warp] = kmax;
    }
    __syncthreads();
    kmin = s_mm[0];
    kmax = s_mm[NT / 32];
    for (int w = 1; w < NT / 32; w++) {
        kmin = min(kmin, s_mm[w]);
        kmax = max(kmax, s_mm[NT / 32 + w]);
    }

    // Bits at and above `hi` are shared by every key of the row: the passes
    // over digits above them would find one bucket holding every key and
    // decide nothing.  The exact select starts its 8-bit digits right below
    // them (the first pass then splits the row); the lossy select keeps the
    // key's fixed digits (bits 31..24, 23..16, ...), on which its early exit
    // is defined, and only skips the digits shared by every key.
    const uint32_t diff = kmin ^ kmax;
    int hi = diff ? 32 - __clz(diff) : 0;
    if (a.need_max > 0) hi = (hi + 7) & ~7;
    uint32_t prefix = hi >= 32 ? 0u : (kmax & ~((1u << hi) - 1u));
    int need = K;  // keys still to take among those matching `prefix` above `hi`
    int lo = hi;
    while (hi > 0) {
        // lossy early exit: few enough keys are still undecided
        if (a.need_max > 0 && need <= a.need_max) break;
        lo = hi > 8 ? hi - 8 : 0;
        const uint32_t mask = (1u << (hi - lo)) - 1u;
        for (int i = tid; i < 256; i += NT) s_hist[i] = 0u;
        __syncthreads();
        const uint32_t want = shr32(prefix, hi);
        for (int i = tid; i < n_b; i += NT) {
            const uint32_t k = key_at(i);
            if (shr32(k, hi) == want) atomicAdd(&s_hist[(k >> lo) & mask], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            uint32_t h[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                h[j] = s_hist[lane * 8 + j];
                sum += h[j];
            }
            uint32_t suf = sum;  // inclusive suffix sum over lanes >= this one
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += t;
            }
            uint32_t acc = suf - sum;  // keys in higher lanes' bins
#pragma unroll
            for (int j = 7; j >= 0; j--) {
                if (acc < uint32_t(need) && acc + h[j] >= uint32_t(need)) {
                    s_pick[0] = lane * 8 + j;
                    s_pick[1] = int(acc);
                    s_pick[2] = int(h[j]);
                }
                acc += h[j];
            }
        }
        __syncthreads();
        const int bin = s_pick[0], above = s_pick[1], cnt = s_pick[2];
        prefix |= uint32_t(bin) << lo;
        need -= above;
        __syncthreads();
        if (cnt == need) break;  // the whole bucket is taken: no tie to cut
        hi = lo;
    }

    // Stable compaction in page order: every key above the threshold bucket,
    // and `need` of the bucket's m keys.  Exact rule: the first `need` in
    // page order.  After a lossy early exit: bucket key t (0-based, page
    // order) is kept iff c(t + 1) - c(t) = 1 with c(t) = (t need + o) / m
    // (integer division; o = a SplitMix64 draw mod m): systematic sampling
    // with a random start, every bucket key kept with probability need / m.
    // Either way c(t) keys of the bucket precede bucket key t in the output.
    if (n_b <= kSelectBallotKeys) {
        // Warp w walks the contiguous keys [w0, w1) 32 at a time; ballot
        // prefix counts give key i's gi / ei (keys above / in the bucket
        // before it).  Measured faster than the per-thread runs below on
        // rows of up to 2048 keys, slower on longer ones.
        const uint32_t thr = shr32(prefix, lo);
        const uint32_t lt = (1u << lane) - 1u;
        const int cw = ((n_b + NW - 1) / NW + 31) & ~31;
        const int w0 = min(warp * cw, n_b), w1 = min(w0 + cw, n_b);
        int cg = 0, ce = 0;
        for (int base = w0; base < w1; base += 32) {
            const int i = base + lane;
            const uint32_t k = i < w1 ? shr32(key_at(i), lo) : 0u;
            cg += __popc(__ballot_sync(0xffffffffu, i < w1 && k > thr));
            ce += __popc(__ballot_sync(0xffffffffu, i < w1 && k == thr));
        }
        if (lane == 0) {
            s_tmp[warp] = cg;
            s_tmp[NW + warp] = ce;
        }
        __syncthreads();
        int gb = 0, eb = 0, m = 0;
        for (int w = 0; w < NW; w++) {
            if (w < warp) {
                gb += s_tmp[w];
                eb += s_tmp[NW + w];
            }
            m += s_tmp[NW + w];
        }
        const bool sampled = a.need_max > 0 && need < m;
        // t need + o < m (need + 1) < 2^32 here
        const uint32_t o = sampled ? uint32_t(splitmix64(a.seed, uint64_t(row) + 1u) % uint64_t(m)) : 0u;
        const int n_gt = K - need;               // keys above the bucket
        const int eq_last = sampled ? m : need;  // bucket keys to walk past
        for (int base = w0; base < w1; base += 32) {
            if (gb >= n_gt && eb >= eq_last) break;  // every kept key is placed
            const int i = base + lane;
            const uint32_t k = i < w1 ? shr32(key_at(i), lo) : 0u;
            const bool gt = i < w1 && k > thr, eq = i < w1 && k == thr;
            const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
            const int gi = gb + __popc(bg & lt), ei = eb + __popc(be & lt);
            if (!sampled) {
                if (gt) {
                    const int pos = gi + min(ei, need);
                    if (pos < K) put(pos, i);
                } else if (eq && ei < need && gi + ei < K) {
                    put(gi + ei, i);
                }
            } else {
                const uint32_t x = uint32_t(ei) * uint32_t(need) + o;
                const int c = int(x / uint32_t(m));
                if (gt) {
                    if (gi + c < K) put(gi + c, i);
                } else if (eq && int((x + uint32_t(need)) / uint32_t(m)) != c && gi + c < K) {
                    put(gi + c, i);
                }
            }
            gb += __popc(bg);
            eb += __popc(be);
        }
    } else {
        // thread t walks the keys [t per, (t + 1) per); an odd run length
        // puts the 32 lanes' reads of one step in 32 different banks
        const uint32_t thr = shr32(prefix, lo);
        const int per = ((n_b + NT - 1) / NT) | 1;
        const int i0 = min(tid * per, n_b), i1 = min(i0 + per, n_b);
        int cg = 0, ce = 0;
        for (int i = i0; i < i1; i++) {
            const uint32_t k = shr32(key_at(i), lo);
            cg += k > thr;
            ce += k == thr;
        }
        int gb = cg, eb = ce, m = 0;
        block_exclusive_scan2<NT>(gb, eb, m, s_tmp);
        const bool sampled = a.need_max > 0 && need < m;
        if (!sampled) {
            for (int i = i0; i < i1; i++) {
                const uint32_t k = shr32(key_at(i), lo);
                if (k > thr) {
                    const int pos = gb + min(eb, need);
                    if (pos < K) put(pos, i);
                    gb++;
                } else if (k == thr) {
                    if (eb < need && gb + eb < K) put(gb + eb, i);
                    eb++;
                }
            }
        } else {
            // c(t) and the remainder of (t need + o) by m, stepped per bucket key
            // (t need + o < m (need + 1) < 2^32 for rows held in shared memory)
            const uint64_t o = splitmix64(a.seed, uint64_t(row) + 1u) % uint64_t(m);
            const uint64_t x = uint64_t(eb) * uint64_t(need) + o;
            int c = int(x / uint64_t(m));
            int rem = int(x - uint64_t(c) * uint64_t(m));
            for (int i = i0; i < i1; i++) {
                const uint32_t k = shr32(key_at(i), lo);
                if (k > thr) {
                    const int pos = gb + c;
                    if (pos < K) put(pos, i);
                    gb++;
                } else if (k == thr) {
                    rem += need;
                    if (rem >= m) {  // c(t + 1) = c(t) + 1: this key is kept
                        rem -= m;
                        if (gb + c < K) put(gb + c, i);
                        c++;
                    }
                }
            }
        }
    }
    if (tid == 0 && write_global) a.n_selected[row] = K;
    return K;
}

}  // namespace qskv

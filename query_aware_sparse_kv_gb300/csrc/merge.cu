// Log-sum-exp merge of split decode rows (Quail AI-SQL engine article:
// partial attention results combined by log-sum-exp rescaling, as in flash
// decoding; CS336 Lecture 10 s9.2, FlashDecoding).
//
// Row `row` was split over decode warps w0..w1; warp w left a normalised
// partial o_w and its log2-domain log-sum-exp in slot row + w.  Another
// kernel may have left extra_pieces more in slots extra_slot0 + row *
// extra_pieces + e (the shared-prefix part of a cascade decode).  With
// m = max_w lse_w:
//   out = sum_w 2^(lse_w - m) o_w / sum_w 2^(lse_w - m)
//   lse = (m + log2 sum_w 2^(lse_w - m)) * ln 2
// One CTA per row.  Its threads form `groups` copies of the row's G x D/4
// float4 columns; copy k folds pieces k, k + groups, ... with a running
// maximum (eight pieces' loads in flight per thread), and the copies are
// combined the same way through shared memory.  The host picks `groups`
// from the largest piece count a row can have, so rows split over many
// warps (long sequences, few rows) are folded by many threads.  Rows a
// single warp covered alone were finished by that warp.
#include "qskv_device.cuh"
#include "qskv_internal.h"

namespace qskv {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMergeMaxThreads = 1024;

struct Fold {
    float mx, den;
    float4 acc;
};

// Folds pieces first, first + stride, ... < n of one contiguous slot range
// (lse_p / o_p point at this thread's column of the range's first slot).
template <int SC>
__device__ __forceinline__ void fold_range(Fold &f, const float *lse_p, const float4 *o_p, int n, int first,
                                           int stride, int lse_step, int o_step) {
    for (int s0 = first; s0 < n; s0 += SC * stride) {
        float l[SC];
        float4 v[SC];
#pragma unroll
        for (int j = 0; j < SC; j++) {
            const int sidx = s0 + j * stride;
            const bool ok = sidx < n;
            // o is loaded with its lse (one round trip); an empty piece's o
            // (never written) is loaded too but not used
            l[j] = ok ? __ldcg(lse_p + int64_t(sidx) * lse_step) : -INFINITY;
            v[j] = ok ? __ldcg(o_p + int64_t(sidx) * o_step) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float m = f.mx;
#pragma unroll
        for (int j = 0; j < SC; j++) m = fmaxf(m, l[j]);
        if (m == -INFINITY) continue;
        const float sc = exp2f(f.mx - m);
        f.den *= sc;
        f.acc.x *= sc;
        f.acc.y *= sc;
        f.acc.z *= sc;
        f.acc.w *= sc;
#pragma unroll
        for (int j = 0; j < SC; j++) {
            if (l[j] == -INFINITY) continue;  // an empty piece: its o holds no data
            const float w = exp2f(l[j] - m);
            f.den += w;
            f.acc.x = fmaf(w, v[j].x, f.acc.x);
            f.acc.y = fmaf(w, v[j].y, f.acc.y);
            f.acc.z = fmaf(w, v[j].z, f.acc.z);
            f.acc.w = fmaf(w, v[j].w, f.acc.w);
        }
        f.mx = m;
    }
}

template <int D>
__global__ void __launch_bounds__(kMergeMaxThreads) merge_partials_kernel(DecodeArgs a, int groups) {
    extern __shared__ float4 s_red[];  // [groups][cols] acc, then mx / den as float2 pairs
    pdl_trigger();
    pdl_wait();
    const int row = blockIdx.x;
    int64_t w0, w1;
    row_warps(a, row, w0, w1);
    if (row_is_final(a, w0, w1)) return;
    constexpr int V4 = D / 4;
    const int G = a.group;
    const int cols = G * V4;
    const int b = row / a.num_kv_heads, g = row % a.num_kv_heads;
    const int nd = int(w1 - w0 + 1);  // pieces from decode warps: slots row + w0 ..
    const int ne = a.extra_pieces;    // pieces from another kernel: slots extra_slot0 + row * ne ..
    const int64_t slot_d = row + w0, slot_e = a.extra_slot0 + int64_t(row) * ne;
    const float4 *o_all = reinterpret_cast<const float4 *>(a.part_o);
    const int col = threadIdx.x % cols, grp = threadIdx.x / cols;
    const int h = col / V4;

    Fold f{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
    if (grp < groups) {
        fold_range<8>(f, a.part_lse + slot_d * G + h, o_all + slot_d * cols + col, nd, grp, groups, G, cols);
        if (ne > 0)
            fold_range<8>(f, a.part_lse + slot_e * G + h, o_all + slot_e * cols + col, ne, grp, groups, G, cols);
    }
    if (groups > 1) {
        float2 *s_md = reinterpret_cast<float2 *>(s_red + groups * cols);
        if (grp < groups) {
            s_red[grp * cols + col] = f.acc;
            s_md[grp * cols + col] = make_float2(f.mx, f.den);
        }
        __syncthreads();
        if (grp != 0) return;
        float m = -INFINITY;
        for (int k = 0; k < groups; k++) m = fmaxf(m, s_md[k * cols + col].x);
        f = Fold{m, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
        if (m != -INFINITY) {
            for (int k = 0; k < groups; k++) {
                const float2 md = s_md[k * cols + col];
                if (md.x == -INFINITY) continue;
                const float w = exp2f(md.x - m);
                const float4 ac = s_red[k * cols + col];
                f.den = fmaf(w, md.y, f.den);
                f.acc.x = fmaf(w, ac.x, f.acc.x);
                f.acc.y = fmaf(w, ac.y, f.acc.y);
                f.acc.z = fmaf(w, ac.z, f.acc.z);
                f.acc.w = fmaf(w, ac.w, f.acc.w);
            }
        }
    } else if (grp != 0) {
        return;
    }
    const int64_t qh0 = int64_t(b) * a.num_q_heads + int64_t(g) * G;
    const int c4 = col % V4;
    const float inv = f.den > 0.f ? 1.f / f.den : 0.f;
    reinterpret_cast<float4 *>(a.out + (qh0 + h) * D)[c4] =
        make_float4(f.acc.x * inv, f.acc.y * inv, f.acc.z * inv, f.acc.w * inv);
    if (c4 == 0 && a.lse) a.lse[qh0 + h] = f.den > 0.f ? (f.mx + log2f(f.den)) * kLn2 : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const DecodeArgs &a, int head_dim, cudaStream_t stream) {
    // the most pieces a row can have: the warps its slots span, plus the
    // other kernel's pieces; about eight per thread
    const int64_t upw = a.units_per_warp > 0 ? a.units_per_warp : 1;
    const int64_t spr = a.total_units > 0 ? a.slots_per_row : 0;
    const int64_t pieces = (spr + upw - 1) / upw + 1 + a.extra_pieces;
    const int cols = a.group * head_dim / 4;
    int groups = int((pieces + 7) / 8);
    groups = groups < 1 ? 1 : (groups > kMergeMaxThreads / cols ? kMergeMaxThreads / cols : groups);
    const int threads = (cols * groups + 31) / 32 * 32;
    const size_t smem = groups > 1 ? size_t(groups) * cols * (sizeof(float4) + sizeof(float2)) : 0;
    const dim3 g(unsigned(int64_t(a.batch) * a.num_kv_heads));
    const dim3 b(static_cast<unsigned>(threads));
    return head_dim == 128 ? launch_pdl(merge_partials_kernel<128>, g, b, smem, stream, a, groups)
                           : launch_pdl(merge_partials_kernel<64>, g, b, smem, stream, a, groups);
}

}  // namespace qskv

// Per-page min/max key metadata (TinyServe query-aware page selection, s2.1:
// for every page the element-wise minimum m_j and maximum M_j of its key
// vectors, 2d values per page; refreshed every decode step, s5.3).
//
// One warp per (listed page, KV head) tile of P x D keys.  Lanes read the
// tile in 16-byte vectors, row-interleaved so a warp instruction covers whole
// 128-byte lines; each lane keeps an element-wise running min and max of its
// vector column, lanes holding the same column combine by shuffles, and the
// two rows (min, max) are written back as 16-byte vectors.  Min/max are
// exact, so the result is bit-identical to any other evaluation order (up to
// the sign of zero).  Only tokens t < valid_tokens are read.
#include "qskv_device.cuh"
#include "qskv_internal.h"

namespace qskv {
namespace {

// ROW_BYTES = D * element size.
template <class Ops, int ROW_BYTES>
__global__ void __launch_bounds__(256) meta_build_kernel(MetaArgs a) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t tile = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (tile >= int64_t(a.n_list) * a.num_kv_heads) return;
    const int e = int(tile / a.num_kv_heads);
    const int g = int(tile % a.num_kv_heads);
    const int p = a.page_ids[e];
    const int valid = a.valid_tokens[e];
    if (p < 0 || p >= a.num_pool_pages) {
        if (lane == 0) raise_error(a.flags, kErrPageId);
        return;
    }
    if (valid < 1 || valid > a.page_size) {
        if (lane == 0) raise_error(a.flags, kErrValid);
        return;
    }
    meta_tile_warp<Ops, ROW_BYTES>(a.k_pool, a.meta, p, g, valid, a.num_kv_heads, a.page_size);
}

// Block summary for the Block Top-K scorer (Vortex sparse-attention digest,
// method overview item 1: the cache phase keeps each block's mean key).  One
// warp per (listed page, KV head): lanes read the tile in 16-byte vectors,
// row-interleaved as above, and keep fp32 running sums of their vector
// column; lanes holding the same column add by shuffles (a fixed order), and
// the mean (sum / valid) is written as fp32 [Npool][Hkv][D].
template <bool BF16, int ROW_BYTES>
__global__ void __launch_bounds__(256) centroid_build_kernel(MetaArgs a) {
    constexpr int CPR = ROW_BYTES / 16;
    constexpr int RP = 32 / CPR;
    constexpr int EPC = BF16 ? 8 : 4;                   // elements per 16-byte chunk
    constexpr int D = ROW_BYTES / (BF16 ? 2 : 4);
    static_assert(CPR >= 1 && CPR <= 32 && 32 % CPR == 0, "row must be 16..512 bytes");
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t tile = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (tile >= int64_t(a.n_list) * a.num_kv_heads) return;
    const int e = int(tile / a.num_kv_heads);
    const int g = int(tile % a.num_kv_heads);
    const int p = a.page_ids[e];
    const int valid = a.valid_tokens[e];
    if (p < 0 || p >= a.num_pool_pages) {
        if (lane == 0) raise_error(a.flags, kErrPageId);
        return;
    }
    if (valid < 1 || valid > a.page_size) {
        if (lane == 0) raise_error(a.flags, kErrValid);
        return;
    }
    const int c = lane % CPR;
    const int r0 = lane / CPR;
    const uint8_t *base =
        static_cast<const uint8_t *>(a.k_pool) + ((int64_t(p) * a.num_kv_heads + g) * a.page_size) * ROW_BYTES;
    constexpr int ITER = 32 / RP;  // P <= 32
    uint4 v[ITER];
#pragma unroll
    for (int i = 0; i < ITER; i++) {
        const int r = r0 + i * RP;
        v[i] = r < valid ? ldg_stream_v4(base + int64_t(r) * ROW_BYTES + c * 16) : make_uint4(0, 0, 0, 0);
    }
    float acc[EPC];
#pragma unroll
    for (int k = 0; k < EPC; k++) acc[k] = 0.f;
#pragma unroll
    for (int i = 0; i < ITER; i++) {
        if (r0 + i * RP >= valid) continue;
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; k++) {
            if (BF16) {
                acc[2 * k] += __uint_as_float(w[k] << 16);
                acc[2 * k + 1] += __uint_as_float(w[k] & 0xffff0000u);
            } else {
                acc[k] += __uint_as_float(w[k]);
            }
        }
    }
#pragma unroll
    for (int off = CPR; off < 32; off <<= 1)
#pragma unroll
        for (int k = 0; k < EPC; k++) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
    if (r0 == 0) {
        float *out = static_cast<float *>(a.meta) + (int64_t(p) * a.num_kv_heads + g) * D + c * EPC;
        const float n = float(valid);
#pragma unroll
        for (int k = 0; k < EPC; k += 4)
            *reinterpret_cast<float4 *>(out + k) =
                make_float4(acc[k] / n, acc[k + 1] / n, acc[k + 2] / n, acc[k + 3] / n);
    }
}

}  // namespace

cudaError_t launch_centroid_build(const MetaArgs &a, int kv_dtype, int head_dim, cudaStream_t stream) {
    const int64_t tiles = int64_t(a.n_list) * a.num_kv_heads;
    if (tiles == 0) return cudaSuccess;
    const int warps = 8;
    const dim3 grid(unsigned((tiles + warps - 1) / warps));
    const dim3 block(32 * warps);
    if (kv_dtype == kDtypeBf16)
        return head_dim == 128 ? launch_pdl(centroid_build_kernel<true, 256>, grid, block, 0, stream, a)
                               : launch_pdl(centroid_build_kernel<true, 128>, grid, block, 0, stream, a);
    return head_dim == 128 ? launch_pdl(centroid_build_kernel<false, 512>, grid, block, 0, stream, a)
                           : launch_pdl(centroid_build_kernel<false, 256>, grid, block, 0, stream, a);
}

cudaError_t launch_meta_build(const MetaArgs &a, int kv_dtype, int head_dim, cudaStream_t stream) {
    const int64_t tiles = int64_t(a.n_list) * a.num_kv_heads;
    if (tiles == 0) return cudaSuccess;
    const int warps = 8;
    const dim3 grid(unsigned((tiles + warps - 1) / warps));
    const dim3 block(32 * warps);
    if (kv_dtype == kDtypeBf16)
        return head_dim == 128 ? launch_pdl(meta_build_kernel<Bf16Ops, 256>, grid, block, 0, stream, a)
                               : launch_pdl(meta_build_kernel<Bf16Ops, 128>, grid, block, 0, stream, a);
    return head_dim == 128 ? launch_pdl(meta_build_kernel<F32Ops, 512>, grid, block, 0, stream, a)
                           : launch_pdl(meta_build_kernel<F32Ops, 256>, grid, block, 0, stream, a);
}

}  // namespace qskv

// Device-side helpers shared by the qskv kernels: error flags, inline-PTX
// wrappers for mbarrier / TMA / ldmatrix / mma.sync / movmatrix, and the
// argument blocks the host passes to each kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qskv {

// ----------------------------------------------------------------- errors --
// Bits of the device error word at the head of the workspace.
enum : uint32_t {
    kErrPageId = 1u,    // page-table entry or listed page outside [0, num_pool_pages)
    kErrSelected = 2u,  // selected index outside [0, n_b) or n_selected out of range
    kErrSeqLen = 4u,    // seq_len < 0 or > max_pages * page_size
    kErrValid = 8u,     // valid-token count outside [1, page_size]
    kErrTimeout = 16u,  // a bounded mbarrier wait gave up
};

// A wait on a TMA transfer that has not completed after this long is treated
// as lost: the kernel flags kErrTimeout and abandons its remaining work.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void raise_error(uint32_t *flags, uint32_t bit) { atomicOr(flags, bit); }

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// --------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------- programmatic dependent launch --
// Every kernel is launched with programmatic stream serialization, so it may
// start while the previous kernel in the stream drains.  pdl_wait() blocks
// until that kernel has completed and its writes are visible; no kernel
// touches global memory before it.  pdl_trigger() lets the next kernel in
// the stream begin its own launch early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

#ifdef __CUDACC__
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
#endif

// ------------------------------------------------------------------- TMA --
// 2-D tiled bulk tensor load into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int32_t x, int32_t y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------ warp matrix ops --
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// D(16x8, fp32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transposes an 8x8 b16 matrix held one fragment register per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Two floats -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo_to_float(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi_to_float(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// 16-byte read-only global load that skips L1 allocation (streamed data).
__device__ __forceinline__ uint4 ldg_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------- kernel arguments --
struct MetaArgs {
    const void *k_pool;
    const int32_t *page_ids;
    const int32_t *valid_tokens;
    void *meta;
    uint32_t *flags;
    int32_t n_list, num_kv_heads, page_size, num_pool_pages;
};

struct SelectArgs {
    const void *q;          // [B][Hq][D]
    const void *meta;       // [Npool][Hkv][2][D]
    const int32_t *page_table;
    const int32_t *seq_lens;
    int32_t *selected;      // [rows][top_k]
    int32_t *n_selected;    // [rows]
    float *scores;          // [rows][max_pages]
    uint32_t *flags;
    int32_t batch, num_q_heads, num_kv_heads, group, page_size, max_pages, num_pool_pages, top_k;
};

struct DecodeArgs {
    const void *q;          // [B][Hq][D]
    const void *k_pool;     // [Npool][Hkv][P][D]   (used by the SIMT kernel)
    const void *v_pool;
    const int32_t *page_table;
    const int32_t *seq_lens;
    const int32_t *selected;   // [rows][top_k] or nullptr (all pages)
    const int32_t *n_selected; // [rows]
    float *out;             // [B][Hq][D]
    float *lse;             // [B][Hq] or nullptr
    float *part_o;          // [slots][G][D]
    float *part_lse;        // [slots][G], log2 domain
    uint32_t *flags;
    int32_t batch, num_q_heads, num_kv_heads, group, page_size, max_pages, num_pool_pages, top_k;
    int32_t slots_per_row;  // top_k (sparse) or max_pages (dense)
    int32_t stages;
    int64_t total_units;    // rows * slots_per_row
    int64_t units_per_warp; // ceil(total_units / total_warps)
    float scale_log2;       // sm_scale * log2(e)
};

constexpr int kScoreThreads = 128;    // scoring CTA: 4 warps x 32 pages
constexpr int kSelectThreads = 256;   // ranking CTA: one row
constexpr int kSelectKeyCap = 4096;   // keys held in shared memory by the select stage
constexpr int kDecodeCtasPerSm = 2;   // decode grid = this x SM count
// Decode pipeline shape per head dim: warps per CTA, 16-token halves per
// stage, stages per warp (2 CTAs x warps x stages x stage bytes <= 227 KB).
#ifndef QSKV_D128_WARPS
#define QSKV_D128_WARPS 6
#define QSKV_D128_HALVES 1
#define QSKV_D128_STAGES 2
#endif
#ifndef QSKV_D64_WARPS
#define QSKV_D64_WARPS 6
#define QSKV_D64_HALVES 2
#define QSKV_D64_STAGES 2
#endif
constexpr int kDecodeWarpsD128 = QSKV_D128_WARPS, kDecodeHalvesD128 = QSKV_D128_HALVES,
              kDecodeStagesD128 = QSKV_D128_STAGES;
constexpr int kDecodeWarpsD64 = QSKV_D64_WARPS, kDecodeHalvesD64 = QSKV_D64_HALVES,
              kDecodeStagesD64 = QSKV_D64_STAGES;
constexpr int kMaxStages = 8;

}  // namespace qskv

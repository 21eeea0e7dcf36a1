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
    kErrPrefix = 32u,   // a row breaks the shared-prefix contract of the cascade decode
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

// Invalidates an mbarrier with no pending arrivals so that it can be initialised again.
__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
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

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// 16-byte asynchronous copy global -> shared through L2 (not L1), and the
// wait for every copy this thread issued.
__device__ __forceinline__ void cp_async_cg16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Barrier over every thread of the thread-block cluster: the release /
// acquire pair makes each CTA's earlier memory writes (global included)
// visible to the other CTAs of the cluster after it.  All threads of every
// CTA of the cluster execute it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------- programmatic dependent launch --
// Every kernel is launched with programmatic stream serialization, so it may
// start while the previous kernel in the stream drains.  pdl_wait() blocks
// until that kernel has completed and its writes are visible; no kernel
// touches global memory before it.  pdl_trigger() lets the next kernel in
// the stream begin its own launch early; single-wave grids call it at entry,
// the multi-wave scoring grids do not (their dependents would take SM
// resources from their later waves).
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

// launch_pdl with the CTAs grouped into thread-block clusters of
// `cluster` consecutive blocks (1: no cluster).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t stream, unsigned cluster, Args... args) {
    if (cluster <= 1) return launch_pdl(kernel, grid, block, smem, stream, args...);
    if (grid.x % cluster != 0) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
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

// L2 policy for data read once per step (the KV stream of the decode, the
// page metadata of the scan): its lines are evicted first, so the stream
// does not push out of L2 the small buffers the next kernel reads (scores,
// split partials, page tables).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}


// tma_load_2d with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int32_t x, int32_t y,
                                                 uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Asks L2 to fetch `bytes` (a multiple of 16) at a 16-byte aligned global address.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------ tcgen05 tensor cores --
// One CTA (cta_group::1).  Tensor memory (TMEM) is 128 lanes x 512 columns
// of 32 bits per SM; an address is lane << 16 | column.  Warp w of a CTA may
// read and write lanes 32 (w % 4) .. 32 (w % 4) + 31 only.

// Allocates `ncols` TMEM columns (a power of two >= 32) for the CTA and
// stores the base address at `dst`.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Frees an allocation; executed by the warp that made it, after every
// tensor-core operation on it has completed.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tcgen05 operations against thread synchronisation (mbarrier or
// bar.sync): "before" ahead of the signalling side, "after" behind the
// waiting side.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Instruction descriptor of a dense kind::f16 MMA with bf16 A and B and an
// fp32 accumulator: M x N tile, A / B either K-major or MN-major in shared
// memory.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4)                         // D: fp32
           | (1u << 7) | (1u << 10)          // A, B: bf16
           | (uint32_t(a_mn_major) << 15) | (uint32_t(b_mn_major) << 16) |
           (uint32_t(N >> 3) << 17)          // N / 8
           | (uint32_t(M >> 4) << 24);       // M / 16
}

// Shared-memory matrix descriptor for the 128-byte swizzled layout (rows of
// 128 bytes, 8-row / 1024-byte swizzle atoms whose base is 1024-aligned).
// K-major operand: `sbo` = bytes between 8-row groups, `lbo` unused.
// MN-major operand: `lbo` = bytes between 64-element groups along M/N,
// `sbo` = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t tc_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46)  // descriptor version
           | (uint64_t(2) << 61);                                          // 128-byte swizzle
}

// D[tmem] (+)= A[smem] . B[smem]^T, issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
        : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T, issued by one thread: A is M x 16 bf16
// elements held in TMEM lanes 0..M-1, two per 32-bit column, K-ascending.
__device__ __forceinline__ void tc_mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
        : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued
// before it has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive columns of this thread's TMEM lane -> registers, waited
// for before returning.  Warp-collective.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Registers -> 32 consecutive columns of this thread's TMEM lane, waited for
// before returning.  Warp-collective.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Named barrier over `count` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also returns whether `pred` held on any participant.
__device__ __forceinline__ bool named_bar_any(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
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

// 8-byte streaming load with an L2 cache policy.
__device__ __forceinline__ uint2 ldg_stream_v2_hint(const void *p, uint64_t policy) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0, %1}, [%2], %3;"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p), "l"(policy));
    return v;
}

// ldg_stream_v4 with an L2 cache policy.
__device__ __forceinline__ uint4 ldg_stream_v4_hint(const void *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

// ------------------------------------------- element-wise min / max of keys --
// The metadata of a page is the element-wise min and max of its key rows
// (exact in the KV dtype); these are the operations every kernel that builds
// it uses, so the results agree bit for bit.
struct Bf16Ops {
    using vec = uint4;  // 8 bf16
    static __device__ __forceinline__ vec lowest() {
        const uint32_t w = 0xff80ff80u;  // -inf, -inf
        return make_uint4(w, w, w, w);
    }
    static __device__ __forceinline__ vec highest() {
        const uint32_t w = 0x7f807f80u;  // +inf, +inf
        return make_uint4(w, w, w, w);
    }
    static __device__ __forceinline__ uint32_t vmin(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hmin2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
    static __device__ __forceinline__ uint32_t vmax(uint32_t a, uint32_t b) {
        __nv_bfloat162 r = __hmax2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
};

struct F32Ops {
    using vec = uint4;  // 4 fp32
    static __device__ __forceinline__ vec lowest() {
        const uint32_t w = 0xff800000u;
        return make_uint4(w, w, w, w);
    }
    static __device__ __forceinline__ vec highest() {
        const uint32_t w = 0x7f800000u;
        return make_uint4(w, w, w, w);
    }
    static __device__ __forceinline__ uint32_t vmin(uint32_t a, uint32_t b) {
        return __float_as_uint(fminf(__uint_as_float(a), __uint_as_float(b)));
    }
    static __device__ __forceinline__ uint32_t vmax(uint32_t a, uint32_t b) {
        return __float_as_uint(fmaxf(__uint_as_float(a), __uint_as_float(b)));
    }
};

template <class Ops>
__device__ __forceinline__ uint4 vmin4(uint4 a, uint4 b) {
    return make_uint4(Ops::vmin(a.x, b.x), Ops::vmin(a.y, b.y), Ops::vmin(a.z, b.z), Ops::vmin(a.w, b.w));
}
template <class Ops>
__device__ __forceinline__ uint4 vmax4(uint4 a, uint4 b) {
    return make_uint4(Ops::vmax(a.x, b.x), Ops::vmax(a.y, b.y), Ops::vmax(a.z, b.z), Ops::vmax(a.w, b.w));
}

__device__ __forceinline__ uint4 shfl_xor4(uint4 v, int m) {
    return make_uint4(__shfl_xor_sync(0xffffffffu, v.x, m), __shfl_xor_sync(0xffffffffu, v.y, m),
                      __shfl_xor_sync(0xffffffffu, v.z, m), __shfl_xor_sync(0xffffffffu, v.w, m));
}

// Metadata of one (page p, KV head g) tile with one warp: meta[p][g][0] =
// element-wise min, meta[p][g][1] = max over the key rows t < valid.  Lanes
// read the tile in 16-byte vectors, row-interleaved so a warp instruction
// covers whole 128-byte lines (every row load of a lane issued before any is
// used, page_size <= 32); each lane keeps a running min and max of its
// vector column, lanes holding the same column combine by shuffles, and the
// two rows are written as 16-byte vectors.  Min / max are exact, so any
// evaluation order gives the same bits (up to the sign of zero).
// TO_SMEM: the two rows also go to srow in shared memory, 16-byte chunk c of
// the [m | M] row at chunk position c ^ swz.
template <class Ops, int ROW_BYTES, bool TO_SMEM = false>
__device__ __forceinline__ void meta_tile_warp(const void *k_pool, void *meta, int p, int g, int valid,
                                               int num_kv_heads, int page_size, uint8_t *srow = nullptr,
                                               int swz = 0) {
    constexpr int CPR = ROW_BYTES / 16;  // 16-byte chunks per token row
    constexpr int RP = 32 / CPR;         // token rows read in parallel by one warp
    static_assert(CPR >= 1 && CPR <= 32 && 32 % CPR == 0, "row must be 16..512 bytes");
    const int lane = threadIdx.x & 31;
    const int c = lane % CPR;
    const int r0 = lane / CPR;
    const uint8_t *base =
        static_cast<const uint8_t *>(k_pool) + ((int64_t(p) * num_kv_heads + g) * page_size) * ROW_BYTES;
    constexpr int ITER = 32 / RP;
    uint4 v[ITER];
#pragma unroll
    for (int i = 0; i < ITER; i++) {
        const int r = r0 + i * RP;
        v[i] = r < valid ? ldg_stream_v4(base + int64_t(r) * ROW_BYTES + c * 16) : Ops::highest();
    }
    uint4 mn = Ops::highest(), mx = Ops::lowest();
#pragma unroll
    for (int i = 0; i < ITER; i++) {
        if (r0 + i * RP < valid) {
            mn = vmin4<Ops>(mn, v[i]);
            mx = vmax4<Ops>(mx, v[i]);
        }
    }
#pragma unroll
    for (int off = CPR; off < 32; off <<= 1) {
        mn = vmin4<Ops>(mn, shfl_xor4(mn, off));
        mx = vmax4<Ops>(mx, shfl_xor4(mx, off));
    }
    uint8_t *out = static_cast<uint8_t *>(meta) + (int64_t(p) * num_kv_heads + g) * 2 * ROW_BYTES;
    if (r0 == 0) *reinterpret_cast<uint4 *>(out + c * 16) = mn;
    if (r0 == (RP > 1 ? 1 : 0)) *reinterpret_cast<uint4 *>(out + ROW_BYTES + c * 16) = mx;
    if constexpr (TO_SMEM) {
        if (r0 == 0) *reinterpret_cast<uint4 *>(srow + ((c ^ swz) << 4)) = mn;
        if (r0 == (RP > 1 ? 1 : 0)) *reinterpret_cast<uint4 *>(srow + (((CPR + c) ^ swz) << 4)) = mx;
    }
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
    const void *k_pool;     // [Npool][Hkv][P][D] (metadata refresh of the last pages only)
    void *meta_w;           // = meta, written by the refresh of the last pages
    const int32_t *page_table;
    const int32_t *seq_lens;
    int32_t *selected;      // [rows][top_k]
    int32_t *n_selected;    // [rows]
    float *scores;          // [rows][max_pages]
    uint32_t *flags;
    int32_t batch, num_q_heads, num_kv_heads, group, page_size, max_pages, num_pool_pages, top_k;
    int32_t need_max;       // lossy top-K: stop refining once <= need_max keys are undecided (0: exact)
    uint64_t seed;          // lossy top-K: seed of the sample's random start
    int32_t meta_evict_first;  // 1: the metadata scan exceeds L2, read it evict-first
    int32_t head_quads;     // bound scan: > 0 selects the head-major grid (num_kv_heads / 4)
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
    int32_t slots_per_row;  // top_k (sparse) or max_pages - page_begin (dense)
    int32_t page_begin;     // dense: slot s is logical page page_begin + s
    int32_t extra_pieces;   // partials per row written by another kernel (0: none)
    int64_t extra_slot0;    // row r's extra piece e sits in slot extra_slot0 + r * extra_pieces + e
    int32_t wait_at_exit;   // 1: wait for the previous grid at exit, not before the first access
    int32_t kv_evict_first; // 1: this call's K/V stream exceeds L2, read it evict-first
                            // (the previous grid is the cascade's prefix kernel, which itself
                            // waited for everything before it)
    int32_t stages;
    uint32_t *tickets;      // [rows] per-row counters of the in-grid fold (zero between calls)
    int32_t fold;           // 1: split rows are folded by their last warp (no merge kernel)
    int64_t total_units;    // rows * slots_per_row
    int64_t units_per_warp; // ceil(total_units / total_warps)
    float scale_log2;       // sm_scale * log2(e)
    int32_t row_blocks = 1; // one-row-per-CTA decode: CTAs per row (1: the CTA finishes the row)
    int32_t pt_in_smem = 0; // one-row-per-CTA decode: the row's page-table entries are staged in
                            // shared memory before the wait for the previous kernel
    // Fused rank + decode (one row per k CTAs): each CTA first ranks its row's
    // `scores` (top_k, exact) itself; block 0 of the row writes the list and
    // count to selected_out / n_selected_out.
    float *scores = nullptr;
    int32_t *selected_out = nullptr;
    int32_t *n_selected_out = nullptr;
    // Fused score + rank + decode (one row per k CTAs, the k CTAs of a row
    // one thread-block cluster): each CTA first scores its share of the
    // row's pages from `meta` into `scores` (all rows when score_all, else
    // only rows with more pages than top_k), after the last CTA of the row
    // has recomputed the last page's metadata into meta_w when `refresh`.
    const void *meta = nullptr;
    void *meta_w = nullptr;
    int32_t refresh = 0;
    int32_t score_all = 0;
};

// Shared-prefix cascade: the attention of all B x G query rows of one KV head
// over the shared prefix, in work items of (128-row tile, KV head, key split)
// taken by a persistent grid of `ctas` CTAs.
struct PrefixArgs {
    const void *q;          // [B][Hq][D]
    const void *k_pool;     // [Npool][Hkv][P][D] bf16 (for L2 prefetch; loads go through the tensor maps)
    const void *v_pool;
    const int32_t *page_table;
    const int32_t *seq_lens;
    float *part_o;          // [slots][G][D]
    float *part_lse;        // [slots][G], log2 domain
    uint32_t *flags;
    int32_t batch, num_q_heads, num_kv_heads, group, page_size, max_pages, num_pool_pages;
    int32_t prefix_pages;   // logical pages [0, prefix_pages) are shared by every row
    int32_t splits;         // key splits per (tile, head)
    int32_t ctas;           // persistent grid size (<= tiles x heads x splits)
    int64_t slot0;          // row r's split s writes slot slot0 + r * splits + s
    float scale_log2;
};

constexpr int kPrefixRows = 128;      // query rows per prefix CTA (the MMA's M)
constexpr int kPrefixKeys = 128;      // keys per prefix block (the S tile's N)
constexpr int kPrefixRowThreads = 2;  // softmax threads per query row (each owns 64 of a block's keys)
constexpr int kPrefixThreads = 128 * kPrefixRowThreads + 96;  // softmax warps, MMA warp, K and V TMA warps
constexpr int kMaxPrefixSplits = 64;
// Share of the SMs the persistent prefix grid of a cascade decode takes; the
// paged decode of the rows' own pages gets the others.  Measured on GB300 at
// the shared-prefix workload (128 prefix items): 26 / 32 / 43 / 64 CTAs gave
// 146 / 127 / 106 / 105 us per step (the prefix items slow to ~30 us each
// beside the decode's HBM stream, so the prefix needs ~40 % of the SMs).
constexpr float kPrefixSmShare = 0.43f;

// Warps whose unit ranges intersect row `row` (none when there are no units).
__device__ __forceinline__ void row_warps(const DecodeArgs &a, int row, int64_t &w0, int64_t &w1) {
    if (a.total_units == 0) {
        w0 = 0;
        w1 = -1;
        return;
    }
    const int64_t first = int64_t(row) * a.slots_per_row;
    const int64_t last = min(first + a.slots_per_row, a.total_units) - 1;
    w0 = first / a.units_per_warp;
    w1 = last / a.units_per_warp;
}

// A warp that covers a whole row writes the final output itself, unless
// another kernel contributes pieces to the row.
__device__ __forceinline__ bool row_is_final(const DecodeArgs &a, int64_t w0, int64_t w1) {
    return w0 == w1 && a.extra_pieces == 0;
}

constexpr int kScoreThreads = 128;    // scoring CTA: 4 warps x 32 pages
constexpr int kSelectThreads = 256;   // ranking CTA: one row
constexpr int kSelectKeyCap = 4096;   // keys held in shared memory by the select stage
constexpr int kSelectBallotKeys = 2048;  // rows up to this long: warp-ballot compaction
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
// Most units a row may have for the one-row-per-CTA decode (their codes sit
// in shared memory beside the rings), and the most CTAs it splits a row over
// (their pieces are folded with one round of loads).
constexpr int kRowCtaMaxSlots = 1024;
constexpr int kRowBlocksMax = 8;
// One-call steps (bf16 KV, exact top-K): rows split over at least this many
// decode CTAs are scored by those CTAs themselves (one cluster per row)
// instead of by the scoring grid.
#ifndef QSKV_FUSED_SCORE_MIN_BLOCKS
#define QSKV_FUSED_SCORE_MIN_BLOCKS 2
#endif
constexpr int kFusedScoreMinBlocks = QSKV_FUSED_SCORE_MIN_BLOCKS;
// The decode grid folds a split row itself when one warp can load all of the
// row's pieces in a single round of at most this many 16-byte loads per lane
// (pieces x G x D / 128).  Measured on GB300: the GPT2-like rows (15 pieces
// of 64 floats) fold faster in the grid than in the merge kernel (decode call
// 30.4 -> 29.0 us); the Llama-like rows (9 pieces of 4 x 128 floats, three
// rounds for one warp) are slower that way (58.3 -> 61.9 us).
constexpr int kFoldMaxLoads = 16;

}  // namespace qskv

// hs_common.cuh -- shared device/host helpers of libhs (sm_103a only).
//
// PTX wrappers for mbarriers and bulk (TMA) copies, the bounded wait that
// every spin in this library goes through, block-wide scans, and host-side
// launch checks.  Nothing here is shared with the oracle.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hs_api.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libhs is written for sm_103a (Blackwell) only"
#endif

namespace hs {

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// ----------------------------------------------------------------------------
// Device status word: the first error code stored wins.
__device__ __forceinline__ void set_status(int32_t* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------------------
// mbarrier (shared::cta, 64-bit).
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// `count` arrivals at once (a thread standing in for others).
__device__ __forceinline__ void mbar_arrive_count(uint64_t* bar, uint32_t count) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(count)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: returns true when the phase with `parity` completed, false if
// `timeout_ns` of wall time passed first or *abort became non-zero (another
// role of the CTA gave up).  Never traps, never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t timeout_ns,
                                                  const volatile int* abort = nullptr) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort != nullptr && *abort != 0) return false;
            if (global_timer_ns() - t0 > timeout_ns) return false;
        }
    }
}

// ----------------------------------------------------------------------------
// Bulk (non-tensor) async copies, [HC] "cp.async.bulk of the whole span".
// global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// shared -> global, tracked by bulk groups.
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk group has finished READING shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk group has completed (writes visible).
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 16-byte global -> shared copy, completion tracked by cp.async groups or
// cp.async.mbarrier.arrive.
__device__ __forceinline__ void tc_cp_async16(uint32_t dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}

// Arrive on `bar` once this thread's cp.async copies issued so far complete
// (the arrival counts toward the barrier's expected count).
__device__ __forceinline__ void tc_cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------
// Warp / block scans (integer, exact).
__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

// Block-wide exclusive scan of v over threadIdx.x order with one barrier:
// each warp publishes its total, then every warp scans the (at most 32) warp
// totals itself.  `scratch` holds >= 32 ints of shared memory; *total
// receives the block sum.  Must be called by every thread.  `scratch` is
// read after the barrier, so a second call needs a barrier before it.
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    const int incl = warp_incl_scan(v);
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    const int w = lane < nwarps ? scratch[lane] : 0;
    const int wi = warp_incl_scan(w);
    *total = __shfl_sync(0xffffffffu, wi, nwarps - 1);
    return __shfl_sync(0xffffffffu, wi - w, warp) + incl - v;
}

// ----------------------------------------------------------------------------
// Programmatic dependent launch (PTX griddepcontrol).  Every kernel of the
// library lets its dependents start launching (pdl_trigger) at once, except
// the fp8 row reconstruction, which does so when it is done, and
// the kernels on the decode step's critical path are launched with
// programmatic stream serialization, so each may start while its stream
// predecessor still runs.  Rule kept by every such kernel: before pdl_wait
// it writes no global memory and reads only inputs that no kernel of this
// library writes (the query); pdl_wait returns once the predecessor grid has
// completed and its writes are visible (at once when there is none).
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Default time limit of every bounded wait in this library (wall time).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s

}  // namespace hs

// ----------------------------------------------------------------------------
// Host-side helpers.
namespace hs_host {

int num_sms();  // SM count of the current device (cached per device)

// Opt `func` in to `bytes` of dynamic shared memory on the current device.
// The attribute is raised only when a launch needs more than was set before
// (per device); fails with HS_ERR_CAPACITY beyond the device's limit.
int ensure_dynamic_smem(const void* func, size_t bytes, int* cache /* [64] */);

inline int launch_status() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

// Launch with programmatic stream serialization (the kernel follows the
// pdl_trigger / pdl_wait rule above).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, hs_stream_t stream,
               Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) {
        cudaGetLastError();
        return HS_ERR_CUDA;
    }
    return HS_OK;
}

}  // namespace hs_host

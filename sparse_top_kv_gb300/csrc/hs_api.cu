// hs_api.cu -- host-side helpers of the C ABI (status strings, pinned host
// pointers, device properties).
#include "hs_common.cuh"

extern "C" const char* hs_status_string(int status) {
    switch (status) {
        case HS_OK: return "HS_OK";
        case HS_ERR_INVALID_ARG: return "HS_ERR_INVALID_ARG";
        case HS_ERR_MISALIGNED: return "HS_ERR_MISALIGNED";
        case HS_ERR_CAPACITY: return "HS_ERR_CAPACITY";
        case HS_ERR_CUDA: return "HS_ERR_CUDA";
        case HS_ERR_TIMEOUT: return "HS_ERR_TIMEOUT";
        case HS_ERR_BAD_INDEX: return "HS_ERR_BAD_INDEX";
        case HS_ERR_UNSUPPORTED: return "HS_ERR_UNSUPPORTED";
        default: return "HS_ERR_UNKNOWN";
    }
}

extern "C" int hs_host_device_pointer(const void* host_ptr, void** dev_ptr) {
    if (host_ptr == nullptr || dev_ptr == nullptr) return HS_ERR_INVALID_ARG;
    void* d = nullptr;
    if (cudaHostGetDevicePointer(&d, const_cast<void*>(host_ptr), 0) != cudaSuccess) {
        cudaGetLastError();
        return HS_ERR_CUDA;
    }
    *dev_ptr = d;
    return HS_OK;
}

// Self-test of the bounded wait every kernel of the library goes through
// (hs::mbar_wait_bounded): one CTA, one mbarrier that expects one arrival.
//  mode 0: nothing arrives -> the wait gives up after timeout_ns;
//  mode 1: thread 0 arrives first -> the wait completes;
//  mode 2: nothing arrives, a second warp raises the CTA's abort flag after
//          ~20 us -> the wait gives up early, as a role does when another
//          role of its CTA failed.
// A wait that gives up stores HS_ERR_TIMEOUT; elapsed_ns receives the wait's
// wall time.  Nothing else is in flight, so giving up leaves no copy or
// tensor-memory operation behind.
namespace {
__global__ void wait_selftest_kernel(int32_t mode, uint64_t timeout_ns, int32_t* status,
                                     int64_t* elapsed_ns) {
    __shared__ uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        hs::mbar_init(&bar, 1);
        abort_flag = 0;
        hs::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (mode == 1) hs::mbar_arrive(&bar);
        const uint64_t t0 = hs::global_timer_ns();
        const bool ok = hs::mbar_wait_bounded(&bar, 0, timeout_ns, mode == 2 ? &abort_flag : nullptr);
        *elapsed_ns = int64_t(hs::global_timer_ns() - t0);
        if (!ok) hs::set_status(status, HS_ERR_TIMEOUT);
    } else if (threadIdx.x == 32 && mode == 2) {
        const uint64_t t0 = hs::global_timer_ns();
        while (hs::global_timer_ns() - t0 < 20000) {
        }
        abort_flag = 1;
    }
}
}  // namespace

extern "C" int hs_wait_selftest(int32_t mode, uint64_t timeout_ns, int32_t* status,
                                int64_t* elapsed_ns, hs_stream_t stream) {
    if (mode < 0 || mode > 2 || status == nullptr || elapsed_ns == nullptr)
        return HS_ERR_INVALID_ARG;
    wait_selftest_kernel<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(mode, timeout_ns,
                                                                                status, elapsed_ns);
    return hs_host::launch_status();
}

namespace hs_host {

int num_sms() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

int ensure_dynamic_smem(const void* func, size_t bytes, int* cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
    if (dev >= 0 && dev < 64 && cache[dev] >= int(bytes)) return HS_OK;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, func) != cudaSuccess) return HS_ERR_CUDA;
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
        return HS_ERR_CUDA;
    if (bytes + fa.sharedSizeBytes > size_t(optin)) return HS_ERR_CAPACITY;
    // Without the opt-in, static + dynamic shared memory must fit 48 KB.
    if (bytes + fa.sharedSizeBytes > 48 * 1024 &&
        cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) !=
            cudaSuccess)
        return HS_ERR_CUDA;
    if (dev >= 0 && dev < 64) cache[dev] = int(bytes);
    return HS_OK;
}

}  // namespace hs_host

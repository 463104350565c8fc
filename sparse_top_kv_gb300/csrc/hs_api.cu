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

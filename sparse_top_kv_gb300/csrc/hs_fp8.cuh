// hs_fp8.cuh -- reconstruction of fp8_ds_mla latent columns: eight E4M3
// codes and their group's fp32 scale -> eight bf16 values code * scale
// (product in fp32, rounded to nearest even; the codes go through the
// hardware e4m3x2 -> f16x2 conversion, which is exact).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace hs {

__device__ __forceinline__ uint4 fp8_dequant8(uint2 codes, float scale) {
    const uint32_t w[2] = {codes.x, codes.y};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t word = w[k >> 1];
        const __nv_fp8x2_storage_t pair =
            static_cast<__nv_fp8x2_storage_t>((k & 1) ? (word >> 16) : (word & 0xFFFFu));
        const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3));
        const float2 f = __half22float2(h);
        const __nv_bfloat162 b =
            __floats2bfloat162_rn(__fmul_rn(f.x, scale), __fmul_rn(f.y, scale));
        o[k] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace hs

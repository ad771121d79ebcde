// Element-wise arithmetic that several kernels must perform identically (the
// fused epilogues give the same bits as the stand-alone kernels).
#pragma once

#include <cuda_fp8.h>

namespace moe {

// silu(g) * u = g / (1 + exp(-g)) * u, each step rounded to fp32.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

// Scale of a 128-element FP8 group: amax / 448 (448 = largest e4m3 value),
// 1 for an all-zero group.
__device__ __forceinline__ float fp8_group_scale(float amax) {
    return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

// e4m3 code of v / scale, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint8_t fp8_code(float v, float scale) {
    return (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(v, scale), __NV_SATFINITE, __NV_E4M3);
}

}  // namespace moe

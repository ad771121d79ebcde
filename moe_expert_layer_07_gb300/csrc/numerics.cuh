// Element-wise arithmetic that several kernels must perform identically (the
// fused epilogues give the same bits as the stand-alone kernels).
#pragma once

#include <cuda_fp8.h>

namespace moe {

// silu(g) * u = g / (1 + exp(-g)) * u in fp32, with the hardware's fast
// exponential and division (each a couple of units in the last place; the
// method fixes no rounding here, and every kernel uses this one function, so
// they agree bit for bit).  In the gate/up epilogues this evaluation is the
// per-tile tail that the MMAs wait on: the correctly rounded expf and
// division made the wide SwiGLU GEMM 10-16% slower.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fmul_rn(__fdividef(g, __fadd_rn(1.0f, __expf(-g))), u);
}

// Scale of a 128-element FP8 group: amax / 448 (448 = largest e4m3 value),
// 1 for an all-zero group.
__device__ __forceinline__ float fp8_group_scale(float amax) {
    return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

// Requantisation of h: e4m3 code of v * inv with inv = fp8_group_inv(scale)
// (the correctly rounded 1 / scale, formed once per 128-feature group, so v
// * inv lies within one fp32 unit of v / scale), round to nearest even,
// saturating to +-448.  x's codes keep the IEEE division (quant_row_segment).
__device__ __forceinline__ float fp8_group_inv(float scale) { return __frcp_rn(scale); }
__device__ __forceinline__ uint8_t fp8_code(float v, float inv) {
    return (uint8_t)__nv_cvt_float_to_fp8(__fmul_rn(v, inv), __NV_SATFINITE, __NV_E4M3);
}

// FP8 quantisation of one 256-column segment of a bf16 row by one warp:
// lanes 0-15 take 128-column group 2 seg, lanes 16-31 group 2 seg + 1, 8
// consecutive values per lane.  Each group's scale is its amax / 448 and each
// value's code e4m3_rn_sat(v / scale) (IEEE division).  Columns at or past H
// (a multiple of 128) are skipped.
__device__ __forceinline__ void quant_row_segment(const uint16_t *__restrict__ in_row,
                                                  uint8_t *__restrict__ out_row,
                                                  float *__restrict__ scales_row, int seg,
                                                  int lane, int H) {
    const int col = seg * 256 + lane * 8;
    const bool active = col < H;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (active) v = *reinterpret_cast<const uint4 *>(in_row + col);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // bf16 -> fp32 is exact: the bits move up 16 places
        f[2 * j] = __uint_as_float(w[j] << 16);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = fp8_group_scale(amax);
    if (!active) return;
    uint32_t q[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint16_t lo = (uint16_t)__nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(f[4 * h], sc), __fdiv_rn(f[4 * h + 1], sc)), __NV_SATFINITE,
            __NV_E4M3);
        const uint16_t hi = (uint16_t)__nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(f[4 * h + 2], sc), __fdiv_rn(f[4 * h + 3], sc)), __NV_SATFINITE,
            __NV_E4M3);
        q[h] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *reinterpret_cast<uint2 *>(out_row + col) = make_uint2(q[0], q[1]);
    if ((lane & 15) == 0) scales_row[col / 128] = sc;
}

}  // namespace moe

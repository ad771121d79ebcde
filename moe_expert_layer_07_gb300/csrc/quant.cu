// Activation quantisation: x -> FP8 (per token, per 128 columns) and the
// SwiGLU activation h = silu(gate) * up with its FP8 requantisation (or bf16
// rounding in BF16 layers).  FP8 layout of the R1-shaped workload: e4m3
// codes with one fp32 scale per row and 128-column group, scale = amax/448
// (SGLang/H20 article, section "MoE": block-scale handling in the MoE
// GEMMs).  The x quantiser takes its decision in the same fp32 arithmetic
// the definition states (IEEE division, round-to-nearest-even saturating
// conversion), so its codes are exact.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "numerics.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// two fp32 -> two e4m3 codes (round to nearest even, saturate to +-448)
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// One warp per (row, 256-column segment): lanes 0-15 quantise group 2s,
// lanes 16-31 group 2s+1; each lane holds 8 consecutive bf16 values.
__global__ void __launch_bounds__(256)
    quant_rows_kernel(const uint16_t *__restrict__ in, uint8_t *__restrict__ out,
                      float *__restrict__ scales, int rows, const int32_t *rows_dev, int H) {
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();
    const int lane = threadIdx.x & 31;
    const long warp = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int segs = (H + 255) / 256;
    const long row = warp / segs;
    const int seg = (int)(warp % segs);
    const int nrows = rows_dev ? min(rows, max(0, *rows_dev)) : rows;
    if (row >= nrows) return;
    quant_row_segment(in + row * H, out + row * H, scales + row * (H / 128), seg, lane, H);
}

// One warp per (row, 128-wide group of h); each lane 4 consecutive values.
template <bool FP8>
__global__ void __launch_bounds__(256)
    silu_mul_kernel(const float *__restrict__ in, void *__restrict__ out,
                    float *__restrict__ scales, int rows, const int32_t *rows_dev, int I) {
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();   // the gate/up rows (and their count) of the previous kernel
    const int lane = threadIdx.x & 31;
    const long warp = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int groups = I / 128;
    const long row = warp / groups;
    const int grp = (int)(warp % groups);
    const int nrows = rows_dev ? min(rows, max(0, *rows_dev)) : rows;
    if (row >= nrows) return;
    const int col = grp * 128 + lane * 4;
    const float4 g = *reinterpret_cast<const float4 *>(in + row * 2 * I + col);
    const float4 u = *reinterpret_cast<const float4 *>(in + row * 2 * I + I + col);
    const float h[4] = {silu_mul(g.x, u.x), silu_mul(g.y, u.y), silu_mul(g.z, u.z),
                        silu_mul(g.w, u.w)};
    if (FP8) {
        float amax = fmaxf(fmaxf(fabsf(h[0]), fabsf(h[1])), fmaxf(fabsf(h[2]), fabsf(h[3])));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = fp8_group_scale(amax), inv = fp8_group_inv(sc);
        const uint32_t q = (uint32_t)e4m3x2(__fmul_rn(h[0], inv), __fmul_rn(h[1], inv)) |
                           ((uint32_t)e4m3x2(__fmul_rn(h[2], inv), __fmul_rn(h[3], inv)) << 16);
        *reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(out) + row * I + col) = q;
        if (lane == 0) scales[row * (I / 128) + grp] = sc;
    } else {
        __nv_bfloat162 a = __floats2bfloat162_rn(h[0], h[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(h[2], h[3]);
        uint2 p;
        p.x = *reinterpret_cast<uint32_t *>(&a);
        p.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + row * I + col) = p;
    }
}

}  // namespace

int launch_act_requant(const moe_config *cfg, int mode, int rows, const int32_t *rows_dev,
                       const void *in, void *out, float *out_scales, cudaStream_t s) {
    if (rows == 0) return MOE_OK;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    int rc;
    if (mode == MOE_ACT_IDENTITY) {
        const int H = cfg->hidden;
        const long warps = (long)rows * ((H + 255) / 256);
        rc = launch_dependent(quant_rows_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s,
                              static_cast<const uint16_t *>(in), static_cast<uint8_t *>(out),
                              out_scales, rows, rows_dev, H);
    } else {
        const int I = cfg->inter;
        const long warps = (long)rows * (I / 128);
        const dim3 grid((unsigned)((warps + 7) / 8));
        rc = fp8 ? launch_dependent(silu_mul_kernel<true>, grid, dim3(256), 0, s,
                                    static_cast<const float *>(in), out, out_scales, rows,
                                    rows_dev, I)
                 : launch_dependent(silu_mul_kernel<false>, grid, dim3(256), 0, s,
                                    static_cast<const float *>(in), out, out_scales, rows,
                                    rows_dev, I);
    }
    if (rc) return rc;
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace moe

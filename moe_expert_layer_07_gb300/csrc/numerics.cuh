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

// ---- sigmoid score: fp32(1 / (1 + exp(-l))) with the quotient in fp64 ------
// The routing score is the fp64 sigmoid rounded to fp32.  This GPU's fp64
// rate is a small fraction of its fp32 rate, so the value is first evaluated
// in double-float arithmetic: pairs (hi, lo) of fp32 numbers, about 2^-42
// relative error after every step below.  If that value lies more than 2^-38
// (relative) from each midpoint between neighbouring fp32 numbers, the fp64
// evaluation (within a few 2^-53) rounds to the same fp32 number, which is
// returned.  Otherwise, or for |l| > 80, the fp64 expression itself is
// evaluated.  The result is therefore always that of the fp64 expression;
// the fallback takes about one value in 2^13.
namespace dfl {
struct F2 {
    float hi, lo;
};
__device__ __forceinline__ F2 two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ F2 fast_two_sum(float a, float b) {   // |a| >= |b|
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ F2 add(F2 a, F2 b) {
    const F2 s = two_sum(a.hi, b.hi);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ F2 mul(F2 a, F2 b) {
    const float p = __fmul_rn(a.hi, b.hi);
    float e = __fmaf_rn(a.hi, b.hi, -p);   // the product's rounding error, exactly
    e = __fmaf_rn(a.hi, b.lo, e);
    e = __fmaf_rn(a.lo, b.hi, e);
    return fast_two_sum(p, e);
}
}  // namespace dfl

__device__ __forceinline__ float sigmoid_score_fp64(float l) {
    return (float)(1.0 / (1.0 + exp(-(double)l)));
}

__device__ __forceinline__ float sigmoid_score(float l, bool *fell_back = nullptr) {
    using dfl::F2;
    const float x = -l;
    if (!(fabsf(x) <= 80.0f)) {
        if (fell_back) *fell_back = true;
        return sigmoid_score_fp64(l);
    }
    // x = k ln2/8 + r, |r| <= ln2/16: ln2/8 in three parts, the first two of
    // 13 significant bits so that k times them is exact (|k| <= 924)
    const float k = rintf(__fmul_rn(x, 0x1.715476p+3f));
    const F2 rr = dfl::two_sum(__fmaf_rn(-k, 0x1.62ep-4f, x), -__fmul_rn(k, 0x1.0cp-18f));
    const F2 r = dfl::fast_two_sum(rr.hi, __fmaf_rn(k, 0x1.05c61p-32f, rr.lo));
    // exp(r) = 1 + r + r^2/2 + r^3/6 + r^4/24 + r^5 (1/5! + r/6! + r^2/7! + r^3/8!),
    // the last factor in fp32 (it weighs under 2^-29 of the sum)
    const float t = __fmaf_rn(
        r.hi, __fmaf_rn(r.hi, __fmaf_rn(r.hi, 0x1.a01a02p-16f, 0x1.a01a02p-13f), 0x1.6c16c2p-10f),
        0x1.111112p-7f);
    F2 u = dfl::add(F2{0x1.555556p-5f, -0x1.555556p-30f}, dfl::mul(r, F2{t, 0.0f}));
    u = dfl::add(F2{0x1.555556p-3f, -0x1.555556p-28f}, dfl::mul(r, u));
    u = dfl::add(F2{0.5f, 0.0f}, dfl::mul(r, u));
    u = dfl::add(F2{1.0f, 0.0f}, dfl::mul(r, u));
    u = dfl::add(F2{1.0f, 0.0f}, dfl::mul(r, u));
    // times 2^(k/8) = 2^(k >> 3) 2^((k & 7) / 8)
    const int ki = (int)k;
    F2 p2;
    switch (ki & 7) {
        case 0: p2 = F2{1.0f, 0.0f}; break;
        case 1: p2 = F2{0x1.172b84p+0f, -0x1.c15742p-27f}; break;
        case 2: p2 = F2{0x1.306fe0p+0f, 0x1.4636e2p-25f}; break;
        case 3: p2 = F2{0x1.4bfdaep+0f, -0x1.593abcp-25f}; break;
        case 4: p2 = F2{0x1.6a09e6p+0f, 0x1.9fcef4p-26f}; break;
        case 5: p2 = F2{0x1.8ace54p+0f, 0x1.15506ep-27f}; break;
        case 6: p2 = F2{0x1.ae89fap+0f, -0x1.a94b14p-26f}; break;
        default: p2 = F2{0x1.d5818ep+0f, -0x1.822dbcp-27f}; break;
    }
    F2 e = dfl::mul(p2, u);
    e.hi = ldexpf(e.hi, ki >> 3);
    e.lo = ldexpf(e.lo, ki >> 3);
    const F2 d = dfl::add(F2{1.0f, 0.0f}, e);
    // y = 1 / d: y0 correctly rounded from d.hi, then one correction term
    const float y0 = __fdiv_rn(1.0f, d.hi);
    const float ph = __fmul_rn(d.hi, y0);
    const float pl = __fmaf_rn(d.hi, y0, -ph);
    const float tt = __fmaf_rn(-d.lo, y0, __fsub_rn(__fsub_rn(1.0f, ph), pl));
    const float c = __fmul_rn(y0, tt);
    // the nearest fp32 number to y0 + c and the distance of y0 + c from it
    const float s = __fadd_rn(y0, c);
    const float dist = __fadd_rn(__fsub_rn(y0, s), c);
    const int si = __float_as_int(s);
    const float half_up = 0.5f * (__int_as_float(si + 1) - s);
    const float half_dn = 0.5f * (s - __int_as_float(si - 1));
    const float margin = s * 0x1p-38f;
    const bool safe = dist >= 0.0f ? (half_up - dist > margin) : (half_dn + dist > margin);
    if (safe) return s;
    if (fell_back) *fell_back = true;
    return sigmoid_score_fp64(l);
}

}  // namespace moe

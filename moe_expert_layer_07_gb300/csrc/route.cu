// Gating and top-k routing (Moreh report "21K output tokens/s DeepSeek
// inference on MI300X with Expert Parallelism", section "Overview": a light
// gating network picks a few experts per token; section "Load balancing
// across GPUs": the gate emits ids in the permuted expert order).
//
// Two kernels:
//  gate_logits_kernel  l[t,e] = sum_h x[t,h] Wg[e,h] on CUDA cores with a
//                      fixed order: lane L of a warp owns the 16-byte chunks
//                      c = L, L+32, ... of the hidden dimension (elements
//                      h with (h/8) mod 32 == L), accumulates them in
//                      increasing h with fp32 FMA, and the 32 lane partials
//                      meet in an xor butterfly (16, 8, 4, 2, 1).  A bf16
//                      product is exact in fp32, so the result is a fixed
//                      sequence of rounded additions: the routing decision
//                      is reproducible bit for bit.  A CTA stages a 16-token x
//                      16-expert tile through shared memory; each warp
//                      computes 4 tokens x 8 experts (32 accumulators).
//  route_select_kernel one warp per token: sigmoid (fp64, rounded to fp32)
//                      or softmax scores, group scores from each group's
//                      best group_topn, top groups, then top_k experts by
//                      repeated warp-wide arg-max with ties to the lower
//                      index; weights; ids mapped through log2phys.
#include <cuda_bf16.h>

#include <algorithm>
#include <cfloat>
#include <climits>
#include <mutex>

#include "internal.h"
#include "numerics.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kEB = 8;   // experts per warp tile (tokens per warp tile: TB, 4 or 8)

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two independent fp32 FMAs in one instruction (each lane an IEEE fma, the
// same result as fmaf): d = a * b + c on {lo, hi} pairs.
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// element e (0..7, increasing h) of 8 packed bf16 values, widened to fp32
__device__ __forceinline__ float bf_elem(const uint4 &a, int e) {
    const uint32_t w = e < 2 ? a.x : e < 4 ? a.y : e < 6 ? a.z : a.w;
    return (e & 1) ? bf_hi(w) : bf_lo(w);
}

// CTA tile of 16 tokens x 16 experts: 8 warps of 4 tokens x 8 experts each
// (TB = 4), or 4 warps of 8 x 8 (TB = 8: each staged value feeds twice the
// FMAs, for fewer shared-memory loads and widenings per output, at the cost
// of registers; taken for large batches).  The CTA stages 256 hidden
// elements of its 32 rows per step in shared memory (cp.async, 4-deep ring),
// so every row is fetched once per CTA instead of once per warp.  Lane L
// reads elements 8L..8L+7 of every 256-element step, i.e. the hidden slice
// (h/8) mod 32 == L, in increasing h, whatever TB.
constexpr int kCT = 16, kCE = 16;           // CTA tile
constexpr int kStepElems = 256;             // hidden elements per stage
constexpr int kLogitStages = 4;
constexpr int kStageBytes = (kCT + kCE) * kStepElems * 2;   // 16 KB

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    // src-size 0 fills the 16 bytes with zeros (rows past T or E, H tail)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

template <int TB>
__global__ void __launch_bounds__(TB == 4 ? 256 : 128)
    gate_logits_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ wg,
                       const float *__restrict__ offset, float *__restrict__ logits, int T,
                       int E, int H, const L2Prefetch pf) {
    extern __shared__ __align__(16) uint8_t smem[];
    ptx::pdl_launch_dependents();   // the selection kernel may take its SM slots now
    if (pf.units > 0 && pf.tiled) {
        // tiled weights: the first K blocks of a 128-row block are one
        // contiguous run of 16 KB tiles; one prefetch per tile
        const int mt1 = pf.inter / 128, kbt = pf.hidden * pf.elem_bytes / 128;
        const int nt = pf.bytes / 128;
        const long jobs = (long)pf.units * 2 * nt;
        const long nthreads = (long)gridDim.x * gridDim.y * blockDim.x;
        for (long j = ((long)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
             j < jobs; j += nthreads) {
            const int u = (int)(j / (2 * nt)), r = (int)(j % (2 * nt));
            const int g = u / mt1, mt = u - g * mt1;
            if (g >= pf.groups) break;
            const long block = (long)g * 2 * mt1 + (r < nt ? 0 : mt1) + mt;
            const long tile = block * kbt + (r % nt);
            ptx::prefetch_l2(pf.w13 + tile * (128 * 128), 128 * 128);
        }
    } else if (pf.units > 0) {   // L2 prefetch of the expert FFN's first weight rows (a hint)
        const int mt1 = pf.inter / 128;
        const long jobs = (long)pf.units * 256;
        const long nthreads = (long)gridDim.x * gridDim.y * blockDim.x;
        for (long j = ((long)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
             j < jobs; j += nthreads) {
            const int u = (int)(j >> 8), r = (int)(j & 255);
            const int g = u / mt1, mt = u - g * mt1;
            if (g >= pf.groups) break;
            const long row = (long)g * 2 * pf.inter + (r < 128 ? 0 : pf.inter) + mt * 128 + (r & 127);
            ptx::prefetch_l2(pf.w13 + row * pf.hidden * pf.elem_bytes, (uint32_t)pf.bytes);
        }
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t_base = blockIdx.x * kCT, e_base = blockIdx.y * kCE;
    const int steps = (H + kStepElems - 1) / kStepElems;
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(smem));

    // stage s: 32 rows (16 tokens then 16 experts) x 32 pieces of 16 bytes
    constexpr int NT = TB == 4 ? 256 : 128;   // threads: (16 / TB) x 2 warps
    auto issue = [&](int step) {
        const uint32_t buf = sbase + (step % kLogitStages) * kStageBytes;
#pragma unroll
        for (int i = 0; i < 1024 / NT; ++i) {
            const int p = tid + NT * i;
            const int r = p >> 5, piece = p & 31;
            const int h = step * kStepElems + piece * 8;
            const bool is_x = r < kCT;
            const int row = is_x ? t_base + r : e_base + (r - kCT);
            const bool ok = h < H && (is_x ? row < T : row < E);
            const uint16_t *src = (is_x ? x : wg) + (ok ? (size_t)row * H + h : 0);
            cp_async16(buf + r * (kStepElems * 2) + piece * 16, src, ok);
        }
    };

    // accumulators of experts (2p, 2p + 1) side by side for the paired FMA
    uint64_t acc2[TB][kEB / 2];
#pragma unroll
    for (int i = 0; i < TB; ++i)
#pragma unroll
        for (int p = 0; p < kEB / 2; ++p) acc2[i][p] = 0ull;
    const int wt = warp >> 1, we = warp & 1;   // warp tile: tokens TB wt.., experts 8we..

#pragma unroll
    for (int st = 0; st < kLogitStages - 1; ++st) {
        if (st < steps) issue(st);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int step = 0; step < steps; ++step) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kLogitStages - 2) : "memory");
        __syncthreads();   // stage `step` is visible; stage step-1 is no longer read
        if (step + kLogitStages - 1 < steps) issue(step + kLogitStages - 1);
        asm volatile("cp.async.commit_group;" ::: "memory");
        const uint8_t *buf = smem + (step % kLogitStages) * kStageBytes;
        uint4 xv[TB], wv[kEB];
#pragma unroll
        for (int i = 0; i < TB; ++i)
            xv[i] = *reinterpret_cast<const uint4 *>(buf + (wt * TB + i) * (kStepElems * 2) + lane * 16);
#pragma unroll
        for (int j = 0; j < kEB; ++j)
            wv[j] = *reinterpret_cast<const uint4 *>(buf + (kCT + we * kEB + j) * (kStepElems * 2) + lane * 16);
        // outer products over the chunk's 8 elements: each bf16 value is
        // widened once per step, and every accumulator still takes its 8
        // products in increasing h (two accumulators per paired FMA)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            uint64_t x2[TB], w2[kEB / 2];
#pragma unroll
            for (int i = 0; i < TB; ++i) {
                const float xf = bf_elem(xv[i], e);
                x2[i] = pack2(xf, xf);
            }
#pragma unroll
            for (int p = 0; p < kEB / 2; ++p)
                w2[p] = pack2(bf_elem(wv[2 * p], e), bf_elem(wv[2 * p + 1], e));
#pragma unroll
            for (int i = 0; i < TB; ++i)
#pragma unroll
                for (int p = 0; p < kEB / 2; ++p) acc2[i][p] = fma2(x2[i], w2[p], acc2[i][p]);
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");

    // output o = i kEB + j of the warp tile ends in lane o mod 32, slot o / 32
    constexpr int NO = TB * kEB / 32;
    float mine[NO];
#pragma unroll
    for (int q = 0; q < NO; ++q) mine[q] = 0.0f;
#pragma unroll
    for (int i = 0; i < TB; ++i)
#pragma unroll
        for (int j = 0; j < kEB; ++j) {
            float v = (j & 1) ? hi2(acc2[i][j >> 1]) : lo2(acc2[i][j >> 1]);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == ((i * kEB + j) & 31)) mine[(i * kEB + j) >> 5] = v;
        }
#pragma unroll
    for (int q = 0; q < NO; ++q) {
        const int o = q * 32 + lane;
        const int t = t_base + wt * TB + o / kEB, e = e_base + we * kEB + o % kEB;
        if (t < T && e < E)
            logits[(size_t)t * E + e] = offset ? __fadd_rn(mine[q], offset[e]) : mine[q];
    }
}

struct SelectArgs {
    int T, E, k, groups, topk_groups, topn, sigmoid, norm;
    float scaling;
    const float *logits, *bias;
    const int32_t *log2phys;
    int32_t *ids;
    float *w;
    int32_t *status;
    // optional: the FP8 quantisation of x (xq e4m3 [T, H], xs [T, H/128])
    const uint16_t *x;
    uint8_t *xq;
    float *xs;
    int H;
};

// warp-wide arg-max with ties to the lower index; every lane gets the result
__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

// One CTA per token. All four warps of the CTA (one per SM sub-partition)
// evaluate the scores into shared memory (the sigmoid in fp32 double-float
// arithmetic, fp64 only where that cannot decide the rounding:
// sigmoid_score); warp 0 then does the selection alone, holding expert
// e = q*32 + lane in its registers.
constexpr int kSelThreads = 128;

template <int PL>   // experts per lane of warp 0: e = q*32 + lane, q < PL
__global__ void __launch_bounds__(kSelThreads) route_select_kernel(const SelectArgs a) {
    __shared__ float sh_l[PL * 32], sh_s[PL * 32], sh_sel[PL * 32];
    ptx::pdl_launch_dependents();
    if (a.xq && (int)blockIdx.x < a.T) {
        // this token's row of x to FP8, while the gate logits are still being
        // computed: x is the call's input (complete before the logit kernel,
        // a full-dependency launch, started), not a previous kernel's output
        const size_t t0 = blockIdx.x;
        const int segs = (a.H + 255) / 256;
        for (int seg = threadIdx.x >> 5; seg < segs; seg += kSelThreads / 32)
            quant_row_segment(a.x + t0 * a.H, a.xq + t0 * a.H, a.xs + t0 * (a.H / 128), seg,
                              threadIdx.x & 31, a.H);
    }
    ptx::pdl_wait();   // logits of the previous kernel
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    if (t >= a.T) return;   // block-uniform
    const float *lrow = a.logits + (size_t)t * a.E;

    for (int e = threadIdx.x; e < PL * 32; e += kSelThreads) {
        const bool ok = e < a.E;
        const float lv = ok ? lrow[e] : 0.0f;
        float sv = lv, selv = lv;
        if (a.sigmoid) {
            sv = sigmoid_score(lv);
            selv = (ok && a.bias) ? __fadd_rn(sv, a.bias[e]) : sv;
        }
        sh_l[e] = lv;
        sh_s[e] = sv;
        sh_sel[e] = selv;
    }
    __syncthreads();
    if (threadIdx.x >= 32) return;   // warp-uniform

    float l[PL], s[PL], sel[PL];
    uint32_t valid = 0;
#pragma unroll
    for (int q = 0; q < PL; ++q) {
        const int e = q * 32 + lane;
        l[q] = sh_l[e];
        s[q] = sh_s[e];
        sel[q] = sh_sel[e];
        if (e < a.E) valid |= 1u << q;
    }
    uint32_t allowed = valid;

    if (a.groups > 1) {
        const int gs = a.E / a.groups;
        uint32_t gmask = 0;
        if (gs == 32 && a.topn <= 4) {
            // Groups of 32: lane L holds expert L of every group (group g is
            // q == g), so all groups reduce at once; same order, ties and
            // sums as the general path below.
            float gsum[PL];
            uint32_t taken = 0;
            for (int r = 0; r < a.topn; ++r) {
                float v[PL];
                int id[PL];
#pragma unroll
                for (int q = 0; q < PL; ++q) {
                    const bool ok = ((valid >> q) & 1u) && !((taken >> q) & 1u);
                    v[q] = ok ? sel[q] : -FLT_MAX;
                    id[q] = ok ? q * 32 + lane : INT_MAX;
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
                    for (int q = 0; q < PL; ++q) {
                        const float ov = __shfl_xor_sync(0xffffffffu, v[q], o);
                        const int oi = __shfl_xor_sync(0xffffffffu, id[q], o);
                        if (ov > v[q] || (ov == v[q] && oi < id[q])) {
                            v[q] = ov;
                            id[q] = oi;
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < PL; ++q) {
                    if (id[q] != INT_MAX && (id[q] & 31) == lane) taken |= 1u << q;
                    gsum[q] = (r == 0) ? v[q] : __fadd_rn(gsum[q], v[q]);
                }
            }
            for (int r = 0; r < a.topk_groups; ++r) {   // group scores are warp-uniform
                float bv = -FLT_MAX;
                int bg = INT_MAX;
#pragma unroll
                for (int q = 0; q < PL; ++q)
                    if (q < a.groups && !((gmask >> q) & 1u) &&
                        (gsum[q] > bv || (gsum[q] == bv && q < bg))) {
                        bv = gsum[q];
                        bg = q;
                    }
                if (bg != INT_MAX) gmask |= 1u << bg;
            }
        } else {
            float my_gscore = -FLT_MAX;
            for (int g = 0; g < a.groups; ++g) {
                uint32_t taken = 0;
                float sum = 0.0f;
                for (int r = 0; r < a.topn; ++r) {
                    float bv = -FLT_MAX;
                    int bi = INT_MAX;
#pragma unroll
                    for (int q = 0; q < PL; ++q) {
                        const int e = q * 32 + lane;
                        if (((valid >> q) & 1u) && !((taken >> q) & 1u) && e >= g * gs &&
                            e < (g + 1) * gs && (sel[q] > bv || (sel[q] == bv && e < bi))) {
                            bv = sel[q];
                            bi = e;
                        }
                    }
                    warp_argmax(bv, bi);
                    if (bi != INT_MAX && (bi & 31) == lane) taken |= 1u << (bi >> 5);
                    sum = (r == 0) ? bv : __fadd_rn(sum, bv);
                }
                if (lane == g) my_gscore = sum;
            }
            for (int r = 0; r < a.topk_groups; ++r) {
                float v = (lane < a.groups && !((gmask >> lane) & 1u)) ? my_gscore : -FLT_MAX;
                int i = (lane < a.groups && !((gmask >> lane) & 1u)) ? lane : INT_MAX;
                warp_argmax(v, i);
                if (i != INT_MAX) gmask |= 1u << i;
            }
        }
#pragma unroll
        for (int q = 0; q < PL; ++q) {
            const int e = q * 32 + lane;
            if (((valid >> q) & 1u) && !((gmask >> (e / gs)) & 1u)) allowed &= ~(1u << q);
        }
    }

    // top-k by repeated arg-max; lane j keeps slot j
    uint32_t chosen = 0;
    int my_id = 0;
    float my_score = 0.0f;   // sigmoid s or softmax logit of slot `lane`
    for (int j = 0; j < a.k; ++j) {
        float bv = -FLT_MAX;
        int bi = INT_MAX;
#pragma unroll
        for (int q = 0; q < PL; ++q) {
            const int e = q * 32 + lane;
            if (((allowed >> q) & 1u) && !((chosen >> q) & 1u) &&
                (sel[q] > bv || (sel[q] == bv && e < bi))) {
                bv = sel[q];
                bi = e;
            }
        }
        warp_argmax(bv, bi);
        if (bi == INT_MAX) {   // fewer candidates than k (rejected on the host)
            if (lane == 0 && a.status) atomicOr(a.status, MOE_DEV_BAD_EXPERT_ID);
            return;
        }
        const int owner = bi & 31, oq = bi >> 5;
        float sv = 0.0f;
#pragma unroll
        for (int q = 0; q < PL; ++q)
            if (q == oq) sv = s[q];
        sv = __shfl_sync(0xffffffffu, sv, owner);
        if (lane == owner) chosen |= 1u << oq;
        if (lane == j) {
            my_id = bi;
            my_score = sv;
        }
    }

    float w = 0.0f;
    if (a.sigmoid) {
        float total = 0.0f;
        for (int j = 0; j < a.k; ++j) total = __fadd_rn(total, __shfl_sync(0xffffffffu, my_score, j));
        w = a.norm ? __fmul_rn(__fdiv_rn(my_score, total), a.scaling)
                   : __fmul_rn(my_score, a.scaling);
    } else {
        // The ids above depend on the logits alone; the weights are
        // exp(l - m) / sum exp(l' - m) with m the largest logit.  Each
        // exponential is taken in fp32 (expf, within 2 ulp) of the exact
        // difference: l - m rounded, plus its rounding error from a two-sum,
        // applied in fp64 as exp(d + e) = exp(d) (1 + e).  Sums, the quotient
        // and the scaling are fp64, so a weight lies within 5.4e-7 (relative)
        // of the fp64 definition while its exponential is a normal fp32
        // number (l - m > -87).  This GPU's fp64 rate is a small fraction of
        // its fp32 rate.
        float m = -FLT_MAX;
#pragma unroll
        for (int q = 0; q < PL; ++q)
            if ((valid >> q) & 1u) m = fmaxf(m, l[q]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        auto ex = [&](float lv) -> double {
            const float d = __fsub_rn(lv, m);
            const float bb = __fsub_rn(d, lv);
            const float e = __fadd_rn(__fsub_rn(lv, __fsub_rn(d, bb)), __fsub_rn(-m, bb));
            const double x = (double)expf(d);
            return fma(x, (double)e, x);
        };
        double denom = 0.0;
        if (a.norm) {
            for (int j = 0; j < a.k; ++j) denom += ex(__shfl_sync(0xffffffffu, my_score, j));
        } else {
            double part = 0.0;
#pragma unroll
            for (int q = 0; q < PL; ++q)
                if ((valid >> q) & 1u) part += ex(l[q]);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            denom = part;
        }
        w = (float)(ex(my_score) / denom * (double)a.scaling);
    }

    if (lane < a.k) {
        int id = my_id;
        if (a.log2phys) {
            id = a.log2phys[my_id];
            if (id < 0 || id >= a.E) {
                if (a.status) atomicOr(a.status, MOE_DEV_BAD_EXPERT_ID);
                id = -1;
            }
        }
        a.ids[(size_t)t * a.k + lane] = id;
        a.w[(size_t)t * a.k + lane] = w;
    }
}

template <int PL>
int launch_select(const SelectArgs &a, cudaStream_t s) {
    return launch_dependent(route_select_kernel<PL>, dim3(a.T), dim3(kSelThreads), 0, s, a);
}

}  // namespace

int route_kernel_count() { return 2; }

int launch_route(const moe_config *cfg, int T, const void *x, const void *w_gate,
                 const float *e_bias, const float *logit_offset, const int32_t *log2phys,
                 float *logits, int32_t *topk_ids, float *topk_w, int32_t *status,
                 cudaStream_t s, const L2Prefetch *pf, uint8_t *xq, float *xs) {
    if (T == 0) return MOE_OK;
    const int E = cfg->num_experts, H = cfg->hidden;
    const dim3 grid((unsigned)ceil_div(T, kCT), (unsigned)ceil_div(E, kCE));
    const int smem = kLogitStages * kStageBytes;
    static std::once_flag attr_once[64];
    static int attr_rc[64];
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return cuda_fail("device ordinal beyond 63");
    std::call_once(attr_once[dev], [&] {
        cudaError_t e = cudaFuncSetAttribute(gate_logits_kernel<4>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gate_logits_kernel<8>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        attr_rc[dev] = (int)e;
    });
    if (attr_rc[dev]) return cuda_fail("cudaFuncSetAttribute", (cudaError_t)attr_rc[dev]);
    const L2Prefetch none;
    // 8 x 8 warp tiles once the CTAs outnumber a few per SM; decode batches
    // keep 8 warps per CTA for latency hiding.  Both give the same bits.
    const bool big = (int64_t)grid.x * grid.y >= 4 * (int64_t)sm_count();
    if (big)
        gate_logits_kernel<8><<<grid, 128, smem, s>>>(static_cast<const uint16_t *>(x),
                                                      static_cast<const uint16_t *>(w_gate),
                                                      logit_offset, logits, T, E, H,
                                                      pf ? *pf : none);
    else
        gate_logits_kernel<4><<<grid, 256, smem, s>>>(static_cast<const uint16_t *>(x),
                                                      static_cast<const uint16_t *>(w_gate),
                                                      logit_offset, logits, T, E, H,
                                                      pf ? *pf : none);
    MOE_LAUNCH_CHECK();

    SelectArgs a;
    a.T = T;
    a.E = E;
    a.k = cfg->top_k;
    a.groups = cfg->num_groups;
    a.topk_groups = cfg->topk_groups;
    a.topn = cfg->group_topn;
    a.sigmoid = cfg->scoring == MOE_SCORING_SIGMOID;
    a.norm = cfg->norm_topk;
    a.scaling = cfg->routed_scaling;
    a.logits = logits;
    a.bias = e_bias;
    a.log2phys = log2phys;
    a.ids = topk_ids;
    a.w = topk_w;
    a.status = status;
    a.x = static_cast<const uint16_t *>(x);
    a.xq = xq;
    a.xs = xs;
    a.H = H;
    const int pl = (int)ceil_div(E, 32);
    int rc;
    if (pl <= 1) rc = launch_select<1>(a, s);
    else if (pl <= 2) rc = launch_select<2>(a, s);
    else if (pl <= 4) rc = launch_select<4>(a, s);
    else if (pl <= 8) rc = launch_select<8>(a, s);
    else if (pl <= 16) rc = launch_select<16>(a, s);
    else rc = launch_select<32>(a, s);
    if (rc) return rc;
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace moe

// ---- self-test of the sigmoid score --------------------------------------
namespace moe {
namespace {
__global__ void sigmoid_selftest_kernel(const float *l, int n, float *fast, float *ref,
                                        int32_t *fallbacks) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        bool fb = false;
        fast[i] = sigmoid_score(l[i], &fb);
        ref[i] = sigmoid_score_fp64(l[i]);
        if (fb) atomicAdd(fallbacks, 1);
    }
}
}  // namespace
}  // namespace moe

extern "C" MOE_API int moe_selftest_sigmoid(const float *logits, int32_t n, float *fast,
                                            float *ref, int32_t *fallbacks, void *stream) {
    if (n < 0 || (n > 0 && (!logits || !fast || !ref || !fallbacks))) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    const int grid = (int)std::min<int64_t>(moe::ceil_div(n, 256), 4096);
    moe::sigmoid_selftest_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        logits, n, fast, ref, fallbacks);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

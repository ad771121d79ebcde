// Combine (Moreh report "21K output tokens/s DeepSeek inference on MI300X
// with Expert Parallelism", section "Overview": expert outputs return to
// their tokens and are summed with the routing weights; section
// "Parallelisation": the shared expert runs for every token).
//
//   out[t] = sum_s Y[expert_offsets[E+s] + t] + sum_j w[t,j] Y[row_of_slot[t,j]]
//
// Y holds each expert's fp32 output rows.  A gather per token in fp32
// (shared experts first, then j ascending):
// every output element is written once by one thread, no atomics.
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxK = 16;
constexpr int kMaxShared = 4;

// grid: (T, column blocks); each thread handles 8 consecutive columns
__global__ void __launch_bounds__(kThreads)
    combine_kernel(const float *__restrict__ y, const int32_t *__restrict__ row_of_slot,
                   const float *__restrict__ topk_w, const int32_t *__restrict__ offsets,
                   void *__restrict__ out, int out_bf16, int T, int H, int E, int S, int k) {
    __shared__ long rows[kMaxShared + kMaxK];
    __shared__ float wts[kMaxShared + kMaxK];
    const int t = blockIdx.x;
    if (threadIdx.x < S) {
        rows[threadIdx.x] = (long)offsets[E + threadIdx.x] + t;
        wts[threadIdx.x] = 1.0f;
    } else if (threadIdx.x < S + k) {
        const int j = threadIdx.x - S;
        rows[threadIdx.x] = row_of_slot[(long)t * k + j];
        wts[threadIdx.x] = topk_w[(long)t * k + j];
    }
    __syncthreads();
    const int v = blockIdx.y * kThreads + threadIdx.x;   // 8-column vector index
    if (v * 8 >= H) return;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int r = 0; r < S + k; ++r) {
        const long row = rows[r];
        if (row < 0) continue;
        const float4 *src = reinterpret_cast<const float4 *>(y + row * H) + 2 * v;
        const float4 a = __ldg(src), b = __ldg(src + 1);
        const float val[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if (r < S) {
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], val[q]);
        } else {
            const float w = wts[r];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = fmaf(w, val[q], acc[q]);
        }
    }
    if (out_bf16) {
        uint4 o;
        uint32_t *p = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
            p[q] = *reinterpret_cast<uint32_t *>(&b2);
        }
        reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + (long)t * H)[v] = o;
    } else {
        float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + (long)t * H) + 2 * v;
        o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

}  // namespace

int launch_combine(const moe_config *cfg, int T, const void *y, const int32_t *row_of_slot,
                   const float *topk_w, const int32_t *offsets, void *out, int out_dtype,
                   cudaStream_t s) {
    if (T == 0) return MOE_OK;
    const int H = cfg->hidden;
    dim3 grid(T, (unsigned)ceil_div(H / 8, kThreads));
    combine_kernel<<<grid, kThreads, 0, s>>>(static_cast<const float *>(y), row_of_slot, topk_w,
                                             offsets, out, out_dtype == MOE_OUT_BF16, T, H,
                                             cfg->num_experts, cfg->num_shared, cfg->top_k);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace moe

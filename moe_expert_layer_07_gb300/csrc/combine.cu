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
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxK = 16;
constexpr int kMaxShared = 4;
constexpr int kMaxRows = kMaxShared + kMaxK;

// grid: (T, column blocks); each thread handles 4 consecutive columns.  All
// rows of the token are loaded before the first addition, so their memory
// latencies overlap; the additions then run in the fixed order.  NR bounds
// the rows per token (shared + top-k) held in registers: a small bound keeps
// the kernel's registers, and so its resident CTAs and loads in flight, up.
template <int NR>
__global__ void __launch_bounds__(kThreads)
    combine_kernel(const float *__restrict__ y, const int32_t *__restrict__ row_of_slot,
                   const float *__restrict__ topk_w, const int32_t *__restrict__ offsets,
                   void *__restrict__ out, int out_bf16, int T, int H, int E, int S, int k) {
    __shared__ long rows[kMaxRows];
    __shared__ float wts[kMaxRows];
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();   // expert outputs of the previous kernel
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
    const int v = blockIdx.y * kThreads + threadIdx.x;   // 4-column vector index
    if (v * 4 >= H) return;
    const int n = S + k;
    float4 val[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r)
        if (r < n && rows[r] >= 0)
            val[r] = __ldg(reinterpret_cast<const float4 *>(y + rows[r] * H) + v);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        if (r >= n || rows[r] < 0) continue;
        const float x[4] = {val[r].x, val[r].y, val[r].z, val[r].w};
        if (r < S) {
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = __fadd_rn(acc[q], x[q]);
        } else {
            const float w = wts[r];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = fmaf(w, x[q], acc[q]);
        }
    }
    if (out_bf16) {
        __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0], acc[1]);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[2], acc[3]);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t *>(&b0);
        o.y = *reinterpret_cast<uint32_t *>(&b1);
        reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + (long)t * H)[v] = o;
    } else {
        reinterpret_cast<float4 *>(static_cast<float *>(out) + (long)t * H)[v] =
            make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
}

}  // namespace

int launch_combine(const moe_config *cfg, int T, const void *y, const int32_t *row_of_slot,
                   const float *topk_w, const int32_t *offsets, void *out, int out_dtype,
                   cudaStream_t s) {
    if (T == 0) return MOE_OK;
    const int H = cfg->hidden;
    if (cfg->num_shared + cfg->top_k > kMaxRows) return MOE_ERR_UNSUPPORTED_SHAPE;
    const dim3 grid(T, (unsigned)ceil_div(H / 4, kThreads));
    auto kern = cfg->num_shared + cfg->top_k <= 10 ? combine_kernel<10> : combine_kernel<kMaxRows>;
    if (launch_dependent(kern, grid, dim3(kThreads), 0, s, static_cast<const float *>(y),
                         row_of_slot, topk_w, offsets, out, (int)(out_dtype == MOE_OUT_BF16), T,
                         H, cfg->num_experts, cfg->num_shared, cfg->top_k))
        return MOE_ERR_CUDA;
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace moe

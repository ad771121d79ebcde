// Continuous load balancing (Moreh report "21K output tokens/s DeepSeek
// inference on MI300X with Expert Parallelism", section "Load balancing
// across GPUs": in serving, expert activation frequencies are re-measured
// periodically and a new expert permutation is generated from them).
//
//   count_rows_kernel  counts[p] += rows of routed expert p in this batch,
//                      read from the dispatch offsets (int64, exact: the
//                      result does not depend on launch order).
//   coactivation_kernel  A[a][b] += tokens whose top-k holds both a and b
//                      (logical ids), for affinity-aware placement (SGLang/H20
//                      article, section "Expert Affinity EPLB").
//   relayout_kernel    dst block p = src block src_slot[p]: the weight (or
//                      scale) re-layout that applies a new permutation, with
//                      16-byte vector copies; run it on a side stream into a
//                      second buffer while the layer keeps serving.
#include <algorithm>

#include "internal.h"

namespace moe {
namespace {

__global__ void count_rows_kernel(const int32_t *__restrict__ offsets, int64_t *__restrict__ counts,
                                  int E) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p < E) counts[p] += (int64_t)(offsets[p + 1] - offsets[p]);
}

// One thread per ordered pair (j1 != j2) of a token's top-k: A[a][b] += 1 with
// a, b the LOGICAL ids; integer atomics, so the sum does not depend on order.
__global__ void coactivation_kernel(const int32_t *__restrict__ ids,
                                    const int32_t *__restrict__ phys2log,
                                    unsigned long long *__restrict__ A, int T, int k, int E) {
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)T * k * k) return;
    const int t = (int)(i / (k * k)), r = (int)(i % (k * k));
    const int j1 = r / k, j2 = r % k;
    if (j1 == j2) return;
    int a = ids[(long)t * k + j1], b = ids[(long)t * k + j2];
    if (a < 0 || a >= E || b < 0 || b >= E) return;
    if (phys2log) {
        a = phys2log[a];
        b = phys2log[b];
        if (a < 0 || a >= E || b < 0 || b >= E) return;
    }
    if (a != b) atomicAdd(&A[(long)a * E + b], 1ull);
}

__global__ void __launch_bounds__(256)
    relayout_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                    const int32_t *__restrict__ src_slot, int64_t vec_per_block, int groups,
                    int32_t *__restrict__ bad) {
    const int p = blockIdx.y;
    const int q = src_slot[p];
    if (q < 0 || q >= groups) {   // reject an invalid table: copy nothing for this block
        if (threadIdx.x == 0 && blockIdx.x == 0 && bad) atomicOr(bad, MOE_DEV_BAD_EXPERT_ID);
        return;
    }
    const uint4 *s = src + (int64_t)q * vec_per_block;
    uint4 *d = dst + (int64_t)p * vec_per_block;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < vec_per_block;
         v += (int64_t)gridDim.x * blockDim.x)
        d[v] = __ldg(s + v);
}

}  // namespace
}  // namespace moe

extern "C" MOE_API int moe_count_expert_rows(const moe_config *cfg, const int32_t *expert_offsets,
                                             int64_t *counts, void *stream) {
    int rc = moe::check_config(cfg);
    if (rc) return rc;
    if (!expert_offsets || !counts) return MOE_ERR_INVALID_ARG;
    const int E = cfg->num_experts;
    moe::count_rows_kernel<<<(E + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        expert_offsets, counts, E);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

extern "C" MOE_API int moe_relayout_experts(const void *src, void *dst, const int32_t *src_slot,
                                            int32_t groups, int64_t block_bytes,
                                            int32_t *dev_status, void *stream) {
    if (!src || !dst || !src_slot || groups <= 0 || groups > 65535 || block_bytes <= 0)
        return MOE_ERR_INVALID_ARG;
    if (block_bytes % 16 || !moe::aligned16(src) || !moe::aligned16(dst)) return MOE_ERR_INVALID_ARG;
    const char *s = static_cast<const char *>(src);
    const char *d = static_cast<const char *>(dst);
    const int64_t total = block_bytes * groups;
    if (s < d + total && d < s + total) return MOE_ERR_INVALID_ARG;   // buffers overlap
    const int64_t vec = block_bytes / 16;
    const int64_t per_cta = 256 * 8;   // 8 vectors per thread per pass
    const unsigned gx = (unsigned)std::min<int64_t>((vec + per_cta - 1) / per_cta, 1024);
    moe::relayout_kernel<<<dim3(gx, groups), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), src_slot, vec, groups,
        dev_status);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

extern "C" MOE_API int moe_count_coactivation(const moe_config *cfg, int32_t T,
                                              const int32_t *topk_ids, const int32_t *phys2log,
                                              int64_t *coact, void *stream) {
    int rc = moe::check_config(cfg);
    if (rc) return rc;
    if (T < 0 || (T > 0 && (!topk_ids || !coact))) return MOE_ERR_INVALID_ARG;
    const long n = (long)T * cfg->top_k * cfg->top_k;
    if (n == 0) return MOE_OK;
    moe::coactivation_kernel<<<(unsigned)((n + 255) / 256), 256, 0,
                               static_cast<cudaStream_t>(stream)>>>(
        topk_ids, phys2log, reinterpret_cast<unsigned long long *>(coact), T, cfg->top_k,
        cfg->num_experts);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

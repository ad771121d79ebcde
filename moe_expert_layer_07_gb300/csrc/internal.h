// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

namespace moe {

// Every buffer is 256-byte aligned inside a workspace.
constexpr size_t kAlign = 256;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates a configuration; returns MOE_OK or an error code.
int check_config(const moe_config *cfg);

// Rows of the permuted activations for T tokens.
inline int64_t total_rows(const moe_config *cfg, int64_t T) {
    return T * (int64_t)(cfg->top_k + cfg->num_shared);
}
inline int groups_of(const moe_config *cfg) { return cfg->num_experts + cfg->num_shared; }

// Number of streaming multiprocessors of the current device (cached).
int sm_count();

// Records what failed (for moe_last_error_detail on this thread) and returns
// MOE_ERR_CUDA.  e = cudaSuccess when the failure has no CUDA error code.
int cuda_fail(const char *where, cudaError_t e = cudaSuccess);

// ---- launchers (validated arguments; return MOE_OK or MOE_ERR_CUDA) ----
// Weight rows the expert FFN will read first, for the gate-logit kernel to
// prefetch into L2 while routing keeps HBM idle: the first `bytes` of every
// gate and up row of the first `units` gate/up units, taking unit u as
// (expert u / (inter/128), weight tile u % (inter/128)).
struct L2Prefetch {
    const uint8_t *w13 = nullptr;   // e4m3 or bf16 [groups, 2*inter, hidden]
    int hidden = 0, inter = 0, groups = 0, units = 0, bytes = 0;
    int elem_bytes = 1;             // 1 (e4m3) or 2 (bf16)
    int tiled = 0;                  // MOE_LAYOUT_TILES: the K prefix of a row block is contiguous
};
// With xq and xs (FP8 layers), the selection kernel also quantises x
// (e4m3 [T, H] + scales [T, H/128]) while the logits are computed.
int launch_route(const moe_config *cfg, int T, const void *x, const void *w_gate,
                 const float *e_bias, const float *logit_offset, const int32_t *log2phys,
                 float *logits, int32_t *topk_ids, float *topk_w, int32_t *status,
                 cudaStream_t s, const L2Prefetch *pf = nullptr, uint8_t *xq = nullptr,
                 float *xs = nullptr);
int launch_act_requant(const moe_config *cfg, int mode, int rows, const int32_t *rows_dev,
                       const void *in, void *out, float *out_scales, cudaStream_t s);
size_t permute_scratch_bytes(const moe_config *cfg, int T);
// Rows of groups with more than copy_max_rows rows get their table entries
// but are not copied into xp / xp_scales.
int launch_permute(const moe_config *cfg, int T, const int32_t *topk_ids, const void *x_rows,
                   const float *x_scales, int32_t *offsets, int32_t *src_of_row,
                   int32_t *row_of_slot, void *xp, float *xp_scales, void *ws,
                   int32_t *status, cudaStream_t s, int copy_max_rows = 0x7fffffff);
// Row windows: every expert launcher below processes only the groups whose
// row count n satisfies min_rows <= n <= max_rows (the others' rows of its
// outputs are left as they are), so that groups of few and of many rows can
// go to different kernels of one batch.
constexpr int kAllRows = 0x7fffffff;
int launch_grouped_gemm(bool fp8, int groups, int n_out, int k_dim, int rows, const void *a,
                        const float *a_scales, const int32_t *offsets, const void *w,
                        const float *w_scales, bool w_tiled, void *c, int c_dtype,
                        int32_t *status, cudaStream_t s, int min_rows = 0,
                        int max_rows = kAllRows);
int launch_grouped_gemm_swiglu(bool fp8, int groups, int inter, int k_dim, int rows,
                               const void *a, const float *a_scales, const int32_t *offsets,
                               const void *w13, const float *w13_scales, bool w_tiled, void *h,
                               float *h_scales, int32_t *status, cudaStream_t s,
                               int min_rows = 0, int max_rows = kAllRows);
// Wide FP8 batches (groups averaging 16 rows or more): gate/up + SwiGLU +
// FP8 requantisation with token rows on the MMA's M side (gemm_wide.cu).
int launch_swiglu_wide(int groups, int inter, int k_dim, int rows, const void *a,
                       const float *a_scales, const int32_t *offsets, const void *w13,
                       const float *w13_scales, bool w_tiled, void *h, float *h_scales,
                       int32_t *status, cudaStream_t s, int min_rows = 0,
                       int max_rows = kAllRows);
// The same with the activation rows gathered (TMA gather4) from the token
// rows of x: row r of group g is token t(r) of slot src_of_row[r] (routed
// slots t top_k + j, then the shared experts' T rows each); xq e4m3
// [T, k_dim], xs fp32 [T, k_dim / 128].  Same result bits as on dispatched rows.
int launch_swiglu_wide_gather(int groups, int inter, int k_dim, int rows, const void *xq,
                              const float *xs, int T, int top_k, const int32_t *src_of_row,
                              const int32_t *offsets, const void *w13, const float *w13_scales,
                              bool w_tiled, void *h, float *h_scales, int32_t *status,
                              cudaStream_t s, int min_rows = 0, int max_rows = kAllRows);
// Wide FP8 batches, fp32 C with n_out a multiple of 256: the same kernel
// with a plain epilogue (TMA stores of 32 x 32 fp32 blocks).
int launch_gemm_wide(int groups, int n_out, int k_dim, int rows, const void *a,
                     const float *a_scales, const int32_t *offsets, const void *w,
                     const float *w_scales, bool w_tiled, float *c, int32_t *status,
                     cudaStream_t s, int min_rows = 0, int max_rows = kAllRows);
// The experts' FFN in one persistent kernel (FP8 or BF16): gate/up + SwiGLU
// (+ FP8 requant), then down.  `sched` holds ffn_sched_bytes(groups, rows) bytes; it is
// cleared on `s` unless the caller has already zeroed it in stream order.
size_t ffn_sched_bytes(int groups, int rows);
int launch_expert_ffn(bool fp8, int groups, int hidden, int inter, int rows, const void *xp,
                      const float *xp_scales, const int32_t *offsets, const void *w13,
                      const float *w13_scales, const void *w2, const float *w2_scales,
                      bool w_tiled, void *h, float *h_scales, float *y, int32_t *sched,
                      bool sched_zeroed, int32_t *status, cudaStream_t s, int min_rows = 0,
                      int max_rows = kAllRows);
int launch_combine(const moe_config *cfg, int T, const void *y, const int32_t *row_of_slot,
                   const float *topk_w, const int32_t *offsets, void *out, int out_dtype,
                   cudaStream_t s);

// Programmatic dependent launch: `kernel` may start while the previous
// kernel in the stream drains.  Every CTA of such a kernel executes
// pdl_wait() (griddepcontrol.wait) before it reads data that an earlier
// kernel wrote and before it exits, so stream order stays transitive.
template <typename... KArgs, typename... Args>
int launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t s, Args... args) {
    cudaLaunchConfig_t c = {};
    c.gridDim = grid;
    c.blockDim = block;
    c.dynamicSmemBytes = smem;
    c.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = at;
    c.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&c, kernel, args...);
    return e == cudaSuccess ? MOE_OK : cuda_fail("cudaLaunchKernelEx", e);
}

// Kernel launches per call, for the layer's launch count.
int route_kernel_count();
int permute_kernel_count(const moe_config *cfg, int T);

}  // namespace moe

#define MOE_CUDA_TRY(expr)                                   \
    do {                                                     \
        cudaError_t _e = (expr);                             \
        if (_e != cudaSuccess) return moe::cuda_fail(#expr, _e); \
    } while (0)

#define MOE_LAUNCH_CHECK()                                   \
    do {                                                     \
        cudaError_t _e = cudaGetLastError();                 \
        if (_e != cudaSuccess) return moe::cuda_fail("kernel launch", _e); \
    } while (0)

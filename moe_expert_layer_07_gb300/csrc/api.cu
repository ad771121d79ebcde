// The C ABI: argument checks, workspace layout, the layer's launch sequence,
// device status.  Every entry point validates before enqueuing anything and
// never synchronises the host (except moe_get_device_status, which exists to).
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdio>
#include <mutex>

#include "internal.h"

namespace moe {

namespace {
// An NVTX range around each entry point (and each step of the layer call),
// so that a profiler's timeline names the library's calls; without a tool
// attached a push/pop is a call to an empty function.
struct Range {
    explicit Range(const char *name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range &) = delete;
    Range &operator=(const Range &) = delete;
};
}  // namespace

namespace {
thread_local char g_error_detail[256] = "";
}

int cuda_fail(const char *where, cudaError_t e) {
    std::snprintf(g_error_detail, sizeof g_error_detail, "%s: %s", where,
                  e == cudaSuccess ? "failed" : cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

int check_config(const moe_config *c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->scoring != MOE_SCORING_SOFTMAX && c->scoring != MOE_SCORING_SIGMOID)
        return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_DTYPE_BF16 && c->dtype != MOE_DTYPE_FP8_BLOCK128) return MOE_ERR_INVALID_ARG;
    if (c->hidden <= 0 || c->inter <= 0 || c->num_experts <= 0 || c->top_k <= 0 ||
        c->num_shared < 0 || c->max_tokens < 0 || c->num_groups <= 0)
        return MOE_ERR_INVALID_ARG;
    if (c->hidden % 128 || c->inter % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->dtype == MOE_DTYPE_FP8_BLOCK128 && (c->hidden > 7168 || c->inter > 7168))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->num_experts > 1024 || c->num_shared > 4 || c->top_k > 16) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (c->num_groups > 32 || c->num_experts % c->num_groups) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int gs = c->num_experts / c->num_groups;
    if (c->num_groups > 1) {
        if (c->topk_groups <= 0 || c->topk_groups > c->num_groups) return MOE_ERR_INVALID_ARG;
        if (c->group_topn <= 0 || c->group_topn > gs) return MOE_ERR_INVALID_ARG;
        if (c->top_k > c->topk_groups * gs) return MOE_ERR_INVALID_ARG;
    } else if (c->top_k > c->num_experts) {
        return MOE_ERR_INVALID_ARG;
    }
    if (!(c->routed_scaling == c->routed_scaling)) return MOE_ERR_INVALID_ARG;   // NaN
    return MOE_OK;
}

int sm_count() {
    static int counts[64];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::call_once(once[dev], [&] {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 1;
        counts[dev] = n > 0 ? n : 1;
    });
    return counts[dev];
}

namespace {

bool al16(const void *p) { return p == nullptr || aligned16(p); }

bool layout_ok(int32_t l) { return l == MOE_LAYOUT_ROWS || l == MOE_LAYOUT_TILES; }

// Tiled weights are addressed as rows of a [tiles * 128, 128-byte] view.
bool tiled_fits(int64_t groups, int64_t n_out, int64_t k_dim, bool fp8) {
    return groups * n_out * (k_dim / (fp8 ? 128 : 64)) <= INT32_MAX;
}

// Rows per group from which FP8 batches take the wide GEMMs (gate/up + SwiGLU
// with token rows on the MMA's M side, then the down GEMM) instead of the
// one-kernel FFN.  Same-box timings of both on the same R1 rows (identical
// bits): FFN / GEMMs 1.665 / 1.860 ms at 16 rows per group, 1.800 / 1.898 at
// 26.9, 2.042 / 1.924 at 35.9.
constexpr int64_t kWideRowsPerGroup = 32;

bool wide_rows(const moe_config *cfg, int64_t T) {
    return cfg->dtype == MOE_DTYPE_FP8_BLOCK128 &&
           total_rows(cfg, T) >= kWideRowsPerGroup * (int64_t)groups_of(cfg);
}

// Both expert GEMMs run in one persistent kernel for BF16 layers and FP8
// decode batches.
bool fused_ffn(const moe_config *cfg, int64_t T) {
    return cfg->dtype != MOE_DTYPE_FP8_BLOCK128 || !wide_rows(cfg, T);
}

// In batches that take the wide GEMMs, the groups with at most this many
// rows still go to the one-kernel FFN: one 32-row activation tile streams
// their weights once, where a 128-row token tile of the wide kernels would
// be at most a quarter full.
constexpr int kFfnGroupRowsInWide = 32;

// The experts' FFN on dispatched rows, whichever kernels suit the batch:
// the one-kernel FFN for BF16 and for FP8 groups averaging fewer than 32
// rows; else (FP8) the gate/up GEMM with its SwiGLU epilogue and the down
// GEMM, with token rows on the MMA's M side, for the groups of more than 32
// rows, and the one-kernel FFN for the others (the two sets of groups read
// disjoint weights and rows).  All choices give the same result bits.
int experts_forward(bool fp8, int groups, int hidden, int inter, int rows, const void *xp,
                    const float *xp_scales, const int32_t *offsets, const void *w13,
                    const float *w13_scales, const void *w2, const float *w2_scales,
                    bool tiled, void *h, float *h_scales, float *y, int32_t *sched,
                    bool sched_zeroed, int32_t *status, cudaStream_t s) {
    if (!fp8 || (int64_t)rows < kWideRowsPerGroup * (int64_t)groups)
        return launch_expert_ffn(fp8, groups, hidden, inter, rows, xp, xp_scales, offsets, w13,
                                 w13_scales, w2, w2_scales, tiled, h, h_scales, y, sched,
                                 sched_zeroed, status, s);
    int rc = launch_expert_ffn(fp8, groups, hidden, inter, rows, xp, xp_scales, offsets, w13,
                               w13_scales, w2, w2_scales, tiled, h, h_scales, y, sched,
                               sched_zeroed, status, s, 0, kFfnGroupRowsInWide);
    if (rc) return rc;
    rc = launch_grouped_gemm_swiglu(fp8, groups, inter, hidden, rows, xp, xp_scales, offsets, w13,
                                    w13_scales, tiled, h, h_scales, status, s,
                                    kFfnGroupRowsInWide + 1);
    if (rc) return rc;
    return launch_grouped_gemm(fp8, groups, hidden, inter, rows, h, h_scales, offsets, w2,
                               w2_scales, tiled, y, MOE_OUT_F32, status, s,
                               kFfnGroupRowsInWide + 1);
}

int layout(const moe_config *cfg, int64_t Tm, moe_ws_layout *L) {
    const int64_t E = cfg->num_experts, k = cfg->top_k, H = cfg->hidden, I = cfg->inter;
    const int64_t G = groups_of(cfg), Rt = total_rows(cfg, Tm);
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    size_t off = 0;
    auto take = [&](int64_t bytes) {
        const size_t o = off;
        off = align_up(off + (size_t)bytes);
        return o;
    };
    L->status = take(4);
    // the fused FFN's unit counter and per-tile h counters; sits right after
    // the status word so that one memset clears both
    L->ffn_sched = take((int64_t)ffn_sched_bytes((int)G, (int)Rt));
    L->logits = take(4 * Tm * E);
    L->topk_ids = take(4 * Tm * k);
    L->topk_w = take(4 * Tm * k);
    L->xq = take(fp8 ? Tm * H : 0);
    L->xs = take(fp8 ? 4 * Tm * (H / 128) : 0);
    L->expert_offsets = take(4 * (G + 1));
    L->src_of_row = take(4 * Rt);
    L->row_of_slot = take(4 * Tm * k);
    L->perm_scratch = take((int64_t)permute_scratch_bytes(cfg, (int)Tm));
    L->xp = take(Rt * H * (fp8 ? 1 : 2));
    L->xp_scales = take(fp8 ? 4 * Rt * (H / 128) : 0);
    // no layer path keeps fp32 gate/up rows (the field stays for the ABI)
    L->gate_up = take(0);
    L->h = take(Rt * I * (fp8 ? 1 : 2));
    L->h_scales = take(fp8 ? 4 * Rt * (I / 128) : 0);
    L->y = take(4 * Rt * H);
    L->total = off;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(int32_t code) {
    switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_FAULT: return "device reported invalid data";
    default: return "unknown status";
    }
}

int moe_route(const moe_config *cfg, int32_t T, const void *x, const void *w_gate,
              const float *e_bias, const float *logit_offset, const int32_t *log2phys,
              float *logits, int32_t *topk_ids, float *topk_w, int32_t *dev_status,
              void *stream) {
    Range range("moe_route");
    int rc = check_config(cfg);
    if (rc) return rc;
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !w_gate || !logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!al16(x) || !al16(w_gate)) return MOE_ERR_INVALID_ARG;
    if (e_bias && cfg->scoring != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
    return launch_route(cfg, T, x, w_gate, e_bias, logit_offset, log2phys, logits, topk_ids,
                        topk_w, dev_status, static_cast<cudaStream_t>(stream));
}

int moe_route_quantize(const moe_config *cfg, int32_t T, const void *x, const void *w_gate,
                       const float *e_bias, const float *logit_offset, const int32_t *log2phys,
                       float *logits, int32_t *topk_ids, float *topk_w, void *xq, float *xs,
                       int32_t *dev_status, void *stream) {
    Range range("moe_route_quantize");
    int rc = check_config(cfg);
    if (rc) return rc;
    if (cfg->dtype != MOE_DTYPE_FP8_BLOCK128 || T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !w_gate || !logits || !topk_ids || !topk_w || !xq || !xs) return MOE_ERR_INVALID_ARG;
    if (!al16(x) || !al16(w_gate) || !al16(xq)) return MOE_ERR_INVALID_ARG;
    if (e_bias && cfg->scoring != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
    return launch_route(cfg, T, x, w_gate, e_bias, logit_offset, log2phys, logits, topk_ids,
                        topk_w, dev_status, static_cast<cudaStream_t>(stream), nullptr,
                        static_cast<uint8_t *>(xq), xs);
}

int moe_act_requant(const moe_config *cfg, int32_t mode, int32_t rows, const int32_t *rows_dev,
                    const void *in, void *out, float *out_scales, void *stream) {
    Range range("moe_act_requant");
    int rc = check_config(cfg);
    if (rc) return rc;
    if (rows < 0 || (mode != MOE_ACT_IDENTITY && mode != MOE_ACT_SILU_MUL))
        return MOE_ERR_INVALID_ARG;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    if (mode == MOE_ACT_IDENTITY && !fp8) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!in || !out || (fp8 && !out_scales)) return MOE_ERR_INVALID_ARG;
    if (!al16(in) || !al16(out)) return MOE_ERR_INVALID_ARG;
    return launch_act_requant(cfg, mode, rows, rows_dev, in, out, out_scales,
                              static_cast<cudaStream_t>(stream));
}

int moe_permute_workspace_size(const moe_config *cfg, int32_t T, size_t *bytes) {
    int rc = check_config(cfg);
    if (rc) return rc;
    if (T < 0 || !bytes) return MOE_ERR_INVALID_ARG;
    *bytes = permute_scratch_bytes(cfg, T);
    return MOE_OK;
}

int moe_permute(const moe_config *cfg, int32_t T, const int32_t *topk_ids, const void *x_rows,
                const float *x_scales, int32_t *expert_offsets, int32_t *src_of_row,
                int32_t *row_of_slot, void *xp, float *xp_scales, void *ws, size_t ws_bytes,
                int32_t copy_max_group_rows, int32_t *dev_status, void *stream) {
    Range range("moe_permute");
    int rc = check_config(cfg);
    if (rc) return rc;
    if (T < 0 || !expert_offsets || copy_max_group_rows < 0) return MOE_ERR_INVALID_ARG;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    if (T > 0 && (!topk_ids || !x_rows || !src_of_row || !row_of_slot || !xp ||
                  (fp8 && (!x_scales || !xp_scales))))
        return MOE_ERR_INVALID_ARG;
    if (!al16(x_rows) || !al16(xp)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < permute_scratch_bytes(cfg, T) || (T > 0 && !ws))
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    return launch_permute(cfg, T, topk_ids, x_rows, x_scales, expert_offsets, src_of_row,
                          row_of_slot, xp, xp_scales, ws, dev_status,
                          static_cast<cudaStream_t>(stream), copy_max_group_rows);
}

int moe_grouped_gemm(const moe_config *cfg, int32_t groups, int32_t n_out, int32_t k_dim,
                     int32_t rows, const void *a, const float *a_scales,
                     const int32_t *expert_offsets, const void *w, const float *w_scales,
                     int32_t w_layout, void *c, int32_t c_dtype, int32_t min_group_rows,
                     int32_t max_group_rows, int32_t *dev_status, void *stream) {
    Range range("moe_grouped_gemm");
    int rc = check_config(cfg);
    if (rc) return rc;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    if (groups <= 0 || rows < 0 || n_out <= 0 || k_dim <= 0 || min_group_rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (!layout_ok(w_layout)) return MOE_ERR_INVALID_ARG;
    if (c_dtype != MOE_OUT_F32 && c_dtype != MOE_OUT_BF16) return MOE_ERR_INVALID_ARG;
    if (groups > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (n_out % 128 || k_dim % (fp8 ? 128 : 64)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (fp8 && k_dim > 7168) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)groups * n_out > INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (w_layout == MOE_LAYOUT_TILES && !tiled_fits(groups, n_out, k_dim, fp8))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!a || !w || !c || !expert_offsets || (fp8 && (!a_scales || !w_scales)))
        return MOE_ERR_INVALID_ARG;
    if (!al16(a) || !al16(w) || !al16(c)) return MOE_ERR_INVALID_ARG;
    return launch_grouped_gemm(fp8, groups, n_out, k_dim, rows, a, a_scales, expert_offsets, w,
                               w_scales, w_layout == MOE_LAYOUT_TILES, c, c_dtype, dev_status,
                               static_cast<cudaStream_t>(stream), min_group_rows, max_group_rows);
}

int moe_grouped_gemm_swiglu(const moe_config *cfg, int32_t groups, int32_t inter, int32_t k_dim,
                            int32_t rows, const void *a, const float *a_scales,
                            const int32_t *expert_offsets, const void *w13,
                            const float *w13_scales, int32_t w_layout, void *h, float *h_scales,
                            int32_t min_group_rows, int32_t max_group_rows,
                            int32_t *dev_status, void *stream) {
    Range range("moe_grouped_gemm_swiglu");
    int rc = check_config(cfg);
    if (rc) return rc;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    if (groups <= 0 || rows < 0 || inter <= 0 || k_dim <= 0 || min_group_rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (!layout_ok(w_layout)) return MOE_ERR_INVALID_ARG;
    if (groups > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (inter % 128 || k_dim % (fp8 ? 128 : 64)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (fp8 && k_dim > 7168) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)groups * 2 * inter > INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (w_layout == MOE_LAYOUT_TILES && !tiled_fits(groups, 2 * (int64_t)inter, k_dim, fp8))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!a || !w13 || !h || !expert_offsets || (fp8 && (!a_scales || !w13_scales || !h_scales)))
        return MOE_ERR_INVALID_ARG;
    if (!al16(a) || !al16(w13) || !al16(h)) return MOE_ERR_INVALID_ARG;
    return launch_grouped_gemm_swiglu(fp8, groups, inter, k_dim, rows, a, a_scales,
                                      expert_offsets, w13, w13_scales,
                                      w_layout == MOE_LAYOUT_TILES, h, h_scales, dev_status,
                                      static_cast<cudaStream_t>(stream), min_group_rows,
                                      max_group_rows);
}

int moe_grouped_gemm_swiglu_gather(const moe_config *cfg, int32_t groups, int32_t inter,
                                   int32_t k_dim, int32_t rows, const void *x_rows,
                                   const float *x_scales, int32_t T, const int32_t *src_of_row,
                                   const int32_t *expert_offsets, const void *w13,
                                   const float *w13_scales, int32_t w_layout, void *h,
                                   float *h_scales, int32_t min_group_rows,
                                   int32_t max_group_rows, int32_t *dev_status, void *stream) {
    Range range("moe_grouped_gemm_swiglu_gather");
    int rc = check_config(cfg);
    if (rc) return rc;
    if (cfg->dtype != MOE_DTYPE_FP8_BLOCK128) return MOE_ERR_INVALID_ARG;
    if (groups <= 0 || rows < 0 || T < 0 || inter <= 0 || k_dim <= 0 || min_group_rows < 0)
        return MOE_ERR_INVALID_ARG;
    if (!layout_ok(w_layout)) return MOE_ERR_INVALID_ARG;
    if (groups > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (inter % 128 || k_dim % 128 || k_dim > 7168) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)groups * 2 * inter > INT32_MAX) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (w_layout == MOE_LAYOUT_TILES && !tiled_fits(groups, 2 * (int64_t)inter, k_dim, true))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (T == 0) return MOE_ERR_INVALID_ARG;   // rows to fill but no token rows
    if (!x_rows || !x_scales || !src_of_row || !expert_offsets || !w13 || !w13_scales || !h ||
        !h_scales)
        return MOE_ERR_INVALID_ARG;
    if (!al16(x_rows) || !al16(w13) || !al16(h)) return MOE_ERR_INVALID_ARG;
    return launch_swiglu_wide_gather(groups, inter, k_dim, rows, x_rows, x_scales, T,
                                     cfg->top_k, src_of_row, expert_offsets, w13, w13_scales,
                                     w_layout == MOE_LAYOUT_TILES, h, h_scales, dev_status,
                                     static_cast<cudaStream_t>(stream), min_group_rows,
                                     max_group_rows);
}

size_t moe_expert_ffn_sched_bytes(int32_t groups, int32_t rows) {
    if (groups <= 0 || rows < 0) return 0;
    return ffn_sched_bytes(groups, rows);
}

int moe_expert_ffn(const moe_config *cfg, int32_t groups, int32_t rows, const void *a,
                   const float *a_scales, const int32_t *expert_offsets, const void *w13,
                   const float *w13_scales, const void *w2, const float *w2_scales,
                   int32_t w_layout, void *h, float *h_scales, float *y, int32_t *sched,
                   size_t sched_bytes, int32_t min_group_rows, int32_t max_group_rows,
                   int32_t *dev_status, void *stream) {
    Range range("moe_expert_ffn");
    int rc = check_config(cfg);
    if (rc) return rc;
    if (groups <= 0 || rows < 0 || !layout_ok(w_layout) || min_group_rows < 0)
        return MOE_ERR_INVALID_ARG;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    if (groups > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)groups * 2 * cfg->inter > INT32_MAX || (int64_t)groups * cfg->hidden > INT32_MAX)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (w_layout == MOE_LAYOUT_TILES &&
        (!tiled_fits(groups, 2 * (int64_t)cfg->inter, cfg->hidden, fp8) ||
         !tiled_fits(groups, cfg->hidden, cfg->inter, fp8)))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!a || !expert_offsets || !w13 || !w2 || !h || !y || !sched ||
        (fp8 && (!a_scales || !w13_scales || !w2_scales || !h_scales)))
        return MOE_ERR_INVALID_ARG;
    if (!al16(a) || !al16(w13) || !al16(w2) || !al16(h) || !al16(y)) return MOE_ERR_INVALID_ARG;
    if (sched_bytes < ffn_sched_bytes(groups, rows)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return launch_expert_ffn(fp8, groups, cfg->hidden, cfg->inter, rows, a, a_scales,
                             expert_offsets,
                             w13, w13_scales, w2, w2_scales, w_layout == MOE_LAYOUT_TILES, h,
                             h_scales, y, sched, false, dev_status,
                             static_cast<cudaStream_t>(stream), min_group_rows, max_group_rows);
}

int moe_experts_forward(const moe_config *cfg, int32_t groups, int32_t rows, const void *a,
                        const float *a_scales, const int32_t *expert_offsets, const void *w13,
                        const float *w13_scales, const void *w2, const float *w2_scales,
                        int32_t w_layout, void *h, float *h_scales, float *y, int32_t *sched,
                        size_t sched_bytes, int32_t *dev_status, void *stream) {
    Range range("moe_experts_forward");
    int rc = check_config(cfg);
    if (rc) return rc;
    if (groups <= 0 || rows < 0 || !layout_ok(w_layout)) return MOE_ERR_INVALID_ARG;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    if (groups > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)groups * 2 * cfg->inter > INT32_MAX || (int64_t)groups * cfg->hidden > INT32_MAX)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (w_layout == MOE_LAYOUT_TILES &&
        (!tiled_fits(groups, 2 * (int64_t)cfg->inter, cfg->hidden, fp8) ||
         !tiled_fits(groups, cfg->hidden, cfg->inter, fp8)))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!a || !expert_offsets || !w13 || !w2 || !h || !y || !sched ||
        (fp8 && (!a_scales || !w13_scales || !w2_scales || !h_scales)))
        return MOE_ERR_INVALID_ARG;
    if (!al16(a) || !al16(w13) || !al16(w2) || !al16(h) || !al16(y)) return MOE_ERR_INVALID_ARG;
    if (sched_bytes < ffn_sched_bytes(groups, rows)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    return experts_forward(fp8, groups, cfg->hidden, cfg->inter, rows, a, a_scales,
                           expert_offsets, w13, w13_scales, w2, w2_scales,
                           w_layout == MOE_LAYOUT_TILES, h, h_scales, y, sched, false,
                           dev_status, static_cast<cudaStream_t>(stream));
}

int moe_combine(const moe_config *cfg, int32_t T, const void *y, const int32_t *row_of_slot,
                const float *topk_w, const int32_t *expert_offsets, void *out, int32_t out_dtype,
                void *stream) {
    Range range("moe_combine");
    int rc = check_config(cfg);
    if (rc) return rc;
    if (T < 0 || (out_dtype != MOE_OUT_F32 && out_dtype != MOE_OUT_BF16)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y || !row_of_slot || !topk_w || !expert_offsets || !out) return MOE_ERR_INVALID_ARG;
    if (!al16(y) || !al16(out)) return MOE_ERR_INVALID_ARG;
    return launch_combine(cfg, T, y, row_of_slot, topk_w, expert_offsets, out, out_dtype,
                          static_cast<cudaStream_t>(stream));
}

int moe_workspace_layout(const moe_config *cfg, moe_ws_layout *L) {
    int rc = check_config(cfg);
    if (rc) return rc;
    if (!L) return MOE_ERR_INVALID_ARG;
    return layout(cfg, cfg->max_tokens, L);
}

int moe_workspace_size(const moe_config *cfg, size_t *bytes) {
    if (!bytes) return MOE_ERR_INVALID_ARG;
    moe_ws_layout L;
    int rc = moe_workspace_layout(cfg, &L);
    if (rc) return rc;
    *bytes = L.total;
    return MOE_OK;
}

int moe_layer_kernel_count(const moe_config *cfg, int32_t T) {
    if (check_config(cfg) || T <= 0) return 0;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    // route (with the FP8 quantisation of x), permute, the experts' FFN (one
    // fused kernel, or gate/up GEMM with SwiGLU + down GEMM), combine
    (void)fp8;
    // wide batches: the FFN kernel for groups of few rows, the two GEMMs for the rest
    const int ffn = fused_ffn(cfg, T) ? 1 : 3;
    return route_kernel_count() + permute_kernel_count(cfg, T) + ffn + 1;
}

int moe_layer_forward(const moe_config *cfg, const moe_weights *w, int32_t T, const void *x,
                      void *out, int32_t out_dtype, void *ws, size_t ws_bytes, void *stream) {
    Range range("moe_layer_forward");
    int rc = check_config(cfg);
    if (rc) return rc;
    if (!w || !ws || T < 0 || T > cfg->max_tokens) return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_OUT_F32 && out_dtype != MOE_OUT_BF16) return MOE_ERR_INVALID_ARG;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    if (T > 0 && (!x || !out)) return MOE_ERR_INVALID_ARG;
    if (!w->w_gate || !w->w13 || !w->w2 || (fp8 && (!w->w13_scales || !w->w2_scales)))
        return MOE_ERR_INVALID_ARG;
    if (w->e_bias && cfg->scoring != MOE_SCORING_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (!layout_ok(w->expert_layout)) return MOE_ERR_INVALID_ARG;
    const bool tiled = w->expert_layout == MOE_LAYOUT_TILES;
    if (tiled && (!tiled_fits(groups_of(cfg), 2 * (int64_t)cfg->inter, cfg->hidden, fp8) ||
                  !tiled_fits(groups_of(cfg), cfg->hidden, cfg->inter, fp8)))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!al16(x) || !al16(out) || !al16(ws) || !al16(w->w_gate) || !al16(w->w13) ||
        !al16(w->w2))
        return MOE_ERR_INVALID_ARG;
    moe_ws_layout L;
    layout(cfg, cfg->max_tokens, &L);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(ws);
    int32_t *status = reinterpret_cast<int32_t *>(base + L.status);
    const bool fused = T > 0 && fused_ffn(cfg, T);
    const int rows = (int)total_rows(cfg, T);
    // status word and the one-kernel FFN's scheduler counters (every path
    // runs that kernel, for all groups or for the groups with few rows)
    const size_t clear = L.ffn_sched + ffn_sched_bytes(groups_of(cfg), rows);
    MOE_CUDA_TRY(cudaMemsetAsync(status, 0, clear, s));
    if (T == 0) return MOE_OK;

    const int E = cfg->num_experts, G = groups_of(cfg), H = cfg->hidden, I = cfg->inter;
    float *logits = reinterpret_cast<float *>(base + L.logits);
    int32_t *ids = reinterpret_cast<int32_t *>(base + L.topk_ids);
    float *tw = reinterpret_cast<float *>(base + L.topk_w);
    int32_t *offsets = reinterpret_cast<int32_t *>(base + L.expert_offsets);
    int32_t *src = reinterpret_cast<int32_t *>(base + L.src_of_row);
    int32_t *ros = reinterpret_cast<int32_t *>(base + L.row_of_slot);
    (void)E;

    // The one-kernel FFN claims gate/up units 0, 1, ... first (group-major);
    // at decode every group has one 32-row activation tile, so unit u is
    // (expert u / (inter/128), weight tile u % (inter/128)).  Their first K
    // blocks go to L2 while routing leaves HBM idle: 12 of R1's 56 K blocks,
    // about 117 MB (8 blocks gained 11 us per layer over 4, and 12 another 2 us).
    // BF16 layers take none: with it, the layer call (captured in a graph, L2
    // flushed before each replay) took 0.231 ms instead of 0.218 for the
    // V2-Lite-sized layer and 0.079 ms instead of 0.048 for 64 tokens over 16
    // experts.
    L2Prefetch pf;
    if (fused && fp8) {
        pf.w13 = static_cast<const uint8_t *>(w->w13);
        pf.hidden = H;
        pf.inter = I;
        pf.groups = G;
        pf.units = 2 * sm_count();
        pf.elem_bytes = fp8 ? 1 : 2;
        pf.bytes = H * pf.elem_bytes < 1536 ? H * pf.elem_bytes : 1536;
        pf.tiled = tiled;
    }
    // FP8: the selection kernel also quantises x (while the logits run)
    const void *rows_src = fp8 ? static_cast<const void *>(base + L.xq) : x;
    const float *rows_scales = fp8 ? reinterpret_cast<const float *>(base + L.xs) : nullptr;
    {
        Range r("route");
        rc = launch_route(cfg, T, x, w->w_gate, w->e_bias, w->logit_offset, w->log2phys, logits,
                          ids, tw, status, s, fused ? &pf : nullptr,
                          fp8 ? base + L.xq : nullptr,
                          fp8 ? reinterpret_cast<float *>(base + L.xs) : nullptr);
    }
    if (rc) return rc;
    {
        Range r("dispatch");
        rc = launch_permute(cfg, T, ids, rows_src, rows_scales, offsets, src, ros, base + L.xp,
                            reinterpret_cast<float *>(base + L.xp_scales), base + L.perm_scratch,
                            status, s);
    }
    if (rc) return rc;
    // the one-kernel FFN's scheduler counters were cleared with the status word
    Range r_ffn("experts");
    rc = experts_forward(fp8, G, H, I, rows, base + L.xp,
                         reinterpret_cast<const float *>(base + L.xp_scales), offsets, w->w13,
                         w->w13_scales, w->w2, w->w2_scales, tiled, base + L.h,
                         reinterpret_cast<float *>(base + L.h_scales),
                         reinterpret_cast<float *>(base + L.y),
                         reinterpret_cast<int32_t *>(base + L.ffn_sched), true, status, s);
    if (rc) return rc;
    return launch_combine(cfg, T, base + L.y, ros, tw, offsets, out, out_dtype, s);
}

const char *moe_last_error_detail(void) { return g_error_detail; }

int moe_get_device_status(const void *ws, int32_t *status) {
    if (!ws || !status) return MOE_ERR_INVALID_ARG;
    int32_t v = 0;
    // the status word is the first field of the layer workspace
    MOE_CUDA_TRY(cudaMemcpy(&v, ws, sizeof v, cudaMemcpyDeviceToHost));
    *status = v;
    if (v == 0) return MOE_OK;
    return (v & MOE_DEV_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_ERR_DEVICE_FAULT;
}

}  // extern "C"

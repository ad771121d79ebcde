/*
 * moe_gb300 — the DeepSeek-style Mixture-of-Experts FFN layer at decode time,
 * on one NVIDIA GB300 (sm_103a).
 *
 * The layer (Moreh report "21K output tokens/s DeepSeek inference on MI300X
 * with Expert Parallelism", sections "Overview" and "Parallelisation"):
 * a light gate routes each token to top_k of E small SwiGLU experts, an
 * always-on shared expert runs for every token, and the expert outputs are
 * summed with the routing weights.  Expert-parallel dispatch/combine (the
 * all-to-all of section "Compute-communication overlap") becomes, on one
 * GPU, a permutation of token rows into per-expert contiguous rows and a
 * weighted gather back.
 *
 * Conventions for every call below
 *   - Pointers are DEVICE pointers unless the argument says "host".
 *   - All buffers are allocated by the caller; the library allocates no
 *     memory.  Row-major layouts, innermost dimension last, no padding.
 *     Every device pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device calls only enqueue work: none synchronises the host
 *     or reads device data back, and sizes that depend on the routing
 *     (rows per expert) stay on the device, so every device call can be
 *     captured in a CUDA graph (the report's section "Using HIP Graphs":
 *     tensor sizes kept static so that dispatch and combine can live inside
 *     the captured graph).
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code.  Argument and
 *     shape errors are returned before anything is enqueued.  Problems only
 *     the device can see (an expert id out of range, inconsistent offsets,
 *     a pipeline wait that ran out of time) set bits MOE_DEV_* in a device
 *     status word (int32) instead; kernels never trap.  `dev_status` may be
 *     NULL (no report).
 *
 * Notation: T tokens, H hidden, I expert intermediate width, E routed
 * experts, S shared experts, k = top_k, G = E + S groups, R = T*k routed
 * rows, R_tot = R + S*T rows.  Groups 0..E-1 are the routed experts in
 * PHYSICAL order, groups E..G-1 the shared experts.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- codes ------------------------------------------------------------ */
enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,        /* null pointer, bad enum, T < 0, misalignment */
    MOE_ERR_UNSUPPORTED_SHAPE = -2,  /* a dimension this build does not handle */
    MOE_ERR_WORKSPACE_TOO_SMALL = -3,
    MOE_ERR_CUDA = -4,               /* a CUDA runtime call failed */
    MOE_ERR_TIMEOUT = -5,            /* the device reported MOE_DEV_TIMEOUT */
    MOE_ERR_DEVICE_FAULT = -6        /* the device reported another MOE_DEV_* bit */
};
enum {                               /* bits of the device status word */
    MOE_DEV_BAD_EXPERT_ID = 1,       /* a topk id / log2phys entry outside [0, E) */
    MOE_DEV_BAD_OFFSETS = 2,         /* expert_offsets not non-decreasing within [0, rows] */
    MOE_DEV_TIMEOUT = 4              /* a bounded pipeline wait expired (about 1 s) */
};
enum { MOE_SCORING_SOFTMAX = 0, MOE_SCORING_SIGMOID = 1 };
enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_FP8_BLOCK128 = 1 };
enum { MOE_OUT_F32 = 0, MOE_OUT_BF16 = 1 };
enum { MOE_ACT_IDENTITY = 0, MOE_ACT_SILU_MUL = 1 };
/* Layout of an expert weight tensor W [groups, N, K] (w13, w2):
 *   MOE_LAYOUT_ROWS   row-major, K innermost;
 *   MOE_LAYOUT_TILES  128 x 128-byte tiles, each contiguous, tile-major: tile
 *                     (g, n/128, k/kt) holds rows n%128 of 128 bytes (kt = 128
 *                     e4m3 or 64 bf16 elements), and within row r the 16-byte
 *                     chunk c is stored at chunk position c ^ (r mod 8) (the
 *                     128-byte swizzle the tensor cores read), so a kernel
 *                     places a tile in shared memory with one 16 KB bulk copy.
 * moe_pack_expert_weights converts the first into the second.  Results do
 * not depend on the layout. */
enum { MOE_LAYOUT_ROWS = 0, MOE_LAYOUT_TILES = 1 };

/* ---- layer description -------------------------------------------------- */
typedef struct moe_config {
    int32_t hidden;          /* H; multiple of 128 */
    int32_t inter;           /* I, width of every expert (routed and shared); multiple of 128 */
    int32_t num_experts;     /* E routed experts, 1..1024 */
    int32_t num_shared;      /* S shared experts, 0..4, each of width I */
    int32_t top_k;           /* k, 1..16 */
    int32_t num_groups;      /* expert groups for group-limited routing (1 = none); divides E */
    int32_t topk_groups;     /* groups kept */
    int32_t group_topn;      /* a group's score is the sum of its best group_topn scores */
    int32_t scoring;         /* MOE_SCORING_* */
    int32_t norm_topk;       /* 1: divide the chosen weights by their sum */
    int32_t dtype;           /* MOE_DTYPE_*: weights/activations of the expert GEMMs */
    int32_t max_tokens;      /* largest T the workspace of moe_layer_forward is sized for */
    float routed_scaling;    /* factor on the routed weights (not on shared experts) */
} moe_config;

/* Device pointers to the layer's weights. */
typedef struct moe_weights {
    const void *w_gate;       /* bf16 [E, H], LOGICAL expert order */
    const float *e_bias;      /* fp32 [E] logical, selection-only bias (sigmoid); NULL = none */
    const float *logit_offset;/* fp32 [E] logical, added to the gate logits; NULL = none */
    const int32_t *log2phys;  /* int32 [E]: physical slot of each logical expert; NULL = identity */
    const void *w13;          /* [G, 2I, H]: rows [0, I) gate proj, [I, 2I) up proj; e4m3 or bf16 */
    const float *w13_scales;  /* fp32 [G, 2I/128, H/128], one per 128x128 block (FP8 only) */
    const void *w2;           /* [G, H, I] down proj; e4m3 or bf16 */
    const float *w2_scales;   /* fp32 [G, H/128, I/128] (FP8 only) */
    int32_t expert_layout;    /* MOE_LAYOUT_* of w13 and w2 (scales are always as above) */
} moe_weights;

/* ---- routing -------------------------------------------------------------
 * Gate logits l[t,e] = sum_h x[t,h] Wg[e,h] (+ logit_offset[e]) and top-k
 * selection (report, section "Overview": a light gating network chooses a
 * few experts per token; section "Load balancing across GPUs": after the
 * experts are permuted the gate must emit ids in the new order).
 *   x        bf16 [T, H];  w_gate bf16 [E, H] (logical order)
 *   e_bias   fp32 [E] or NULL (sigmoid scoring only)
 *   logit_offset fp32 [E] or NULL;  log2phys int32 [E] or NULL
 *   logits   fp32 [T, E], written (the gate logits, logical order)
 *   topk_ids int32 [T, k], written: PHYSICAL ids, slot j in descending
 *            selection score (ties: lower logical id first)
 *   topk_w   fp32 [T, k], written: routing weights of the slots
 * Logits are summed in a fixed order (lane-sliced fp32 FMA chains, then a
 * butterfly), so the ids are reproducible bit for bit.  Sigmoid scoring:
 * s = fp32(sigmoid(l)) evaluated in fp64, selection by s + bias, groups
 * scored by the sum of their top group_topn, weights s/sum(s) (x scaling).
 * Softmax scoring: selection by l; weights exp(l - max l) / sum over E (or
 * over the chosen k with norm_topk), each exponential in fp32 of the exact
 * difference, sums and quotient in fp64: within 5.4e-7 (relative) of the
 * fp64 softmax while l - max l > -87. */
MOE_API int moe_route(const moe_config *cfg, int32_t T, const void *x, const void *w_gate,
              const float *e_bias, const float *logit_offset, const int32_t *log2phys,
              float *logits, int32_t *topk_ids, float *topk_w,
              int32_t *dev_status, void *stream);

/* moe_route followed by the FP8 quantisation of x (moe_act_requant with
 * MOE_ACT_IDENTITY) in the launches of moe_route alone: the selection kernel
 * quantises each token's row while the gate logits are computed.  The same
 * results, bit for bit, as the two calls.  FP8 layers only (else
 * MOE_ERR_INVALID_ARG).  xq e4m3 [T, hidden] and xs fp32 [T, hidden/128]
 * (device, caller-owned); other arguments as moe_route.  x must not change
 * until the call's kernels have run (it is read while the logits are
 * computed). */
MOE_API int moe_route_quantize(const moe_config *cfg, int32_t T, const void *x, const void *w_gate,
                               const float *e_bias, const float *logit_offset,
                               const int32_t *log2phys, float *logits, int32_t *topk_ids,
                               float *topk_w, void *xq, float *xs, int32_t *dev_status,
                               void *stream);

/* ---- activation quantisation ----------------------------------------------
 * mode MOE_ACT_IDENTITY (FP8 layers): in bf16 [rows, H] -> out e4m3 [rows, H]
 *   and out_scales fp32 [rows, H/128]: per row and 128-column group,
 *   scale = amax/448 (IEEE fp32 division; 1 if amax = 0),
 *   code = e4m3(v / scale), round to nearest even, saturating.
 * mode MOE_ACT_SILU_MUL: in fp32 [rows, 2I] (gate | up halves), h =
 *   silu(gate) * up in fp32; FP8 layers quantise h as above into
 *   out e4m3 [rows, I] + out_scales [rows, I/128]; BF16 layers write
 *   out bf16 [rows, I] (out_scales unused, may be NULL).
 * rows_dev: NULL, or a device int32 holding the number of rows to process
 *   (clamped to `rows`); e.g. expert_offsets + G.
 * (SGLang/H20 article, section "MoE": the block-scale handling of the MoE
 * GEMMs; the activation format is the R1 FP8 layout, per token x 128.) */
MOE_API int moe_act_requant(const moe_config *cfg, int32_t mode, int32_t rows,
                    const int32_t *rows_dev, const void *in, void *out,
                    float *out_scales, void *stream);

/* ---- dispatch (permutation into per-expert rows) ---------------------------
 * topk_ids int32 [T, k] physical ids.  Routed slot i = t*k + j goes to row
 * expert_offsets[e] + (number of earlier slots with the same expert), so
 * rows of an expert are in increasing slot order (deterministic).  Shared
 * expert s of token t goes to row expert_offsets[E + s] + t.
 *   x_rows     e4m3 [T, H] (FP8) or bf16 [T, H] (BF16): rows to gather
 *   x_scales   fp32 [T, H/128] (FP8 only)
 *   expert_offsets int32 [G + 1], written: first row of every group
 *   src_of_row int32 [R_tot], written: the slot of each row (routed slots
 *              t*k + j; shared slots R + s*T + t)
 *   row_of_slot int32 [T, k], written (-1 for a slot whose id was invalid)
 *   xp         [R_tot, H] gathered rows (e4m3 or bf16), xp_scales fp32
 *              [R_tot, H/128] (FP8 only)
 *   ws         scratch of moe_permute_workspace_size bytes
 *   copy_max_group_rows  the rows of groups with more rows than this get their
 *              src_of_row / row_of_slot entries but are not copied into xp /
 *              xp_scales (a GEMM that gathers them from the token rows,
 *              moe_grouped_gemm_swiglu_gather, reads them there); INT32_MAX
 *              copies every row, < 0 is MOE_ERR_INVALID_ARG.
 * (report, sections "Overview" and "Compute-communication overlap": the
 * dispatch that carries each token to its experts.) */
MOE_API int moe_permute_workspace_size(const moe_config *cfg, int32_t T, size_t *bytes /* host */);
MOE_API int moe_permute(const moe_config *cfg, int32_t T, const int32_t *topk_ids,
                const void *x_rows, const float *x_scales,
                int32_t *expert_offsets, int32_t *src_of_row, int32_t *row_of_slot,
                void *xp, float *xp_scales, void *ws, size_t ws_bytes,
                int32_t copy_max_group_rows, int32_t *dev_status, void *stream);

/* moe_permute without a workspace argument.  The pages have no counterpart:
 * this entry serves callers that cannot allocate device memory, such as a
 * plugin inside a framework that owns every device allocation, or a
 * runtime held to a fixed, pre-reserved memory budget.  Arguments and
 * results are those of moe_permute minus ws/ws_bytes, copying every row.
 *   - Scratch lives in a static device array inside the library, 1 MiB per
 *     device (moe_permute_static_scratch_capacity()), held by every GPU that
 *     loads the library until the process exits.  A call whose scratch need
 *     (moe_permute_workspace_size) exceeds it returns
 *     MOE_ERR_UNSUPPORTED_SHAPE before enqueuing anything; for the R1
 *     shape (256 experts, top 8) that is above 21824 tokens.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is looked up again when the
 *     device's CUDA context has changed since (after a device reset the
 *     module holding the array is reloaded elsewhere), so the call stays
 *     valid across resets; the first call after a reset should again come
 *     before any capture.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing in it needs to start at zero (a call reads only words
 *     it wrote earlier).  Calls that overlap on the GPU (other streams, or
 *     concurrent graph branches) race on it: serialise them.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
MOE_API int moe_permute_static_scratch(const moe_config *cfg, int32_t T, const int32_t *topk_ids,
                                       const void *x_rows, const float *x_scales,
                                       int32_t *expert_offsets, int32_t *src_of_row,
                                       int32_t *row_of_slot, void *xp, float *xp_scales,
                                       int32_t *dev_status, void *stream);
MOE_API size_t moe_permute_static_scratch_capacity(void);

/* ---- group row windows --------------------------------------------------------
 * moe_grouped_gemm, moe_grouped_gemm_swiglu and moe_expert_ffn take a window
 * min_group_rows <= n <= max_group_rows: only the groups whose row count n
 * (expert_offsets[g+1] - expert_offsets[g]) lies in it are computed; the
 * output rows of the other groups are not written.  0 and INT32_MAX select
 * every group; min_group_rows < 0 is MOE_ERR_INVALID_ARG.  A batch can so
 * send its groups of few rows to one kernel and the rest to another: the
 * layer, for wide FP8 batches, runs moe_expert_ffn on the groups of at most
 * 32 rows and the two GEMMs on the others.  Results are bit-identical to a
 * call over every group. */

/* ---- grouped GEMM -----------------------------------------------------------
 * For every group g and row r in [expert_offsets[g], expert_offsets[g+1]):
 *   C[r, n] = sum_k A[r, k] * W[g, n, k]
 * FP8 (cfg->dtype = MOE_DTYPE_FP8_BLOCK128): A e4m3 [rows, K] with a_scales
 *   fp32 [rows, K/128]; W e4m3 [groups, N, K] with w_scales fp32
 *   [groups, N/128, K/128]; every 128-wide K block is scaled by
 *   a_scale[r, kb] * w_scale[g, n/128, kb] (fp32 accumulation).
 * BF16: A bf16 [rows, K], W bf16 [groups, N, K], scales unused.
 * w_layout: MOE_LAYOUT_* of W (else MOE_ERR_INVALID_ARG).
 * C: fp32 or bf16 (c_dtype = MOE_OUT_*) [rows, N]; rows outside every group
 *   are not written.  expert_offsets: device int32 [groups + 1].
 * N multiple of 128; K multiple of 128 and at most 7168 (FP8) or multiple
 * of 64 (BF16); groups <= 1024.
 * Tensor cores (tcgen05, accumulators in tensor memory) fed by TMA; weight
 * rows sit on the MMA's M side and the few token rows of an expert on its
 * N side (the SGLang/H20 article, section "SwapAB GEMM": map the token
 * dimension to the fine-grained side of the MMA for small, variable rows
 * per expert).  FP8 groups averaging 16 rows or more with fp32 C and N a
 * multiple of 256 swap back: 128 token rows on M against 256 output columns
 * on N; same bits. */
MOE_API int moe_grouped_gemm(const moe_config *cfg, int32_t groups, int32_t n_out, int32_t k_dim,
                     int32_t rows, const void *a, const float *a_scales,
                     const int32_t *expert_offsets, const void *w, const float *w_scales,
                     int32_t w_layout, void *c, int32_t c_dtype, int32_t min_group_rows,
                     int32_t max_group_rows, int32_t *dev_status, void *stream);

/* Grouped GEMM with the SwiGLU epilogue (gate/up GEMM and SiLU-mul fused):
 * for the rows r of group g, with W13[g] = [W_gate; W_up] ([2*inter, K]),
 *   g = A[r] W_gate^T, u = A[r] W_up^T (fp32, FP8 block scales as in
 *   moe_grouped_gemm), h = silu(g) * u (fp32), and
 *   FP8 layers: h quantised per row and 128-feature group as in
 *     moe_act_requant -> h e4m3 [rows, inter], h_scales fp32 [rows, inter/128];
 *   BF16 layers: h rounded to bf16 -> h bf16 [rows, inter] (h_scales unused).
 * Gives the same bits as moe_grouped_gemm (fp32 C) followed by
 * moe_act_requant(SILU_MUL), without writing the fp32 gate/up rows.  A tile
 * takes 128 gate rows and the matching 128 up rows, which share one
 * activation tile (the report's "horizontal fusion" of an expert's GEMMs,
 * section "Library optimisation").  FP8 groups averaging 16 rows or more
 * (rows >= 16 * groups) take a second kernel with the orientation swapped:
 * 128 token rows of one expert on the MMA's M side against those 256 weight
 * rows on N, so each thread promotes, applies SwiGLU to and quantises one
 * token row; same bits.  inter multiple of 128; K as in moe_grouped_gemm. */
MOE_API int moe_grouped_gemm_swiglu(const moe_config *cfg, int32_t groups, int32_t inter,
                                    int32_t k_dim, int32_t rows, const void *a,
                                    const float *a_scales, const int32_t *expert_offsets,
                                    const void *w13, const float *w13_scales, int32_t w_layout,
                                    void *h, float *h_scales, int32_t min_group_rows,
                                    int32_t max_group_rows, int32_t *dev_status,
                                    void *stream);

/* moe_grouped_gemm_swiglu without materialised activation rows: the rows of
 * each group are gathered from the token rows of x by the tensor cores' copy
 * engine (TMA tile::gather4, four rows per copy, straight into the MMA's
 * swizzled operand layout), the f1 row gather of the report's fused MoE
 * kernel (section "Library optimisation").  Row r (in expert_offsets' row
 * numbering) is token t(r) of slot src_of_row[r]: routed slots t*top_k + j
 * give t, the shared experts' slots T*top_k + i*T + t give t (moe_permute's
 * tables).  FP8 layers only (else MOE_ERR_INVALID_ARG).
 *   x_rows   e4m3 [T, k_dim] and x_scales fp32 [T, k_dim/128]: the token rows
 *            (moe_route_quantize's xq / xs)
 *   src_of_row int32 [rows]
 * Other arguments, results (h, h_scales rows in dispatch order) and the group
 * row window as moe_grouped_gemm_swiglu, whose token-rows-on-M kernel this is
 * (used for every batch size); the same result bits as that call on the
 * rows moe_permute gathers.  Not the layer's path: each gather4 moves 512
 * bytes, and the 32 of them a 128-row tile needs per 128-byte K block make
 * the copies, not the MMAs or the promotion, set the pace (same box, R1
 * layer: gate/up 1.87 -> 3.72 ms at 4096 tokens, against a 48 us saving in
 * the dispatch). */
MOE_API int moe_grouped_gemm_swiglu_gather(const moe_config *cfg, int32_t groups, int32_t inter,
                                           int32_t k_dim, int32_t rows, const void *x_rows,
                                           const float *x_scales, int32_t T,
                                           const int32_t *src_of_row,
                                           const int32_t *expert_offsets, const void *w13,
                                           const float *w13_scales, int32_t w_layout, void *h,
                                           float *h_scales, int32_t min_group_rows,
                                           int32_t max_group_rows, int32_t *dev_status,
                                           void *stream);

/* ---- the experts' FFN in one kernel ------------------------------------------/* ---- the experts' FFN in one kernel ------------------------------------------
 * For the rows r of every group g (offsets as in moe_grouped_gemm):
 *   g, u = A[r] W13[g]^T     (W13 [groups, 2*inter, hidden], A [rows, hidden];
 *                             FP8: e4m3 with block scales w13_scales fp32
 *                             [groups, 2*inter/128, hidden/128] and a_scales fp32
 *                             [rows, hidden/128]; BF16: bf16, scales unused),
 *   h    = silu(g) * u: FP8 quantised per row and 128-feature group
 *          -> h e4m3 [rows, inter], h_scales fp32 [rows, inter/128];
 *          BF16 rounded -> h bf16 [rows, inter] (h_scales unused),
 *   y[r] = h[r] W2[g]^T      (W2 [groups, hidden, inter], FP8 w2_scales fp32
 *                             [groups, hidden/128, inter/128]) -> y fp32 [rows, hidden].
 * The same bits as moe_grouped_gemm_swiglu followed by moe_grouped_gemm
 * (fp32 C), in one persistent launch: the report's fused MoE kernel
 * (section "Library optimisation") runs an expert's FFN as one kernel.
 * CTAs claim the gate/up tiles, then the down tiles, from a counter; a down
 * tile waits (bounded, about a second, else MOE_DEV_TIMEOUT) until the h
 * rows of its 32-row activation tile are complete, so no wave of either
 * GEMM ends with most of the GPU idle.
 *   sched: device scratch of at least moe_expert_ffn_sched_bytes(groups,
 *   rows) bytes, owned by the caller, cleared by the call on `stream`; one
 *   call at a time per buffer (else MOE_ERR_WORKSPACE_TOO_SMALL if short).
 * cfg supplies dtype, hidden and inter; groups <= 1024 (else
 * MOE_ERR_UNSUPPORTED_SHAPE); a, w13, w2, h and y 16-byte aligned; w_layout
 * the MOE_LAYOUT_* of w13 and w2. */
MOE_API size_t moe_expert_ffn_sched_bytes(int32_t groups, int32_t rows);
MOE_API int moe_expert_ffn(const moe_config *cfg, int32_t groups, int32_t rows, const void *a,
                           const float *a_scales, const int32_t *expert_offsets,
                           const void *w13, const float *w13_scales, const void *w2,
                           const float *w2_scales, int32_t w_layout, void *h,
                           float *h_scales, float *y, int32_t *sched, size_t sched_bytes,
                           int32_t min_group_rows, int32_t max_group_rows,
                           int32_t *dev_status, void *stream);

/* The experts' FFN on dispatched rows with the kernels moe_layer_forward
 * would pick for this batch: moe_expert_ffn for BF16 layers and for FP8
 * groups averaging fewer than 32 rows (rows < 32 * groups); otherwise
 * moe_expert_ffn on the groups of at most 32 rows, then
 * moe_grouped_gemm_swiglu and moe_grouped_gemm (down, fp32 y) on the groups
 * of more (row windows above).  Arguments, layouts, ownership and errors as
 * moe_expert_ffn over every group (sched is cleared on `stream`); every
 * choice gives the same result bits.  Used by the expert-parallel step, where the
 * rows a rank receives for its experts, and its shared-expert rows, are FFN
 * calls of their own. */
MOE_API int moe_experts_forward(const moe_config *cfg, int32_t groups, int32_t rows,
                                const void *a, const float *a_scales,
                                const int32_t *expert_offsets, const void *w13,
                                const float *w13_scales, const void *w2,
                                const float *w2_scales, int32_t w_layout, void *h,
                                float *h_scales, float *y, int32_t *sched, size_t sched_bytes,
                                int32_t *dev_status, void *stream);

/* Packs an expert weight tensor W [groups, n_out, k_dim] (e4m3 for FP8
 * layers, bf16 otherwise, per cfg->dtype) from MOE_LAYOUT_ROWS into
 * MOE_LAYOUT_TILES (w_tiled, same size, device, caller-owned, must not
 * overlap w).  The FFN streams every 128 x 128-byte weight tile as one
 * contiguous 16 KB read instead of 128 rows 7-14 KB apart (a same-box A/B
 * on the R1 decode layer: 1.626 -> 1.560 ms for the one-kernel FFN).
 * n_out multiple of 128; k_dim of 128 (e4m3) or 64 (bf16); 16-byte aligned
 * pointers. */
MOE_API int moe_pack_expert_weights(const moe_config *cfg, int32_t groups, int32_t n_out,
                                    int32_t k_dim, const void *w, void *w_tiled, void *stream);

/* ---- combine -------------------------------------------------------------------
 * out[t, :] = sum_s Y[expert_offsets[E+s] + t, :]
 *           + sum_j topk_w[t, j] * Y[row_of_slot[t, j], :]    (fp32, shared
 * first, then j ascending; slots with row -1 are skipped).
 *   y fp32 [R_tot, H] (the experts' outputs); out fp32 or bf16 [T, H]
 *   (out_dtype = MOE_OUT_*).
 * A gather per token: no atomics, no scatter (report, section "Overview":
 * the combine that brings expert outputs back to their tokens). */
MOE_API int moe_combine(const moe_config *cfg, int32_t T, const void *y, const int32_t *row_of_slot,
                const float *topk_w, const int32_t *expert_offsets, void *out,
                int32_t out_dtype, void *stream);

/* ---- the whole layer -------------------------------------------------------------
 * route (FP8: with the quantisation of x, as moe_route_quantize) -> permute
 * -> the experts' FFN -> combine, all
 * on `stream`.  The experts' FFN is
 *   BF16, and FP8 with groups averaging fewer than 32 rows (decode):
 *     moe_expert_ffn (one persistent kernel);
 *   FP8, groups averaging 32 rows or more: moe_expert_ffn on the groups of
 *     at most 32 rows, then moe_grouped_gemm_swiglu (its token-rows-on-M
 *     kernel) and moe_grouped_gemm down (the same orientation when hidden is
 *     a multiple of 256, else 64-row tiles) on the others;
 * all with the same result bits (fp32 expert outputs), and
 * all intermediates inside `ws` (size from moe_workspace_size for
 * cfg->max_tokens).  x bf16 [T, H]; out fp32 or bf16 [T, H].  T may be 0..
 * max_tokens.  The workspace's device status word is cleared at the start
 * of every call; read it with moe_get_device_status after the stream has
 * finished. */
MOE_API int moe_workspace_size(const moe_config *cfg, size_t *bytes /* host */);
MOE_API int moe_layer_forward(const moe_config *cfg, const moe_weights *w, int32_t T, const void *x,
                      void *out, int32_t out_dtype, void *ws, size_t ws_bytes, void *stream);

/* Byte offsets of the intermediates inside the layer workspace (host), for
 * callers that want to read routing results or rows per expert.  gate_up is
 * an empty region (no layer path keeps fp32 gate/up rows); it stays for
 * layout compatibility. */
typedef struct moe_ws_layout {
    size_t status, logits, topk_ids, topk_w, xq, xs, expert_offsets, src_of_row,
        row_of_slot, perm_scratch, xp, xp_scales, gate_up, h, h_scales, y, ffn_sched, total;
} moe_ws_layout;
MOE_API int moe_workspace_layout(const moe_config *cfg, moe_ws_layout *layout /* host */);

/* Synchronously reads the status word of a layer workspace (device) into
 * *status (host).  Returns MOE_OK when no bit is set, MOE_ERR_TIMEOUT when
 * MOE_DEV_TIMEOUT is set, MOE_ERR_DEVICE_FAULT for any other bit. */
MOE_API int moe_get_device_status(const void *ws, int32_t *status /* host */);

/* Static text for a MOE_OK / MOE_ERR_* code. */
MOE_API const char *moe_status_string(int32_t code);

/* What the last call on this host thread that returned MOE_ERR_CUDA failed
 * at: the CUDA runtime or driver call and its error text (e.g.
 * "cudaLaunchKernelEx: too many resources requested for launch").  Empty
 * until such a failure; a later successful call does not clear it.  The
 * pointer stays valid for the thread's lifetime. */
MOE_API const char *moe_last_error_detail(void);

/* Number of kernels moe_layer_forward enqueues for this configuration. */
MOE_API int moe_layer_kernel_count(const moe_config *cfg, int32_t T);

/* Measurement utility (no counterpart on the pages): streams `bytes` of device
 * memory at `src` through shared memory and discards them, so that the time
 * of the call (timed by the caller with events on `stream`) gives this GPU's
 * read-only HBM rate -- the denominator for kernels bound by streaming
 * weights, which a copy (read + write) figure understates.  One CTA per SM,
 * 64 KB bulk copies, a 3-deep ring.  src 16-byte aligned; bytes a multiple
 * of moe_stream_read_granule() (else MOE_ERR_INVALID_ARG); nothing is written
 * to global memory.  A bounded wait that expires sets MOE_DEV_TIMEOUT in
 * *dev_status (may be NULL). */
MOE_API size_t moe_stream_read_granule(void);
MOE_API int moe_stream_read(const void *src, size_t bytes, int32_t *dev_status, void *stream);

/* Self-test of the bounded waits (no counterpart on the pages: a robustness
 * check of this library).  Launches one warp that waits on a completed
 * mbarrier (must succeed) and on one nothing arrives on (must give up after
 * limit_ns, 1e3..1e8, setting MOE_DEV_TIMEOUT in *dev_status).  Writes
 * *dev_result = 1 (first wait passed) | 2 (second wait gave up).  The
 * kernel always returns; nothing traps. */
MOE_API int moe_selftest_bounded_wait(int32_t *dev_status, int64_t limit_ns, int32_t *dev_result,
                                      void *stream);

/* Self-test of the routing's sigmoid score (csrc/numerics.cuh sigmoid_score):
 * for i < n, fast[i] is the score as the selection kernel computes it (fp32
 * double-float arithmetic, the fp64 expression where that cannot decide the
 * rounding) and ref[i] = fp32(1 / (1 + exp(-logits[i]))) evaluated in fp64;
 * the two must be equal bit for bit.  *fallbacks (device int32, zeroed by the
 * caller) is incremented once per value that took the fp64 evaluation.  All
 * pointers are device pointers of n elements owned by the caller; the call is
 * asynchronous on `stream`.  MOE_ERR_INVALID_ARG: n < 0 or a null pointer. */
MOE_API int moe_selftest_sigmoid(const float *logits, int32_t n, float *fast, float *ref,
                                 int32_t *fallbacks, void *stream);

/* Self-test of moe_expert_ffn's inter-CTA wait (no counterpart on the pages:
 * a robustness check of this library).  Runs the one-kernel FFN on a tiny
 * problem (hidden 128, inter 256, one group, one row) whose scheduler
 * counter starts past the gate/up units, so the down unit waits for h rows
 * that no CTA will write: its bounded wait gives up after about a second,
 * sets MOE_DEV_TIMEOUT in *dev_status, and every CTA drains its copies and
 * MMAs, frees its tensor memory and exits; nothing traps and the context
 * stays usable.  scratch: device, 16-byte aligned, at least
 * moe_selftest_ffn_flag_timeout_scratch_bytes() bytes, owned by the caller
 * (cleared by the call). */
MOE_API size_t moe_selftest_ffn_flag_timeout_scratch_bytes(void);
MOE_API int moe_selftest_ffn_flag_timeout(void *scratch, size_t scratch_bytes,
                                          int32_t *dev_status, void *stream);

/* ---- continuous load balancing ------------------------------------------------
 * Report, section "Load balancing across GPUs": in serving, activation
 * frequencies are re-measured periodically and a new expert permutation is
 * generated from them.
 * moe_count_expert_rows: counts[p] += expert_offsets[p+1] - expert_offsets[p]
 *   for every routed expert p (PHYSICAL order), i.e. this batch's rows per
 *   expert; counts is a device int64 [E] accumulator owned by the caller.
 *   Exact integer sums: the result does not depend on launch order.
 * moe_relayout_experts: dst block p = src block src_slot[p] for p < groups,
 *   each block block_bytes long (a multiple of 16; e.g. one expert's W13,
 *   W2 or scales).  src_slot is a device int32 [groups] table; an entry
 *   outside [0, groups) copies nothing and sets MOE_DEV_BAD_EXPERT_ID in
 *   *dev_status (nullable).  src and dst must not overlap (checked).
 *   Applying a new permutation: with old/new logical->physical tables,
 *   src_slot[p] = old_log2phys[new_phys2log[p]] for routed p, and p itself for
 *   the shared experts; run it on a side stream into second buffers while the
 *   layer keeps serving, then switch pointers. */
MOE_API int moe_count_expert_rows(const moe_config *cfg, const int32_t *expert_offsets,
                                  int64_t *counts, void *stream);
/* SGLang/H20 article, section "Expert Affinity EPLB": track which experts a
 * token selects together.  coact[a*E + b] += 1 for every token of the
 * batch and every two of its k selected experts a != b, as LOGICAL ids
 * (topk_ids are physical; phys2log, device int32 [E], maps them back;
 * NULL = identity).  coact: device int64 [E, E] accumulator, symmetric.
 * Integer atomics: the sums do not depend on order.  Ids out of range are
 * skipped. */
MOE_API int moe_count_coactivation(const moe_config *cfg, int32_t T, const int32_t *topk_ids,
                                   const int32_t *phys2log, int64_t *coact, void *stream);
MOE_API int moe_relayout_experts(const void *src, void *dst, const int32_t *src_slot,
                                 int32_t groups, int64_t block_bytes, int32_t *dev_status,
                                 void *stream);

/* ---- host: balanced expert permutation ----------------------------------------------
 * Report, section "Load balancing across GPUs": from measured activation
 * counts, group the E experts into num_sets sets of E/num_sets with totals
 * as even as possible (a variant of balanced number partitioning) and
 * renumber them so each set is contiguous.  Objective: minimise the largest
 * set total.  Exact (branch and bound) when E <= 16, otherwise
 * cardinality-constrained greedy (largest first into the lightest open set)
 * followed by improving pairwise swaps.  Set s holds physical ids
 * [s*m, (s+1)*m), m = E/num_sets, logical ids ascending inside a set.
 *   counts    host int64 [E], >= 0
 *   log2phys  host int32 [E], written; phys2log host int32 [E], written
 *   max_over_mean host, written (may be NULL): largest set total / mean
 * Pure host code; usable without a GPU. */
MOE_API int expert_balance_permutation(const int64_t *counts, int32_t num_experts, int32_t num_sets,
                               int32_t *log2phys, int32_t *phys2log, double *max_over_mean);

/* Host: the set imbalance of a given permutation (the figure the report,
 * section "Load balancing across GPUs", quotes: the busiest set against the
 * average).  Set s holds physical ids [s*m, (s+1)*m), m = E/num_sets; the
 * load of a set is the sum of counts[e] over the logical experts e with
 * log2phys[e] in it.
 *   counts    host int64 [E], >= 0
 *   log2phys  host int32 [E], a permutation of 0..E-1 (NULL = identity)
 *   max_over_mean host, written: largest set load / mean set load (1 when
 *             every count is 0)
 * MOE_ERR_INVALID_ARG for a negative count, an id out of range or repeated,
 * or E not a multiple of num_sets.  Pure host code; usable without a GPU. */
MOE_API int expert_set_imbalance(const int64_t *counts, const int32_t *log2phys,
                                 int32_t num_experts, int32_t num_sets, double *max_over_mean);

/* Host: affinity-aware placement (SGLang/H20 article, section "Expert
 * Affinity EPLB").  From per-expert counts and the symmetric co-activation
 * matrix coact (host int64 [E, E]), group the experts into num_sets equal
 * sets that keep as much co-activation inside sets as possible while every
 * set total stays within max(L*, floor((1 + load_slack) * mean)), L* being
 * the largest set total of the balanced partition above.  Exact for
 * E <= 16, otherwise best-improvement swaps from the balanced partition.
 * Same layout rule and outputs as expert_balance_permutation, plus
 * *intra_fraction (nullable): co-activation kept inside sets / all of it. */
MOE_API int expert_affinity_permutation(const int64_t *counts, const int64_t *coact,
                                        int32_t num_experts, int32_t num_sets, double load_slack,
                                        int32_t *log2phys, int32_t *phys2log,
                                        double *max_over_mean, double *intra_fraction);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */

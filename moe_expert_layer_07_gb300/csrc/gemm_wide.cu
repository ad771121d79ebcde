// Gate/up GEMM with the SwiGLU + FP8 requantisation epilogue for wide FP8
// batches (expert groups averaging 16 rows or more), on the 5th-generation
// tensor cores:
//
//   g[r, j] = sum_k A[r, k] W13[e, j, k]       u[r, j] = sum_k A[r, k] W13[e, I + j, k]
//   h[r, j] = silu(g[r, j]) * u[r, j]          (block-scaled FP8 products, fp32 sums)
//   h is stored as e4m3 codes with one fp32 scale per row and 128 features.
//
// Orientation: the expert's token rows are the MMA's M side (128 per tile)
// and the weight rows its N side: 128 gate rows and the matching 128 up rows
// of W13, N = 256, one 128 x 256 x 32 MMA per 32 bytes of K.  Every TMEM lane
// is then one token row, so an epilogue thread
//   * promotes its row with ONE scalar factor per K block and weight block
//     (x_scale[r, kb] * w_scale[kb], the same rounded product as the other
//     kernels) instead of a factor per column read from shared memory;
//   * holds the gate and up sums of the same 64 features, so SwiGLU is formed
//     in its own registers, and the row's FP8 group maximum needs a single
//     exchange with the thread that holds the other 64 features.
// With the whole N = 256 in one tile, a weight tile is read once per 128
// token rows of its expert (decode-style 64-row tiles read it once per 64),
// and h leaves as FP8 codes: no fp32 gate/up rows and no SiLU-mul launch.
//
// One persistent CTA per SM (its 4 x 48 KB ring and the 512 TMEM columns of
// two 128 x 256 fp32 accumulators fill the SM), 10 warps:
//   warp 0      TMA producer: per K block one 16 KB box of gate rows, one of
//               up rows (row-major weights, or two contiguous 16 KB tiles of
//               packed weights) and ceil(rows/32) 32-row activation boxes.
//   warp 1      MMA issuer (one thread), accumulators alternate between the
//               two TMEM buffers per K block; completion via tcgen05.commit.
//   warps 2..9  epilogue: warp w reads TMEM lane quarter (w & 3) -- token rows
//               [32 (w & 3), +32) -- and features [64 h, +64) of the tile,
//               h = (w - 2) >> 2: gate columns [64 h, +64) and up columns
//               [128 + 64 h, +64).  It frees the accumulator as soon as its
//               loads have landed and promotes from registers.
// Work units are (group, 128-feature tile of h, 128-row token tile), token
// tile fastest so that the tiles sharing a weight tile run side by side and
// share its L2 copy.  The tile table is built on the device from the expert
// offsets (no host sync; graph-capturable).  Every wait is bounded: after
// about a second the CTA records MOE_DEV_TIMEOUT, drains its copies and MMAs,
// frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "numerics.cuh"
#include "ptx.cuh"
#include "tma_host.h"

namespace moe {
namespace {

constexpr int kTM = 128;            // token rows per tile (MMA M)
constexpr int kTN = 256;            // weight rows per tile: 128 gate + 128 up (MMA N)
constexpr int kStages = 4;
constexpr int kABytes = kTM * 128;  // token rows x 128 bytes of K
constexpr int kBBytes = kTN * 128;  // weight rows x 128 bytes of K
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 1024;   // + 1024-byte alignment slack
constexpr int kABox = 32;           // token rows per activation TMA box
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTmemCols = 2 * kTN;  // two accumulators
constexpr int kMaxGroups = 1024;
static_assert(kSmemBytes + 8 * (kMaxGroups + 1) + 4 * 2 * 2 * kTM + 256 <= 227 * 1024,
              "shared memory");

struct WideArgs {
    int groups, inter, k_dim, rows;
    const int32_t *offsets;
    const float *a_scales;   // [rows, k_dim / 128]
    const float *w_scales;   // [groups, 2 inter / 128, k_dim / 128]
    uint8_t *h;              // [rows, inter] e4m3
    float *h_scales;         // [rows, inter / 128]
    int w_tiled;             // W13 in MOE_LAYOUT_TILES
    int32_t *status;
};

struct WTile {
    int g, nt, row0, nvalid;
};

// Tile t -> (group, feature tile nt, first token row, valid rows); s_tiles
// holds each group's first tile (a prefix over groups).
__device__ __forceinline__ WTile decode_wtile(int t, int G, int NT, const int *s_tiles,
                                              const int *s_off) {
    int lo = 0, hi = G;   // s_tiles[lo] <= t < s_tiles[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tiles[mid] <= t) lo = mid;
        else hi = mid;
    }
    WTile w;
    w.g = lo;
    const int rows = s_off[lo + 1] - s_off[lo];
    const int mtiles = (rows + kTM - 1) / kTM;
    const int local = t - s_tiles[lo];
    w.nt = local / mtiles;
    const int mt = local - w.nt * mtiles;
    w.row0 = s_off[lo] + mt * kTM;
    w.nvalid = min(kTM, rows - mt * kTM);
    (void)NT;
    return w;
}

__device__ __forceinline__ float lo_f(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

__global__ void __launch_bounds__(kThreads, 1)
    swiglu_wide_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmA, const WideArgs args) {
    using namespace ptx;
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t acc_full[2];
    __shared__ __align__(8) uint64_t acc_empty[2];
    __shared__ __align__(8) uint64_t amax_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_abort, s_bad;
    __shared__ int s_off[kMaxGroups + 1];
    __shared__ int s_tiles[kMaxGroups + 1];
    // per tile parity: each warpgroup's |h| maximum of every token row
    __shared__ float s_amax[2][2][kTM];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem_base = (smem_u32(dsmem) + 1023u) & ~1023u;
    const int G = args.groups;
    const int NT = args.inter / 128;            // feature tiles of h per group
    const int MTW = 2 * NT;                      // 128-row blocks of W13 per group
    const int KB = args.k_dim / 128;
    volatile int *abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), kEpiWarps);
            mbar_init(smem_u32(&amax_bar[b]), kEpiWarps);
        }
        mbar_init(smem_u32(&drain_bar), 1);
        s_abort = 0;
        s_bad = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmA);
    }
    pdl_wait();   // the set-up above overlaps the previous kernel's tail
    for (int i = threadIdx.x; i <= G; i += kThreads) s_off[i] = args.offsets[i];
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += kThreads) {
        const int a = s_off[g], b = s_off[g + 1];
        if (a < 0 || b < a || b > args.rows) s_bad = 1;
    }
    __syncthreads();
    if (warp == 0 && !s_bad) {   // tile prefix over groups: lane L owns a contiguous run
        const int per = (G + 31) / 32;
        const int g0 = lane * per;
        int local = 0;
        for (int q = 0; q < per; ++q) {
            const int g = g0 + q;
            if (g < G) local += NT * ((s_off[g + 1] - s_off[g] + kTM - 1) / kTM);
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        int run = incl - local;
        for (int q = 0; q < per; ++q) {
            const int g = g0 + q;
            if (g < G) {
                s_tiles[g] = run;
                run += NT * ((s_off[g + 1] - s_off[g] + kTM - 1) / kTM);
            }
        }
        if (lane == 31) s_tiles[G] = incl;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    const int total_tiles = s_bad ? 0 : s_tiles[G];
    if (s_bad && threadIdx.x == 0 && blockIdx.x == 0 && args.status)
        atomicOr(args.status, MOE_DEV_BAD_OFFSETS);

    if (warp == 0) {
        // ------------------------------ TMA producer
        if (lane == 0) {
            // A weight tile is read by every token tile of its group: those
            // run on neighbouring CTAs at about the same time and share the L2
            // copy.  An activation tile is re-read by every feature tile.
            const uint64_t pol_w_once = policy_evict_first();
            const uint64_t pol_w_shared = policy_evict_normal();
            const uint64_t pol_a = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0, issued = 0, parity_bits = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const WTile tl = decode_wtile(t, G, NT, s_tiles, s_off);
                const int nbox = (tl.nvalid + kABox - 1) / kABox;
                const uint32_t bytes = kBBytes + nbox * kABox * 128;
                const int grow = tl.g * 2 * args.inter + tl.nt * 128;   // row-major: gate rows
                const int urow = grow + args.inter;                     // up rows
                const int tb = (tl.g * MTW + tl.nt) * KB;                // tiles: gate blocks
                const int tbu = tb + NT * KB;                           // up blocks
                const uint64_t pol_w =
                    (s_off[tl.g + 1] - s_off[tl.g] > kTM) ? pol_w_shared : pol_w_once;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag,
                                      args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_base + stage * kStageBytes;
                    const uint32_t sb = sa + kABytes;
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    if (args.w_tiled) {
                        tma_load_2d(sb, &tmW, 0, (tb + kb) * 128, fb, pol_w);
                        tma_load_2d(sb + 128 * 128, &tmW, 0, (tbu + kb) * 128, fb, pol_w);
                    } else {
                        tma_load_2d(sb, &tmW, kb * 128, grow, fb, pol_w);
                        tma_load_2d(sb + 128 * 128, &tmW, kb * 128, urow, fb, pol_w);
                    }
                    for (int b = 0; b < nbox; ++b)
                        tma_load_2d(sa + b * kABox * 128, &tmA, kb * 128, tl.row0 + b * kABox, fb,
                                    pol_a);
                    issued |= 1u << stage;
                    parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {   // let every copy in flight land before the CTA exits
                for (int s = 0; s < kStages; ++s)
                    if ((issued >> s) & 1u) wait_drain(smem_u32(&full_bar[s]), (parity_bits >> s) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3(kTM, kTN);
            int stage = 0, ab = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bounded(smem_u32(&acc_empty[ab]), aphase ^ 1u, abort_flag,
                                      args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (!wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag, args.status,
                                      MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_base + stage * kStageBytes;
                    const uint64_t da = sdesc_k_sw128(sa);
                    const uint64_t db = sdesc_k_sw128(sa + kABytes);
                    const uint32_t d = tmem_base + (uint32_t)(ab * kTN);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)   // 4 x 32 bytes of K
                        mma_f8f6f4(d, da + 2 * kk, db + 2 * kk, idesc, kk > 0);
                    mma_commit(smem_u32(&empty_bar[stage]));
                    mma_commit(smem_u32(&acc_full[ab]));
                    if (++ab == 2) {
                        ab = 0;
                        aphase ^= 1u;
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every MMA issued by this thread completes before teardown
            mma_commit(smem_u32(&drain_bar));
            wait_drain(smem_u32(&drain_bar), 0);
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue (warps 2 .. 9)
        const int q = warp & 3;                   // TMEM lanes [32q, 32q + 32): token rows
        const int wgp = (warp - 2) >> 2;          // features [64 wgp, 64 wgp + 64) of the tile
        const int m = q * 32 + lane;              // this thread's token row within the tile
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
        const uint32_t col_g = (uint32_t)(wgp * 64), col_u = (uint32_t)(128 + wgp * 64);
        int ab = 0, it = 0;
        uint32_t aphase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++it) {
            const WTile tl = decode_wtile(t, G, NT, s_tiles, s_off);
            const bool valid = m < tl.nvalid;
            const int row = tl.row0 + (valid ? m : 0);
            const float *xsp = args.a_scales + (size_t)row * KB;
            const float *wsp = args.w_scales + ((size_t)tl.g * MTW + tl.nt) * KB;
            const int up_off = NT * KB;   // the up rows' block scales follow the gate rows'
            uint64_t ag[32], au[32];   // columns (2p, 2p + 1) of this thread's 64 features
#pragma unroll
            for (int p = 0; p < 32; ++p) ag[p] = au[p] = 0ull;
            // scales one K block ahead of their use
            float xs_n = xsp[0], wg_n = wsp[0], wu_n = wsp[up_off];
            for (int kb = 0; kb < KB; ++kb) {
                const float xs = xs_n, wsg = wg_n, wsu = wu_n;
                if (kb + 1 < KB) {
                    xs_n = xsp[kb + 1];
                    wg_n = wsp[kb + 1];
                    wu_n = wsp[up_off + kb + 1];
                }
                const float fg = __fmul_rn(xs, wsg), fu = __fmul_rn(xs, wsu);
                const uint64_t pfg = pack2(__float_as_uint(fg), __float_as_uint(fg));
                const uint64_t pfu = pack2(__float_as_uint(fu), __float_as_uint(fu));
                if (!wait_bounded(smem_u32(&acc_full[ab]), aphase, abort_flag, args.status,
                                  MOE_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t acc = lane_base + (uint32_t)(ab * kTN);
                uint32_t v[16];
#pragma unroll
                for (int c = 0; c < 8; ++c) {   // 16 columns at a time: gate 0-63, then up 0-63
                    tmem_ld16(acc + (c < 4 ? col_g : col_u) + (uint32_t)((c & 3) * 16), v);
                    tmem_wait_ld(v);
                    if (c == 7) {   // all of this K block is in registers: free the accumulator
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
                    }
                    uint64_t *a = (c < 4 ? ag : au) + (c & 3) * 8;
                    const uint64_t f = c < 4 ? pfg : pfu;
#pragma unroll
                    for (int j = 0; j < 8; ++j) a[j] = fma2(pack2(v[2 * j], v[2 * j + 1]), f, a[j]);
                }
                if (++ab == 2) {
                    ab = 0;
                    aphase ^= 1u;
                }
            }
            if (!ok) break;
            // h = silu(gate) * up for this thread's 64 features of its row; the
            // row's group maximum over all 128 features through shared memory
            float amax = 0.0f;
#pragma unroll
            for (int p = 0; p < 32; ++p) {
                const float h0 = silu_mul(lo_f(ag[p]), lo_f(au[p]));
                const float h1 = silu_mul(hi_f(ag[p]), hi_f(au[p]));
                ag[p] = pack2(__float_as_uint(h0), __float_as_uint(h1));
                amax = fmaxf(amax, fmaxf(fabsf(h0), fabsf(h1)));
            }
            const int par = it & 1;
            s_amax[par][wgp][m] = amax;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&amax_bar[par]));
            if (!wait_bounded(smem_u32(&amax_bar[par]), ((uint32_t)it >> 1) & 1u, abort_flag,
                              args.status, MOE_DEV_TIMEOUT)) {
                ok = false;
                break;
            }
            const float sc = fp8_group_scale(fmaxf(s_amax[par][0][m], s_amax[par][1][m]));
            if (valid) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint64_t a0 = ag[2 * i], a1 = ag[2 * i + 1];
                    w[i] = (uint32_t)fp8_code(lo_f(a0), sc) | ((uint32_t)fp8_code(hi_f(a0), sc) << 8) |
                           ((uint32_t)fp8_code(lo_f(a1), sc) << 16) |
                           ((uint32_t)fp8_code(hi_f(a1), sc) << 24);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(args.h + (size_t)(tl.row0 + m) * args.inter +
                                                       tl.nt * 128 + wgp * 64);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                if (wgp == 0) args.h_scales[(size_t)(tl.row0 + m) * NT + tl.nt] = sc;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

int launch_swiglu_wide(int groups, int inter, int k_dim, int rows, const void *a,
                       const float *a_scales, const int32_t *offsets, const void *w13,
                       const float *w13_scales, bool w_tiled, void *h, float *h_scales,
                       int32_t *status, cudaStream_t s) {
    if (rows == 0) return MOE_OK;
    static std::once_flag attr_once[64];
    static int attr_rc[64];
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return cuda_fail("device ordinal beyond 63");
    std::call_once(attr_once[dev], [&] {
        attr_rc[dev] = (int)cudaFuncSetAttribute(swiglu_wide_kernel,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            kSmemBytes);
    });
    if (attr_rc[dev]) return cuda_fail("cudaFuncSetAttribute", (cudaError_t)attr_rc[dev]);
    WideArgs args;
    args.groups = groups;
    args.inter = inter;
    args.k_dim = k_dim;
    args.rows = rows;
    args.offsets = offsets;
    args.a_scales = a_scales;
    args.w_scales = w13_scales;
    args.h = static_cast<uint8_t *>(h);
    args.h_scales = h_scales;
    args.w_tiled = w_tiled;
    args.status = status;
    const int KB = k_dim / 128;
    CUtensorMap tmW, tmA;
    const bool tmw_ok =
        w_tiled ? encode_2d(&tmW, w13, true, 128, (uint64_t)groups * 2 * inter * KB, 128)
                : encode_2d(&tmW, w13, true, (uint64_t)k_dim, (uint64_t)groups * 2 * inter, 128);
    if (!tmw_ok) return cuda_fail("cuTensorMapEncodeTiled (weights)");
    if (!encode_2d(&tmA, a, true, (uint64_t)k_dim, (uint64_t)rows, kABox))
        return cuda_fail("cuTensorMapEncodeTiled (activations)");
    const int64_t tiles_bound = (int64_t)(inter / 128) * (groups + ceil_div(rows, kTM));
    const int grid = (int)std::min<int64_t>((int64_t)sm_count(), tiles_bound);
    if (grid <= 0) return MOE_OK;
    if (launch_dependent(swiglu_wide_kernel, dim3(grid), dim3(kThreads), kSmemBytes, s, tmW, tmA,
                         args))
        return MOE_ERR_CUDA;
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace moe

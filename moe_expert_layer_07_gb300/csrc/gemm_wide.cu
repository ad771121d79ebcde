// Grouped FP8 GEMMs for wide batches (expert groups averaging 16 rows or
// more) with the token rows on the MMA's M side, on the 5th-generation tensor
// cores.  Two epilogues:
//
//   SwiGLU (gate/up):  g[r, j] = sum_k A[r, k] W13[e, j, k],
//                      u[r, j] = sum_k A[r, k] W13[e, I + j, k],
//                      h[r, j] = silu(g) * u, stored as e4m3 codes with one
//                      fp32 scale per row and 128 features;
//   plain (down):      C[r, n] = sum_k A[r, k] W[e, n, k], stored as fp32;
// both with 128 x 128 FP8 block scales, promoted per 128-wide K block in
// fp32 in the order the other kernels use (same result bits).
//
// Orientation: 128 token rows of one expert are the MMA's M side and 256
// weight rows its N side -- the gate rows of 128 features and the matching
// up rows (SwiGLU), or 256 consecutive output columns (plain) -- one
// 128 x 256 x 32 MMA per 32 bytes of K.  Every TMEM lane is one token row, so
// an epilogue thread promotes its row with ONE scalar factor per K block and
// weight block (x_scale[r, kb] * w_scale[kb], the same rounded product as the
// other kernels) instead of a factor per column read from shared memory.
// SwiGLU is formed in the thread's registers (it holds the gate and up sums
// of the same 64 features) and the row's FP8 group maximum needs a single
// exchange with the thread that holds the other 64 features; the plain
// epilogue stages each warp's 32 rows x 32 columns in 128-byte-swizzled
// shared memory and writes them with a TMA store.  With the whole N = 256 in
// one tile, a weight tile is read once per 128 token rows of its expert
// (decode-style 64-row tiles read it once per 64), and the gate/up GEMM
// leaves h as FP8 codes: no fp32 gate/up rows, no SiLU-mul launch.
//
// One persistent CTA per SM (its ring and the 512 TMEM columns of two
// 128 x 256 fp32 accumulators fill the SM), 10 warps:
//   warp 0      TMA producer: per K block two 16 KB boxes of weight rows
//               (row-major weights, or two contiguous 16 KB tiles of packed
//               weights) and ceil(rows/64) 64-row activation boxes -- or, in
//               the SwiGLU kernel's gather mode, ceil(rows/4) gather4 copies
//               of token rows of x straight into the tile's swizzled rows
//               (the row gather of the dispatch, without materialised rows).
//   warp 1      MMA issuer (one thread); the accumulator alternates between
//               the two TMEM buffers per K block; completion via tcgen05.commit.
//   warps 2..9  epilogue: warp w reads TMEM lane quarter (w & 3) -- token rows
//               [32 (w & 3), +32) -- and warpgroup h = (w - 2) >> 2 takes
//               columns: SwiGLU, gate [64 h, +64) and up [128 + 64 h, +64)
//               (features [64 h, +64)); plain, [128 h, +128) (weight block
//               2 nt + h).  It frees the accumulator as soon as its loads have
//               landed and promotes from registers.
// Work units are (group, 256-column tile, 128-row token tile), token tile
// fastest so that the tiles sharing a weight tile run side by side and share
// its L2 copy.  The tile table is built on the device from the expert offsets
// (no host sync; graph-capturable).  Every wait is bounded: after about a
// second the CTA records MOE_DEV_TIMEOUT, drains its copies, MMAs and stores,
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
constexpr int kTN = 256;            // weight rows per tile (MMA N)
constexpr int kABytes = kTM * 128;  // token rows x 128 bytes of K
constexpr int kBBytes = kTN * 128;  // weight rows x 128 bytes of K
constexpr int kStageBytes = kABytes + kBBytes;
// token rows per activation TMA box.  The count of TMA copies per stage sets
// the pace here: 64-row boxes (two per full tile) against 32-row ones made
// the 4096-token layer's gate/up launch 1.670 -> 1.522 ms and its down
// launch 1.010 -> 0.931 ms; one 128-row box was about as fast on full tiles
// and slower on the ragged ones it over-reads.
constexpr int kABox = 64;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTmemCols = 2 * kTN;  // two accumulators
constexpr int kMaxGroups = 1024;
constexpr int kOutBuf = 32 * 128;   // plain: one warp's 32 rows x 32 fp32 columns

template <bool SW, int ST>
struct WideShape {
    // the plain epilogue's store buffers (two per epilogue warp) take the
    // room of a fourth stage
    static constexpr int kStages = ST;
    static constexpr int kOutBytes = SW ? 0 : 2 * kEpiWarps * kOutBuf;
    static constexpr int kSmemBytes = kStages * kStageBytes + kOutBytes + 1024;
    static_assert(kSmemBytes + 8 * (kMaxGroups + 1) + 4 * 2 * 2 * kTM + 256 <= 227 * 1024,
                  "shared memory");
};

struct WideArgs {
    int groups, n_out, k_dim, rows;   // n_out: 2 * inter (SwiGLU) or the columns of C
    const int32_t *offsets;
    const float *a_scales;   // [rows, k_dim / 128]
    const float *w_scales;   // [groups, n_out / 128, k_dim / 128]
    uint8_t *h;              // SwiGLU: [rows, n_out / 2] e4m3
    float *h_scales;         // SwiGLU: [rows, n_out / 256]
    float *c;                // plain: [rows, n_out] fp32
    int w_tiled;             // W in MOE_LAYOUT_TILES (tiles read by 16 KB bulk copies)
    const uint8_t *w;        // W bytes
    int min_rows, max_rows;  // groups whose row count lies outside are skipped
    // Row gather (SwiGLU): with src_of_row set, row r of a tile is token
    // t(r)'s row of the [T, k_dim] activations that tmA then maps (one row per
    // box), fetched by TMA gather4, and its scales are x_scales[t(r)]; t(r)
    // follows the dispatch's slot numbering (token_of_slot).
    const int32_t *src_of_row;   // [rows]: the slot of each row; null: A in row order
    const float *x_scales;       // [T, k_dim / 128]
    int T, k;
    int32_t *status;
};

// Token of dispatch slot s: routed slots t k + j, then the shared experts'
// slots T k + i T + t.  Clamped into [0, T) so that a gather stays in bounds
// whatever the table holds.
__device__ __forceinline__ int token_of_slot(int s, int T, int k) {
    const int R = T * k;
    const int t = s < R ? s / k : (s - R) % T;
    return min(max(t, 0), T - 1);
}

struct WTile {
    int g, nt, row0, nvalid;
};

// Tile t -> (group, column tile nt, first token row, valid rows); s_tiles
// holds each group's first tile (a prefix over groups).
__device__ __forceinline__ WTile decode_wtile(int t, int G, const int *s_tiles, const int *s_off) {
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
    return w;
}

__device__ __forceinline__ float lo_f(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_f(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// A register file of 64K words is split over the SM's four sub-partitions;
// with 10 warps two sub-partitions hold 3 warps, so a thread gets at most
// 16384 / 96 -> 168 registers.
template <bool SW, bool GATHER, int ST>
__global__ void __launch_bounds__(kThreads, 1)
    wide_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmC, const WideArgs args) {
    using namespace ptx;
    using Sh = WideShape<SW, ST>;
    constexpr int kStages = Sh::kStages;
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
    // SwiGLU, per tile parity: each warpgroup's |h| maximum of every token row
    __shared__ float s_amax[2][2][kTM];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem_base = (smem_u32(dsmem) + 1023u) & ~1023u;
    const int G = args.groups;
    const int MTW = args.n_out / 128;   // 128-row weight blocks per group
    const int NT = MTW / 2;             // 256-row weight tiles per group
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
        if (!SW) tma_prefetch_desc(&tmC);
    }
    pdl_wait();   // the set-up above overlaps the previous kernel's tail
    for (int i = threadIdx.x; i <= G; i += kThreads) s_off[i] = args.offsets[i];
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += kThreads) {
        const int a = s_off[g], b = s_off[g + 1];
        if (a < 0 || b < a || b > args.rows) s_bad = 1;
    }
    __syncthreads();
    // token tiles of group g; none for groups outside the row window
    auto mtiles_of = [&](int g) {
        const int n = s_off[g + 1] - s_off[g];
        return (n < args.min_rows || n > args.max_rows) ? 0 : (n + kTM - 1) / kTM;
    };
    if (warp == 0 && !s_bad) {   // tile prefix over groups: lane L owns a contiguous run
        const int per = (G + 31) / 32;
        const int g0 = lane * per;
        int local = 0;
        for (int q = 0; q < per; ++q) {
            const int g = g0 + q;
            if (g < G) local += NT * mtiles_of(g);
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
                run += NT * mtiles_of(g);
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
      if constexpr (GATHER) {
        // ------------------------------ TMA producer (gather mode)
        // Lane 0 waits for free stages and loads the weight boxes; every lane
        // L then fetches token rows 4L .. 4L + 3 of the tile with one gather4.
        constexpr bool gather = true;
        // A weight tile is read by every token tile of its group: those
        // run on neighbouring CTAs at about the same time and share the L2
        // copy.  An activation tile is re-read by every column tile.
        const uint64_t pol_w_once = policy_evict_first();
        const uint64_t pol_w_shared = policy_evict_normal();
        const uint64_t pol_a = policy_evict_last();
        int stage = 0;
        uint32_t phase = 0, issued = 0, parity_bits = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            const WTile tl = decode_wtile(t, G, s_tiles, s_off);
            int tok[4] = {0, 0, 0, 0};
            int ngather = 0;
            if (gather) {   // this lane's four rows (the tile's last row repeats past nvalid)
                ngather = (tl.nvalid + 3) / 4;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = min(4 * lane + i, tl.nvalid - 1);
                    tok[i] = token_of_slot(args.src_of_row[tl.row0 + r], args.T, args.k);
                }
            }
            const int nbox = gather ? 0 : (tl.nvalid + kABox - 1) / kABox;
            const uint32_t bytes = kBBytes + (uint32_t)(gather ? ngather * 4 : nbox * kABox) * 128;
            // the two 128-row weight blocks of the tile: SwiGLU, gate
            // block nt and up block NT + nt; plain, blocks 2 nt, 2 nt + 1
            const int b0 = tl.g * MTW + (SW ? tl.nt : 2 * tl.nt);
            const int b1 = SW ? b0 + NT : b0 + 1;
            const uint64_t pol_w =
                (s_off[tl.g + 1] - s_off[tl.g] > kTM) ? pol_w_shared : pol_w_once;
            for (int kb = 0; kb < KB; ++kb) {
                int free_stage = 1;
                if (lane == 0)
                    free_stage = wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag,
                                              args.status, MOE_DEV_TIMEOUT);
                if (!__shfl_sync(0xffffffffu, free_stage, 0)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = smem_base + stage * kStageBytes;
                const uint32_t sb = sa + kABytes;
                const uint32_t fb = smem_u32(&full_bar[stage]);
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, bytes);
                    if (args.w_tiled) {   // tile (block b, K block kb): 16 KB at (b KB + kb) 16 KB
                        bulk_load(sb, args.w + (size_t)(b0 * KB + kb) * 16384, 16384, fb, pol_w);
                        bulk_load(sb + 128 * 128, args.w + (size_t)(b1 * KB + kb) * 16384, 16384, fb,
                                  pol_w);
                    } else {
                        tma_load_2d(sb, &tmW, kb * 128, b0 * 128, fb, pol_w);
                        tma_load_2d(sb + 128 * 128, &tmW, kb * 128, b1 * 128, fb, pol_w);
                    }
                    for (int b = 0; b < nbox; ++b)
                        tma_load_2d(sa + b * kABox * 128, &tmA, kb * 128, tl.row0 + b * kABox, fb,
                                    pol_a);
                }
                __syncwarp();   // the stage's byte count is posted before any gather lands
                if (lane < ngather)
                    tma_gather4(sa + lane * 4 * 128, &tmA, kb * 128, tok[0], tok[1], tok[2],
                                tok[3], fb, pol_a);
                issued |= 1u << stage;
                parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {   // let every copy in flight land before the CTA exits
            for (int s = 0; s < kStages; ++s)
                if ((issued >> s) & 1u) wait_drain(smem_u32(&full_bar[s]), (parity_bits >> s) & 1u);
        }
        __syncwarp();
      } else {
        // ------------------------------ TMA producer
        if (lane == 0) {
            // A weight tile is read by every token tile of its group: those
            // run on neighbouring CTAs at about the same time and share the L2
            // copy.  An activation tile is re-read by every column tile.
            const uint64_t pol_w_once = policy_evict_first();
            const uint64_t pol_w_shared = policy_evict_normal();
            const uint64_t pol_a = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0, issued = 0, parity_bits = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const WTile tl = decode_wtile(t, G, s_tiles, s_off);
                const int nbox = (tl.nvalid + kABox - 1) / kABox;
                const uint32_t bytes = kBBytes + nbox * kABox * 128;
                // the two 128-row weight blocks of the tile: SwiGLU, gate
                // block nt and up block NT + nt; plain, blocks 2 nt, 2 nt + 1
                const int b0 = tl.g * MTW + (SW ? tl.nt : 2 * tl.nt);
                const int b1 = SW ? b0 + NT : b0 + 1;
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
                    if (args.w_tiled) {   // tile (block b, K block kb): 16 KB at (b KB + kb) 16 KB
                        bulk_load(sb, args.w + (size_t)(b0 * KB + kb) * 16384, 16384, fb, pol_w);
                        bulk_load(sb + 128 * 128, args.w + (size_t)(b1 * KB + kb) * 16384, 16384, fb,
                                  pol_w);
                    } else {
                        tma_load_2d(sb, &tmW, kb * 128, b0 * 128, fb, pol_w);
                        tma_load_2d(sb + 128 * 128, &tmW, kb * 128, b1 * 128, fb, pol_w);
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
      }
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
        const int wgp = (warp - 2) >> 2;          // warpgroup: its share of the tile's columns
        const int m = q * 32 + lane;              // this thread's token row within the tile
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
        // plain: this warp's two 32-row x 32-column store buffers
        const uint32_t obuf = smem_base + kStages * kStageBytes + (warp - 2) * 2 * kOutBuf;
        int ab = 0, it = 0, nstore = 0;
        uint32_t aphase = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++it) {
            const WTile tl = decode_wtile(t, G, s_tiles, s_off);
            const bool valid = m < tl.nvalid;
            const int row = tl.row0 + (valid ? m : 0);
            const float *xsp;
            if constexpr (GATHER)
                xsp = args.x_scales + (size_t)token_of_slot(args.src_of_row[row], args.T, args.k) * KB;
            else
                xsp = args.a_scales + (size_t)row * KB;
            // block scales: SwiGLU, gate block nt (chunks 0-3) and up block
            // NT + nt (chunks 4-7); plain, block 2 nt + wgp for all chunks
            const float *wsp =
                args.w_scales + ((size_t)tl.g * MTW + (SW ? tl.nt : 2 * tl.nt + wgp)) * KB;
            const int up_off = SW ? NT * KB : 0;
            uint64_t acc[64];   // column pairs (2p, 2p + 1); SwiGLU: gate 0-31, up 32-63
#pragma unroll
            for (int p = 0; p < 64; ++p) acc[p] = 0ull;
            // scales one K block ahead of their use
            float xs_n = xsp[0], wa_n = wsp[0], wb_n = SW ? wsp[up_off] : 0.0f;
            for (int kb = 0; kb < KB; ++kb) {
                const float xs = xs_n, wsa = wa_n, wsb = wb_n;
                if (kb + 1 < KB) {
                    xs_n = xsp[kb + 1];
                    wa_n = wsp[kb + 1];
                    if (SW) wb_n = wsp[up_off + kb + 1];
                }
                const float fa = __fmul_rn(xs, wsa);
                const float fb = SW ? __fmul_rn(xs, wsb) : fa;
                const uint64_t pfa = pack2(__float_as_uint(fa), __float_as_uint(fa));
                const uint64_t pfb = pack2(__float_as_uint(fb), __float_as_uint(fb));
                if (!wait_bounded(smem_u32(&acc_full[ab]), aphase, abort_flag, args.status,
                                  MOE_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t accb = lane_base + (uint32_t)(ab * kTN);
                uint32_t v[16];
#pragma unroll
                for (int c = 0; c < 8; ++c) {   // 16 columns at a time
                    const uint32_t col =
                        SW ? (c < 4 ? wgp * 64 + c * 16 : 128 + wgp * 64 + (c - 4) * 16)
                           : wgp * 128 + c * 16;
                    tmem_ld16(accb + col, v);
                    tmem_wait_ld(v);
                    if (c == 7) {   // all of this K block is in registers: free the accumulator
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
                    }
                    const uint64_t f = c < 4 ? pfa : pfb;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[8 * c + j] = fma2(pack2(v[2 * j], v[2 * j + 1]), f, acc[8 * c + j]);
                }
                if (++ab == 2) {
                    ab = 0;
                    aphase ^= 1u;
                }
            }
            if (!ok) break;
            if constexpr (SW) {
                // h = silu(gate) * up for this thread's 64 features of its row;
                // the row's group maximum over all 128 features through shared memory
                float amax = 0.0f;
#pragma unroll
                for (int p = 0; p < 32; ++p) {
                    const float h0 = silu_mul(lo_f(acc[p]), lo_f(acc[32 + p]));
                    const float h1 = silu_mul(hi_f(acc[p]), hi_f(acc[32 + p]));
                    acc[p] = pack2(__float_as_uint(h0), __float_as_uint(h1));
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
                const float inv = fp8_group_inv(sc);
                if (valid) {
                    const int inter = args.n_out / 2;
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint64_t a0 = acc[2 * i], a1 = acc[2 * i + 1];
                        w[i] = (uint32_t)fp8_code(lo_f(a0), inv) |
                               ((uint32_t)fp8_code(hi_f(a0), inv) << 8) |
                               ((uint32_t)fp8_code(lo_f(a1), inv) << 16) |
                               ((uint32_t)fp8_code(hi_f(a1), inv) << 24);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(args.h + (size_t)(tl.row0 + m) * inter +
                                                           tl.nt * 128 + wgp * 64);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    if (wgp == 0) args.h_scales[(size_t)(tl.row0 + m) * NT + tl.nt] = sc;
                }
            } else {
                // fp32 C: columns [256 nt + 128 wgp, +128) of this warp's 32 rows
                const int vw = min(32, max(0, tl.nvalid - 32 * q));   // valid rows of the warp
                const int col0 = tl.nt * kTN + wgp * 128;
                if (vw == 32) {
                    // 32 x 32 blocks through 128-byte-swizzled shared memory and
                    // one TMA store each (the warp's two buffers alternate)
#pragma unroll
                    for (int j = 0; j < 4; ++j, ++nstore) {
                        const uint32_t buf = obuf + (uint32_t)(nstore & 1) * kOutBuf;
                        if (lane == 0) bulk_wait_group_read<1>();   // its last store has read it
                        __syncwarp();
#pragma unroll
                        for (int c = 0; c < 8; ++c) {   // 16-byte chunk c of this row
                            const uint64_t a0 = acc[16 * j + 2 * c], a1 = acc[16 * j + 2 * c + 1];
                            const uint32_t dst =
                                buf + (uint32_t)(lane * 128 + ((c ^ (lane & 7)) * 16));
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                                         "r"((uint32_t)a0), "r"((uint32_t)(a0 >> 32)),
                                         "r"((uint32_t)a1), "r"((uint32_t)(a1 >> 32))
                                         : "memory");
                        }
                        fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmC, buf, col0 + 32 * j, tl.row0 + 32 * q);
                            bulk_commit_group();
                        }
                    }
                } else if (lane < vw) {   // a ragged last tile: this thread's row directly
                    float4 *dst = reinterpret_cast<float4 *>(
                        args.c + (size_t)(tl.row0 + m) * args.n_out + col0);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        dst[i] = make_float4(lo_f(acc[2 * i]), hi_f(acc[2 * i]),
                                             lo_f(acc[2 * i + 1]), hi_f(acc[2 * i + 1]));
                }
            }
        }
        if (!SW && lane == 0) bulk_wait_group_all();   // every store has landed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <bool SW, bool GATHER, int ST>
int launch_wide(const WideArgs &args_in, const void *a, const void *w, cudaStream_t s) {
    WideArgs args = args_in;
    args.w = static_cast<const uint8_t *>(w);
    using Sh = WideShape<SW, ST>;
    auto kern = wide_gemm_kernel<SW, GATHER, ST>;
    static std::once_flag attr_once[64];
    static int attr_rc[64];
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return cuda_fail("device ordinal beyond 63");
    std::call_once(attr_once[dev], [&] {
        attr_rc[dev] = (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Sh::kSmemBytes);
    });
    if (attr_rc[dev]) return cuda_fail("cudaFuncSetAttribute", (cudaError_t)attr_rc[dev]);
    const int KB = args.k_dim / 128;
    CUtensorMap tmW, tmA, tmC;
    const bool tmw_ok =
        args.w_tiled
            ? encode_2d(&tmW, w, true, 128, (uint64_t)args.groups * args.n_out * KB, 128)
            : encode_2d(&tmW, w, true, (uint64_t)args.k_dim, (uint64_t)args.groups * args.n_out,
                        128);
    if (!tmw_ok) return cuda_fail("cuTensorMapEncodeTiled (weights)");
    // activations: the dispatched rows in boxes of 32, or (gather) the token
    // rows of x, one row per box as gather4 requires
    if (!(GATHER ? encode_2d(&tmA, a, true, (uint64_t)args.k_dim, (uint64_t)args.T, 1)
                 : encode_2d(&tmA, a, true, (uint64_t)args.k_dim, (uint64_t)args.rows, kABox)))
        return cuda_fail("cuTensorMapEncodeTiled (activations)");
    if (SW) {
        tmC = tmA;   // unused by the SwiGLU epilogue
    } else if (!encode_2d_f32(&tmC, args.c, (uint64_t)args.n_out, (uint64_t)args.rows, 32)) {
        return cuda_fail("cuTensorMapEncodeTiled (output)");
    }
    const int64_t tiles_bound =
        (int64_t)(args.n_out / kTN) * (args.groups + ceil_div(args.rows, kTM));
    const int grid = (int)std::min<int64_t>((int64_t)sm_count(), tiles_bound);
    if (grid <= 0) return MOE_OK;
    if (launch_dependent(kern, dim3(grid), dim3(kThreads), Sh::kSmemBytes, s, tmW, tmA, tmC, args))
        return MOE_ERR_CUDA;
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

WideArgs wide_args(int groups, int n_out, int k_dim, int rows, const float *a_scales,
                   const int32_t *offsets, const float *w_scales, bool w_tiled, int32_t *status) {
    WideArgs args;
    args.w = nullptr;
    args.groups = groups;
    args.n_out = n_out;
    args.k_dim = k_dim;
    args.rows = rows;
    args.offsets = offsets;
    args.a_scales = a_scales;
    args.w_scales = w_scales;
    args.h = nullptr;
    args.h_scales = nullptr;
    args.c = nullptr;
    args.w_tiled = w_tiled;
    args.src_of_row = nullptr;
    args.x_scales = nullptr;
    args.T = 0;
    args.k = 0;
    args.min_rows = 0;
    args.max_rows = 0x7fffffff;
    args.status = status;
    return args;
}

}  // namespace

int launch_swiglu_wide(int groups, int inter, int k_dim, int rows, const void *a,
                       const float *a_scales, const int32_t *offsets, const void *w13,
                       const float *w13_scales, bool w_tiled, void *h, float *h_scales,
                       int32_t *status, cudaStream_t s, int min_rows, int max_rows) {
    if (rows == 0) return MOE_OK;
    WideArgs args = wide_args(groups, 2 * inter, k_dim, rows, a_scales, offsets, w13_scales,
                              w_tiled, status);
    args.min_rows = min_rows;
    args.max_rows = max_rows;
    args.h = static_cast<uint8_t *>(h);
    args.h_scales = h_scales;
    // Ring depth by the batch's rows per group (same bits either way).  Past
    // 128 rows a group takes a second token tile that reads the same weights;
    // with three stages instead of four the 4096-token layer's gate/up launch
    // took 1.665 ms instead of 1.727 ms, while the 1024-token Zipf layer's
    // (groups mostly of 33-128 rows) took 0.336 instead of 0.325 ms.
    if ((int64_t)rows > (int64_t)kTM * groups) return launch_wide<true, false, 3>(args, a, w13, s);
    return launch_wide<true, false, 4>(args, a, w13, s);
}

int launch_swiglu_wide_gather(int groups, int inter, int k_dim, int rows, const void *xq,
                              const float *xs, int T, int top_k, const int32_t *src_of_row,
                              const int32_t *offsets, const void *w13, const float *w13_scales,
                              bool w_tiled, void *h, float *h_scales, int32_t *status,
                              cudaStream_t s, int min_rows, int max_rows) {
    if (rows == 0 || T == 0) return MOE_OK;
    WideArgs args = wide_args(groups, 2 * inter, k_dim, rows, nullptr, offsets, w13_scales,
                              w_tiled, status);
    args.h = static_cast<uint8_t *>(h);
    args.h_scales = h_scales;
    args.src_of_row = src_of_row;
    args.x_scales = xs;
    args.T = T;
    args.k = top_k;
    args.min_rows = min_rows;
    args.max_rows = max_rows;
    return launch_wide<true, true, 4>(args, xq, w13, s);
}

int launch_gemm_wide(int groups, int n_out, int k_dim, int rows, const void *a,
                     const float *a_scales, const int32_t *offsets, const void *w,
                     const float *w_scales, bool w_tiled, float *c, int32_t *status,
                     cudaStream_t s, int min_rows, int max_rows) {
    if (rows == 0) return MOE_OK;
    WideArgs args =
        wide_args(groups, n_out, k_dim, rows, a_scales, offsets, w_scales, w_tiled, status);
    args.min_rows = min_rows;
    args.max_rows = max_rows;
    args.c = c;
    return launch_wide<false, false, 3>(args, a, w, s);
}

}  // namespace moe

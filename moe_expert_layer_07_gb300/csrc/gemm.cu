// Grouped GEMM over per-expert row blocks on the 5th-generation tensor cores.
//
//   C[r, n] = sum_k A[r, k] W[g, n, k]   for rows r of group g
//
// Weight rows are the MMA's M side (128 per tile) and the few token rows of
// an expert its N side (16..BN per tile, BN = 32 for decode-sized groups and
// 64 for groups averaging 16 rows or more), so that a decode-sized expert
// with a handful of rows still streams its weights at full tile efficiency.
// The SGLang/H20 article (section "SwapAB GEMM") makes the same swap on
// Hopper, where WGMMA fixes M = 64; tcgen05 with M = 128 and N a multiple of
// 16 is the analogue here.
//
// Persistent CTAs, two per SM, 2 + 4 EW warps each:
//   warp 0      TMA producer: per K-block a 128 x 128-byte weight box (from
//               row-major weights, or one contiguous 16 KB tile of packed
//               weights) and ceil(rows/16) 16 x 128-byte activation boxes
//               (wide FP8 tiles: one 64-row box), 128-byte swizzled, into a
//               STAGES-deep shared-memory ring.
//   warp 1      MMA issuer (one thread): tcgen05.mma, K = 32 bytes per
//               instruction, accumulators in tensor memory, completion
//               signalled with tcgen05.commit.
//   warps 2..   epilogue (EW warpgroups; warp 2 + 4h + j reads TMEM lane
//               quarter j of the h-th BN/EW columns; thread = weight row):
//               tcgen05.ld of the accumulator, then
//                 FP8: per 128-wide K block, the block's partial product is
//                 scaled by w_scale[g, m/128, kb] * a_scale[r, kb] and added
//                 to fp32 registers (paired FMAs); four TMEM buffers rotate
//                 so the MMAs of the next blocks run meanwhile, and the
//                 tile's scales are copied to shared memory one tile ahead
//                 (cp.async, completion on an mbarrier), turned into the
//                 tile's promotion factors once (the SwiGLU instance makes
//                 its gate and up factors per K block), and read back as
//                 16-byte broadcasts;
//                 BF16: one accumulation over all of K (the four TMEM
//                 buffers rotate between tiles);
//               and stores C (coalesced: a warp writes 32 consecutive n).
// Work units are (group, 128-row weight tile, BN-row activation tile); the
// tile table is built on the device from expert_offsets, so no host sync is
// needed and the launch can be captured in a graph.  Every wait is bounded:
// after about a second the CTA records MOE_DEV_TIMEOUT, drains its copies
// and MMAs, frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "numerics.cuh"
#include "ptx.cuh"
#include "tma_host.h"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kMaxGroups = 1024;
// Two CTAs share each SM: each CTA's MMA work does not overlap its own weight
// stream, and a second CTA fills those gaps (measured on the R1 decode layer:
// 5.5 -> 6.8 TB/s for the gate/up GEMM).
constexpr int kCtasPerSm = 2;
constexpr int kBoxRows = 16;   // activation rows per TMA box
constexpr int kMaxKBlocks = 56; // FP8: K <= 7168

// SW (SwiGLU epilogue): a tile covers 128 gate rows and the matching 128 up
// rows of W13 (two A tiles per stage sharing one activation tile) and writes
// h = silu(gate) * up instead of C.
// EW: epilogue warpgroups.  Warp 2 + 4h + j (h < EW) reads TMEM lanes
// [32 (warp & 3), +32) of columns [h BN/EW, (h + 1) BN/EW), so two groups give
// each SM sub-partition twice the warps to hide the promotion's latencies.
template <bool FP8, int BN, int STAGES, bool SW, int EW = 1>
struct GemmShape {
    static constexpr int kEpiThreads = 128 * EW;
    static constexpr int kThreads = 64 + kEpiThreads;    // producer, MMA, epilogue warps
    static constexpr int kCB = BN / EW;                  // columns per epilogue warp
    static_assert(EW == 1 || (FP8 && !SW && kCB % 16 == 0), "EW");
    static constexpr int kNA = SW ? 2 : 1;               // weight tiles per stage
    static constexpr int kABytes = kBM * 128;            // one weight tile
    static constexpr int kBBytes = BN * 128;
    static constexpr int kStageBytes = kNA * kABytes + kBBytes;
    static constexpr int kSmemBytes = STAGES * kStageBytes + 1024;
    static constexpr int kAccBufs = 4;                   // TMEM accumulators in flight
    static constexpr int kAccCols = kNA * BN;
    static constexpr int kTmemCols = kAccBufs * kAccCols;
    static constexpr int kKPerStage = FP8 ? 128 : 64;   // elements of K per stage
    static constexpr int kXsElems = FP8 ? BN * kMaxKBlocks : 1;
    static constexpr int kWsElems = FP8 ? kNA * kMaxKBlocks : 1;
    static constexpr int kAmaxElems = (SW && FP8) ? 4 * BN : 1;
    // activation rows per TMA box: the wide FP8 tiles load all BN rows with
    // one box (a TMA instruction less in the producer's loop per 16 rows);
    // the others ceil(rows / 16) boxes of 16
    static constexpr int kABox = (FP8 && !SW && EW > 1) ? BN : kBoxRows;
    static_assert(BN % 16 == 0 && BN >= 32 && BN <= 64, "BN");
    static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols * kCtasPerSm <= 512,
                  "TMEM columns");
    static constexpr int kSxElems = (FP8 && SW) ? 4 * EW * 2 * kNA * kCB : 1;   // per warp, per K-block parity
    static_assert((kSmemBytes + 8 * kXsElems + 8 * kWsElems + 8 * kAmaxElems + 4 * kSxElems +
                   8 * 1024 + 1024) *
                          kCtasPerSm <=
                      228 * 1024,
                  "shared memory");
};

struct GemmArgs {
    int groups, n_out, k_dim, rows;
    const int32_t *offsets;
    const float *a_scales;
    const float *w_scales;
    void *c;          // C [rows, n_out]; SwiGLU: h [rows, n_out/2] (e4m3 or bf16)
    float *h_scales;  // SwiGLU + FP8: [rows, n_out/256]
    int c_bf16;
    int w_tiled;      // W in MOE_LAYOUT_TILES (tiles read by 16 KB bulk copies)
    const uint8_t *w; // W bytes
    int min_rows, max_rows;   // groups whose row count lies outside are skipped
    int32_t *status;
};

struct Tile {
    int g, mt, row0, nvalid;
};

template <int BN>
__device__ __forceinline__ Tile decode_tile(int t, int G, const int *s_tiles, const int *s_off) {
    int lo = 0, hi = G;   // s_tiles[lo] <= t < s_tiles[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tiles[mid] <= t) lo = mid;
        else hi = mid;
    }
    Tile tl;
    tl.g = lo;
    const int rows = s_off[lo + 1] - s_off[lo];
    const int ntn = (rows + BN - 1) / BN;
    const int local = t - s_tiles[lo];
    tl.mt = local / ntn;
    const int nt = local - tl.mt * ntn;
    tl.row0 = s_off[lo] + nt * BN;
    tl.nvalid = min(BN, rows - nt * BN);
    return tl;
}

template <bool FP8, int BN, int STAGES, bool SW, int EW>
__global__ void __launch_bounds__(64 + 128 * EW, kCtasPerSm)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmA, const GemmArgs args) {
    using S = GemmShape<FP8, BN, STAGES, SW, EW>;
    constexpr int CB = S::kCB;
    constexpr int NB = S::kAccBufs;
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t acc_full[NB];
    __shared__ __align__(8) uint64_t acc_empty[NB];
    __shared__ __align__(8) uint64_t scale_full[2];
    __shared__ __align__(8) uint64_t scale_empty[2];
    __shared__ __align__(8) uint64_t amax_bar[2];
    __shared__ __align__(8) uint64_t fac_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_abort, s_bad;
    __shared__ int s_off[kMaxGroups + 1];
    __shared__ int s_tiles[kMaxGroups + 1];
    // FP8 scales of the tile being reduced (and of the next one): per K block
    // the weight-block scale, and the activation scale of every row n laid
    // out [kb][n] so that lanes read consecutive words.
    __shared__ float s_ws[2][S::kWsElems];
    __shared__ __align__(16) float s_xs[2][S::kXsElems];
    // SwiGLU + FP8: per tile, each epilogue warp's |h| maximum of every row n
    __shared__ float s_amax[2][S::kAmaxElems];
    // FP8: per epilogue warp, the K block's promotion factor of every column
    // n, x_scale[n, kb] * w_scale[kb] (gate, then up), read back as 16-byte
    // broadcasts instead of a shuffle per column
    __shared__ __align__(16) float s_sx[S::kSxElems];

    using namespace ptx;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem_base = (smem_u32(dsmem) + 1023u) & ~1023u;
    const int G = args.groups;
    const int MTW = args.n_out / kBM;            // 128-row blocks of W per group
    const int MT = SW ? MTW / 2 : MTW;           // weight tiles per group
    const int KB = args.k_dim / S::kKPerStage;
    volatile int *abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 4 * EW);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&scale_full[b]), S::kEpiThreads);   // every epilogue thread's copies
            mbar_init(smem_u32(&scale_empty[b]), 4 * EW);          // every epilogue warp done reading
            mbar_init(smem_u32(&amax_bar[b]), 4);       // every epilogue warp's row maxima
            mbar_init(smem_u32(&fac_bar[b]), 4 * EW);   // every epilogue warp's share of factors
        }
        mbar_init(smem_u32(&drain_bar), 1);
        s_abort = 0;
        s_bad = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_slot), S::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmA);
    }
    pdl_wait();   // the set-up above overlaps the previous kernel's tail
    for (int i = threadIdx.x; i <= G; i += S::kThreads) s_off[i] = args.offsets[i];
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += S::kThreads) {
        const int a = s_off[g], b = s_off[g + 1];
        if (a < 0 || b < a || b > args.rows) s_bad = 1;
    }
    __syncthreads();
    // token tiles of group g; none for groups outside the row window
    auto ntiles_of = [&](int g) {
        const int n = s_off[g + 1] - s_off[g];
        return (n < args.min_rows || n > args.max_rows) ? 0 : (n + BN - 1) / BN;
    };
    if (warp == 0) {   // tile prefix over groups: lane L owns a contiguous run
        const int per = (G + 31) / 32;
        const int g0 = lane * per;
        int local = 0;
        for (int q = 0; q < per; ++q) {
            const int g = g0 + q;
            if (g < G) local += MT * ntiles_of(g);
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
                run += MT * ntiles_of(g);
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
            // A weight tile is read once unless its group spans several N
            // tiles: those run on neighbouring CTAs at about the same time and
            // share the L2 copy.  Activation rows are re-read by every weight
            // tile of their group.
            const uint64_t pol_w_once = policy_evict_first();
            const uint64_t pol_w_shared = policy_evict_normal();
            const uint64_t pol_a = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0, issued = 0, parity_bits = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile<BN>(t, G, s_tiles, s_off);
                const int nbox = (tl.nvalid + S::kABox - 1) / S::kABox;
                const uint32_t bytes = S::kNA * S::kABytes + nbox * S::kABox * 128;
                const int wrow = tl.g * args.n_out + tl.mt * kBM;   // SwiGLU: gate rows
                const int wrow_up = wrow + args.n_out / 2;          // SwiGLU: up rows
                // tiled W: the box of (128-row block b, K block kb) is rows
                // (b * KB + kb) * 128 of a [tiles * 128, 128-byte] view
                const int tb = (tl.g * MTW + tl.mt) * KB;
                const int tb_up = tb + (MTW / 2) * KB;
                const uint64_t pol_w =
                    (s_off[tl.g + 1] - s_off[tl.g] > BN) ? pol_w_shared : pol_w_once;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag,
                                      args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_base + stage * S::kStageBytes;
                    const uint32_t sb = sa + S::kNA * S::kABytes;
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    if (args.w_tiled) {   // pre-swizzled 16 KB tiles: plain bulk copies
                        bulk_load(sa, args.w + (size_t)(tb + kb) * S::kABytes, S::kABytes, fb,
                                  pol_w);
                        if (SW)
                            bulk_load(sa + S::kABytes, args.w + (size_t)(tb_up + kb) * S::kABytes,
                                      S::kABytes, fb, pol_w);
                    } else {
                        tma_load_2d(sa, &tmW, kb * S::kKPerStage, wrow, fb, pol_w);
                        if (SW)
                            tma_load_2d(sa + S::kABytes, &tmW, kb * S::kKPerStage, wrow_up, fb,
                                        pol_w);
                    }
                    for (int b = 0; b < nbox; ++b)
                        tma_load_2d(sb + b * S::kABox * 128, &tmA, kb * S::kKPerStage,
                                    tl.row0 + b * S::kABox, fb, pol_a);
                    issued |= 1u << stage;
                    parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {   // let every copy in flight land before the CTA exits
                for (int s = 0; s < STAGES; ++s)
                    if ((issued >> s) & 1u)
                        wait_drain(smem_u32(&full_bar[s]), (parity_bits >> s) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, ab = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
                const Tile tl = decode_tile<BN>(t, G, s_tiles, s_off);
                const int nmma = ((tl.nvalid + 15) / 16) * 16;
                const uint32_t idesc = FP8 ? idesc_e4m3(kBM, nmma) : idesc_bf16(kBM, nmma);
                for (int kb = 0; kb < KB; ++kb) {
                    if (FP8 || kb == 0) {   // FP8: one accumulator per K block
                        if (!wait_bounded(smem_u32(&acc_empty[ab]), aphase ^ 1u, abort_flag,
                                          args.status, MOE_DEV_TIMEOUT)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (!wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag,
                                      args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_base + stage * S::kStageBytes;
                    const uint64_t da = sdesc_k_sw128(sa);
                    const uint64_t da_up = sdesc_k_sw128(sa + S::kABytes);
                    const uint64_t db = sdesc_k_sw128(sa + S::kNA * S::kABytes);
                    const uint32_t d = tmem_base + (uint32_t)(ab * S::kAccCols);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {   // 4 x 32 bytes of K
                        const uint32_t acc = FP8 ? (kk > 0) : (kb > 0 || kk > 0);
                        if (FP8) mma_f8f6f4(d, da + 2 * kk, db + 2 * kk, idesc, acc);
                        else mma_f16(d, da + 2 * kk, db + 2 * kk, idesc, acc);
                        if (SW) {   // up rows into the next BN columns
                            if (FP8) mma_f8f6f4(d + BN, da_up + 2 * kk, db + 2 * kk, idesc, acc);
                            else mma_f16(d + BN, da_up + 2 * kk, db + 2 * kk, idesc, acc);
                        }
                    }
                    mma_commit(smem_u32(&empty_bar[stage]));
                    if (FP8 || kb == KB - 1) {
                        mma_commit(smem_u32(&acc_full[ab]));
                        if (++ab == NB) {
                            ab = 0;
                            aphase ^= 1u;
                        }
                    }
                    if (++stage == STAGES) {
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
        // ------------------------------ epilogue (warps 2 .. 1 + 4 EW)
        const int q = warp & 3;                    // TMEM lanes [32q, 32q + 32)
        const int ew = warp - 2;                   // epilogue warp 0 .. 4 EW - 1
        const int n0 = (ew >> 2) * CB;             // first of this warp's CB columns
        const int etid = threadIdx.x - 64;         // 0 .. 128 EW - 1
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
        const int m_local = q * 32 + lane;
        const int n_h = args.n_out / 2;            // SwiGLU: width of h
        int ab = 0;
        uint32_t aphase = 0;
        bool ok = true;

        // FP8: copy the scales of tile t into buffer b (asynchronously); the
        // buffer's scale_full barrier completes when all 128 threads' copies land.
        auto stage_scales = [&](int t, int b) {
            const Tile tl = decode_tile<BN>(t, G, s_tiles, s_off);
            const float *wsp = args.w_scales + ((size_t)tl.g * MTW + tl.mt) * KB;
            const float *xsp = args.a_scales + (size_t)tl.row0 * KB;
            for (int i = etid; i < KB; i += S::kEpiThreads) cp_async4(smem_u32(&s_ws[b][i]), wsp + i);
            if (SW) {   // up rows' block scales
                const float *wup = wsp + (size_t)(MTW / 2) * KB;
                for (int i = etid; i < KB; i += S::kEpiThreads)
                    cp_async4(smem_u32(&s_ws[b][KB + i]), wup + i);
            }
            const int n_el = tl.nvalid * KB;
            for (int i = etid; i < n_el; i += S::kEpiThreads) {
                const int n = i / KB, kb = i - n * KB;
                cp_async4(smem_u32(&s_xs[b][kb * BN + n]), xsp + i);
            }
            cp_async_mbar_arrive(smem_u32(&scale_full[b]));
        };
        if (FP8 && (int)blockIdx.x < total_tiles) stage_scales(blockIdx.x, 0);

        int it = 0;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++it) {
            const Tile tl = decode_tile<BN>(t, G, s_tiles, s_off);
            const int nchunks = (tl.nvalid + 15) / 16;
            const int m_glob = tl.mt * kBM + m_local;
            if (FP8) {
                // tile iteration `it` reads buffer it&1 (its (it>>1)-th use);
                // the next tile's scales go to the other buffer, whose previous
                // use (iteration it-1) must have been released first
                const int b = it & 1;
                const int tn = t + (int)gridDim.x;
                if (tn < total_tiles) {
                    const uint32_t use = (uint32_t)(it + 1) >> 1;
                    if (!wait_bounded(smem_u32(&scale_empty[b ^ 1]), (use & 1u) ^ 1u, abort_flag,
                                      args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    stage_scales(tn, b ^ 1);
                }
                if (!wait_bounded(smem_u32(&scale_full[b]), ((uint32_t)it >> 1) & 1u, abort_flag,
                                  args.status, MOE_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                if constexpr (!SW) {
                    // promotion factors of the whole tile, in place, once:
                    // s_xs[b][kb BN + n] = x_scale[n, kb] * w_scale[kb] (0 past
                    // the tile's rows); the K loop then reads them directly
                    float *xs = s_xs[b];
                    for (int i = etid; i < KB * BN; i += S::kEpiThreads) {
                        const int kb = i / BN, n = i - kb * BN;
                        xs[i] = n < tl.nvalid ? __fmul_rn(xs[i], s_ws[b][kb]) : 0.0f;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&fac_bar[b]));
                    if (!wait_bounded(smem_u32(&fac_bar[b]), ((uint32_t)it >> 1) & 1u, abort_flag,
                                      args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                }
                // columns n0 + 2p, n0 + 2p + 1 side by side for the paired FMA
                uint64_t acc2[CB / 2];
                float accu[SW ? BN : 1];
#pragma unroll
                for (int p = 0; p < CB / 2; ++p) acc2[p] = 0ull;
#pragma unroll
                for (int n = 0; n < (SW ? BN : 1); ++n) accu[n] = 0.0f;
                for (int kb = 0; kb < KB; ++kb) {
                    // factors of this warp's columns n0 + j: SwiGLU at sxw[j] (gate) and
                    // sxw[CB + j] (up), made per K block; otherwise the tile's own
                    const float *sxw = s_xs[b] + kb * BN + n0;
                    if constexpr (SW) {
                        const float sw = s_ws[b][kb];
                        const float swu = s_ws[b][KB + kb];
                        float *sx = s_sx + (ew * 2 + (kb & 1)) * (S::kNA * CB);
#pragma unroll
                        for (int h = 0; h < (CB + 31) / 32; ++h) {
                            const int j = h * 32 + lane, n = n0 + j;
                            if (j < CB) {
                                const float xv = n < tl.nvalid ? s_xs[b][kb * BN + n] : 0.0f;
                                sx[j] = __fmul_rn(xv, sw);
                                sx[CB + j] = __fmul_rn(xv, swu);
                            }
                        }
                        __syncwarp();
                        sxw = sx;
                    }
                    if (!wait_bounded(smem_u32(&acc_full[ab]), aphase, abort_flag, args.status,
                                      MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t col = (uint32_t)(ab * S::kAccCols);
                    const int nch = nchunks - n0 / 16;   // this warp's valid 16-column chunks
                    uint32_t v[CB / 16][16];
#pragma unroll
                    for (int c = 0; c < CB / 16; ++c)
                        if (c < nch) tmem_ld16(lane_base + col + (uint32_t)(n0 + c * 16), v[c]);
#pragma unroll
                    for (int c = 0; c < CB / 16; ++c)
                        if (c < nch) tmem_wait_ld(v[c]);
#pragma unroll
                    for (int c = 0; c < CB / 16; ++c)
                        if (c < nch) {
#pragma unroll
                            for (int j4 = 0; j4 < 4; ++j4) {
                                const uint4 f = reinterpret_cast<const uint4 *>(sxw)[c * 4 + j4];
                                const int p = (c * 16 + j4 * 4) / 2;
                                acc2[p] = fma2(pack2(v[c][j4 * 4], v[c][j4 * 4 + 1]), pack2(f.x, f.y),
                                               acc2[p]);
                                acc2[p + 1] = fma2(pack2(v[c][j4 * 4 + 2], v[c][j4 * 4 + 3]),
                                                   pack2(f.z, f.w), acc2[p + 1]);
                            }
                        }
                    if constexpr (SW) {   // up rows: same activation scales, their own block scale
#pragma unroll
                        for (int c = 0; c < BN / 16; ++c)
                            if (c < nchunks)
                                tmem_ld16(lane_base + col + (uint32_t)(BN + c * 16), v[c]);
#pragma unroll
                        for (int c = 0; c < BN / 16; ++c)
                            if (c < nchunks) tmem_wait_ld(v[c]);
#pragma unroll
                        for (int c = 0; c < BN / 16; ++c)
                            if (c < nchunks) {
#pragma unroll
                                for (int j4 = 0; j4 < 4; ++j4) {
                                    const float4 f =
                                        reinterpret_cast<const float4 *>(sxw + CB)[c * 4 + j4];
                                    const int n = c * 16 + j4 * 4;
                                    float *au = accu + (SW ? n : 0);
                                    au[0] = fmaf(__uint_as_float(v[c][j4 * 4]), f.x, au[0]);
                                    au[SW ? 1 : 0] = fmaf(__uint_as_float(v[c][j4 * 4 + 1]), f.y, au[SW ? 1 : 0]);
                                    au[SW ? 2 : 0] = fmaf(__uint_as_float(v[c][j4 * 4 + 2]), f.z, au[SW ? 2 : 0]);
                                    au[SW ? 3 : 0] = fmaf(__uint_as_float(v[c][j4 * 4 + 3]), f.w, au[SW ? 3 : 0]);
                                }
                            }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
                    if (++ab == NB) {
                        ab = 0;
                        aphase ^= 1u;
                    }
                }
                if (!ok) break;
                float acc[CB];   // columns n0 .. n0 + CB - 1
#pragma unroll
                for (int p = 0; p < CB / 2; ++p) {
                    acc[2 * p] = __uint_as_float((uint32_t)acc2[p]);
                    acc[2 * p + 1] = __uint_as_float((uint32_t)(acc2[p] >> 32));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&scale_empty[b]));
                if constexpr (SW) {
                    // h = silu(gate) * up; each row n is quantised over the
                    // tile's 128 features (one per thread): warp maxima, then
                    // the four warps' maxima through shared memory.
#pragma unroll
                    for (int n = 0; n < BN; ++n) acc[n] = silu_mul(acc[n], accu[SW ? n : 0]);
                    float mine = 0.0f;
#pragma unroll
                    for (int n = 0; n < BN; ++n) {
                        float m = fabsf(acc[n]);
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                        if ((n & 31) == lane) mine = m;
                        if ((n & 31) == 31 || n == BN - 1) {   // lanes hold rows [n & ~31, ...)
                            const int base = n & ~31;
                            if (lane <= n - base) s_amax[b][q * BN + base + lane] = mine;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&amax_bar[b]));
                    if (!wait_bounded(smem_u32(&amax_bar[b]), ((uint32_t)it >> 1) & 1u, abort_flag,
                                      args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    uint8_t *H8 = static_cast<uint8_t *>(args.c);
#pragma unroll
                    for (int n = 0; n < BN; ++n)
                        if (n < tl.nvalid) {
                            const float amax = fmaxf(fmaxf(s_amax[b][n], s_amax[b][BN + n]),
                                                     fmaxf(s_amax[b][2 * BN + n], s_amax[b][3 * BN + n]));
                            const float sc = fp8_group_scale(amax);
                            const size_t row = (size_t)(tl.row0 + n);
                            H8[row * n_h + tl.mt * kBM + m_local] =
                                fp8_code(acc[n], fp8_group_inv(sc));
                            if (m_local == 0) args.h_scales[row * (n_h / 128) + tl.mt] = sc;
                        }
                } else if (args.c_bf16) {
                    __nv_bfloat16 *C = static_cast<__nv_bfloat16 *>(args.c);
#pragma unroll
                    for (int n = 0; n < CB; ++n)
                        if (n0 + n < tl.nvalid)
                            C[(size_t)(tl.row0 + n0 + n) * args.n_out + m_glob] =
                                __float2bfloat16_rn(acc[n]);
                } else {
                    float *C = static_cast<float *>(args.c);
#pragma unroll
                    for (int n = 0; n < CB; ++n)
                        if (n0 + n < tl.nvalid)
                            C[(size_t)(tl.row0 + n0 + n) * args.n_out + m_glob] = acc[n];
                }
            } else {
                if (!wait_bounded(smem_u32(&acc_full[ab]), aphase, abort_flag, args.status,
                                  MOE_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col = (uint32_t)(ab * S::kAccCols);
#pragma unroll
                for (int c = 0; c < BN / 16; ++c)
                    if (c < nchunks) {
                        uint32_t v[16], vu[16];
                        tmem_ld16(lane_base + col + (uint32_t)(c * 16), v);
                        tmem_wait_ld(v);
                        if (SW) {
                            tmem_ld16(lane_base + col + (uint32_t)(BN + c * 16), vu);
                            tmem_wait_ld(vu);
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int n = c * 16 + j;
                            if (n < tl.nvalid) {
                                if (SW) {
                                    const size_t idx = (size_t)(tl.row0 + n) * n_h + tl.mt * kBM + m_local;
                                    static_cast<__nv_bfloat16 *>(args.c)[idx] = __float2bfloat16_rn(
                                        silu_mul(__uint_as_float(v[j]), __uint_as_float(vu[j])));
                                } else {
                                    const size_t idx = (size_t)(tl.row0 + n) * args.n_out + m_glob;
                                    if (args.c_bf16)
                                        static_cast<__nv_bfloat16 *>(args.c)[idx] =
                                            __float2bfloat16_rn(__uint_as_float(v[j]));
                                    else
                                        static_cast<float *>(args.c)[idx] = __uint_as_float(v[j]);
                                }
                            }
                        }
                    }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
                if (++ab == NB) {
                    ab = 0;
                    aphase ^= 1u;
                }
            }
        }
        if (FP8) asm volatile("cp.async.wait_all;" ::: "memory");   // copies land before exit
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, S::kTmemCols);
    }
}

}  // namespace

// ---- host side ---------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Encoded descriptors, kept by everything they depend on (address, element
// type, extents, box rows): a layer calls with the same buffers every step,
// and the encoder costs about as much host time as a kernel launch.
// Direct-mapped; a colliding key replaces the entry.
namespace {
enum TmType : uint32_t { kTmU8 = 1, kTmBf16 = 2, kTmF32 = 4 };
struct TmKey {
    uint64_t base, inner, outer;
    uint32_t box_rows, type;
    bool operator==(const TmKey &o) const {
        return base == o.base && inner == o.inner && outer == o.outer &&
               box_rows == o.box_rows && type == o.type;
    }
};
struct TmEntry {
    TmKey key;
    CUtensorMap map;
    bool valid;
};
constexpr int kTmCacheSize = 256;
TmEntry g_tm_cache[kTmCacheSize];
std::mutex g_tm_mutex;

size_t tm_slot(const TmKey &k) {
    uint64_t h = k.base >> 4;
    h = h * 0x9E3779B97F4A7C15ull ^ k.inner;
    h = h * 0x9E3779B97F4A7C15ull ^ k.outer;
    h = h * 0x9E3779B97F4A7C15ull ^ ((uint64_t)k.box_rows << 8 | k.type);
    return (size_t)((h * 0x9E3779B97F4A7C15ull) >> 56) % kTmCacheSize;
}

// Row-major [outer, inner] matrix of elements of `type`, box of 128 bytes x
// box_rows, 128-byte swizzle.
bool encode_rows(CUtensorMap *m, const void *base, TmType type, uint64_t inner, uint64_t outer,
                 uint32_t box_rows) {
    const TmKey key{reinterpret_cast<uint64_t>(base), inner, outer, box_rows, (uint32_t)type};
    const size_t slot = tm_slot(key);
    {
        std::lock_guard<std::mutex> lock(g_tm_mutex);
        if (g_tm_cache[slot].valid && g_tm_cache[slot].key == key) {
            *m = g_tm_cache[slot].map;
            return true;
        }
    }
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const uint32_t esize = (uint32_t)type;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * esize};
    cuuint32_t box[2] = {128 / esize, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = type == kTmU8     ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : type == kTmBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lock(g_tm_mutex);
    g_tm_cache[slot].key = key;
    g_tm_cache[slot].map = *m;
    g_tm_cache[slot].valid = true;
    return true;
}
}  // namespace

// Row-major [outer, inner] matrix, box of 128 bytes x box_rows, 128-byte swizzle.
bool encode_2d(CUtensorMap *m, const void *base, bool fp8, uint64_t inner, uint64_t outer,
               uint32_t box_rows) {
    return encode_rows(m, base, fp8 ? kTmU8 : kTmBf16, inner, outer, box_rows);
}

// Row-major fp32 [outer, inner] matrix, box of 32 columns (128 bytes) x
// box_rows, 128-byte swizzle (for TMA stores of fp32 tiles).
bool encode_2d_f32(CUtensorMap *m, void *base, uint64_t inner, uint64_t outer, uint32_t box_rows) {
    return encode_rows(m, base, kTmF32, inner, outer, box_rows);
}

namespace {

template <bool FP8, int BN, int STAGES, bool SW = false, int EW = 1>
int launch_impl(const GemmArgs &args, const void *a, const void *w, cudaStream_t s) {
    using Sh = GemmShape<FP8, BN, STAGES, SW, EW>;
    auto kern = grouped_gemm_kernel<FP8, BN, STAGES, SW, EW>;
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
    CUtensorMap tmW, tmA;
    const bool tmw_ok =
        args.w_tiled
            ? encode_2d(&tmW, w, FP8, (uint64_t)Sh::kKPerStage,
                        (uint64_t)args.groups * args.n_out * (args.k_dim / Sh::kKPerStage), kBM)
            : encode_2d(&tmW, w, FP8, (uint64_t)args.k_dim, (uint64_t)args.groups * args.n_out, kBM);
    if (!tmw_ok) return cuda_fail("cuTensorMapEncodeTiled (weights)");
    if (!encode_2d(&tmA, a, FP8, (uint64_t)args.k_dim, (uint64_t)args.rows, Sh::kABox))
        return cuda_fail("cuTensorMapEncodeTiled (activations)");
    const int64_t tiles_bound =
        (int64_t)(args.n_out / kBM / (SW ? 2 : 1)) * (args.groups + ceil_div(args.rows, BN));
    const int grid = (int)std::min<int64_t>((int64_t)sm_count() * kCtasPerSm, tiles_bound);
    if (grid <= 0) return MOE_OK;
    if (launch_dependent(kern, dim3(grid), dim3(Sh::kThreads), Sh::kSmemBytes, s, tmW, tmA, args))
        return MOE_ERR_CUDA;
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

}  // namespace

int launch_grouped_gemm(bool fp8, int groups, int n_out, int k_dim, int rows, const void *a,
                        const float *a_scales, const int32_t *offsets, const void *w,
                        const float *w_scales, bool w_tiled, void *c, int c_dtype,
                        int32_t *status, cudaStream_t s, int min_rows, int max_rows) {
    if (rows == 0) return MOE_OK;
    GemmArgs args;
    args.groups = groups;
    args.n_out = n_out;
    args.k_dim = k_dim;
    args.rows = rows;
    args.offsets = offsets;
    args.a_scales = a_scales;
    args.w_scales = w_scales;
    args.c = c;
    args.h_scales = nullptr;
    args.c_bf16 = c_dtype == MOE_OUT_BF16;
    args.w_tiled = w_tiled;
    args.w = static_cast<const uint8_t *>(w);
    args.min_rows = min_rows;
    args.max_rows = max_rows;
    args.status = status;
    // Decode-sized groups (a few rows each) stream best with 32-row tiles;
    // larger groups take 128 token rows against 256 output columns per tile
    // (gemm_wide.cu: one weight-tile read per 128 rows of an expert), or,
    // for bf16 C or widths that are not a multiple of 256, 64-row tiles.
    const bool wide = (int64_t)rows >= 16 * (int64_t)groups;
    if (fp8 && wide && n_out % 256 == 0 && c_dtype == MOE_OUT_F32)
        return launch_gemm_wide(groups, n_out, k_dim, rows, a, a_scales, offsets, w, w_scales,
                                w_tiled, static_cast<float *>(c), status, s, min_rows, max_rows);
    if (fp8) return wide ? launch_impl<true, 64, 3, false, 2>(args, a, w, s)
                         : launch_impl<true, 32, 4>(args, a, w, s);
    return launch_impl<false, 32, 4>(args, a, w, s);
}

int launch_grouped_gemm_swiglu(bool fp8, int groups, int inter, int k_dim, int rows,
                               const void *a, const float *a_scales, const int32_t *offsets,
                               const void *w13, const float *w13_scales, bool w_tiled, void *h,
                               float *h_scales, int32_t *status, cudaStream_t s, int min_rows,
                               int max_rows) {
    if (rows == 0) return MOE_OK;
    GemmArgs args;
    args.groups = groups;
    args.n_out = 2 * inter;
    args.k_dim = k_dim;
    args.rows = rows;
    args.offsets = offsets;
    args.a_scales = a_scales;
    args.w_scales = w13_scales;
    args.c = h;
    args.h_scales = h_scales;
    args.c_bf16 = !fp8;
    args.w_tiled = w_tiled;
    args.w = static_cast<const uint8_t *>(w13);
    args.min_rows = min_rows;
    args.max_rows = max_rows;
    args.status = status;
    // Groups averaging 16 rows or more: token rows on the MMA's M side, the
    // gate and up rows of 128 features on N (gemm_wide.cu).
    if (fp8 && (int64_t)rows >= 16 * (int64_t)groups)
        return launch_swiglu_wide(groups, inter, k_dim, rows, a, a_scales, offsets, w13,
                                  w13_scales, w_tiled, h, h_scales, status, s, min_rows,
                                  max_rows);
    if (fp8) return launch_impl<true, 32, 2, true>(args, a, w13, s);
    return launch_impl<false, 32, 2, true>(args, a, w13, s);
}

}  // namespace moe

// The experts' FFN in one persistent kernel (FP8 and BF16 layers):
//
//   for every group g and its rows r:
//     g, u = Xp[r] W13[g]^T            (gate and up; FP8: 128x128 block scales)
//     h    = silu(g) * u  -> FP8: e4m3 + one fp32 scale per 128 features;
//                            BF16: rounded to bf16
//     Y[r] = h W2[g]^T                 (fp32)
//
// Moreh report "21K output tokens/s DeepSeek inference on MI300X with Expert
// Parallelism", section "Library optimisation": its fused MoE kernel runs an
// expert's FFN as one kernel.  Here one launch holds both grouped GEMMs.
// The work units are the gate/up tiles (128 gate + 128 up weight rows x 32
// activation rows, SwiGLU and requantisation in the epilogue, as in the
// stand-alone SwiGLU GEMM) followed by the down tiles (128 rows of W2 x the
// same 32 activation rows).  CTAs claim units from a global counter, so a
// CTA that runs out of gate/up work moves on to down tiles while others
// finish theirs: the last wave of large gate/up tiles no longer idles most
// of the GPU, and the two GEMMs need no launch boundary between them.
//
// A down tile of (group g, activation tile j) reads h rows that the gate/up
// tiles of (g, j) write.  Each finished gate/up tile adds one to a per-j
// counter (release, after a proxy fence); the producer of a down tile waits
// (bounded) until the counter reaches the number of gate/up tiles of j,
// then issues its TMA loads of h, and (FP8) the epilogue threads acquire the
// same count before they read h's scales.  Every gate/up unit is claimed
// before any down unit and a producer issues all loads of a unit before it
// claims the next, so a unit that is waited on is always in some running
// CTA's pipeline: no wait can be circular.
//
// Per CTA (two per SM; one for small BF16 layers), 10 warps:
//   warp 0     scheduler + TMA producer: a 2-deep ring of 40 KB stages (5-deep
//              with one CTA per SM); a
//              gate/up stage holds one 128-byte K block (gate box, up box,
//              activation rows), a down stage two K blocks (two W2 boxes,
//              two h boxes; one of each in the last stage when the count
//              is odd).  Weights are row-major or 128 x 128-byte tiles;
//              a unit's activation or h rows come as one box per K block
//              (16 rows, or 32 when more than 16 are valid).
//   warp 1     MMA issuer: tcgen05.mma (kind::f8f6f4 or kind::f16),
//              tcgen05.commit to mbarriers; four TMEM accumulators rotate,
//              FP8 one per K block, BF16 one per unit.
//   warps 2-9  epilogue: each warp reads one TMEM lane quarter (thread =
//              weight row) of 16 of the 32 activation columns:
//              FP8: per K block the partial product times
//              x_scale[r, kb] * w_scale[g, m/128, kb] is added to fp32
//              registers (paired FMAs; the factors reach the warp as
//              shared-memory broadcasts); BF16: the unit's sums once; then
//              gate/up: SiLU-mul and h (FP8: row maxima across the four
//              lane quarters, e4m3 codes and scales); down: Y rows (fp32).
// The activation scales are read straight from global memory one K block
// ahead (the tile's 32 rows x K/128 floats stay in L1), which frees the
// shared memory that a second stage-sized buffer would need.
//
// Every wait is bounded (about a second): on expiry the CTA records
// MOE_DEV_TIMEOUT, raises its abort flag so that its other warps stop,
// lets its copies and MMAs drain, frees its tensor memory and exits.
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

constexpr int kBM = 128;                // weight rows per tile (MMA M)
constexpr int kBN = 32;                 // activation rows per tile (MMA N)
constexpr int kBoxRows = 16;            // activation rows per TMA box
// Two CTAs per SM with two stages each.  BF16 launches whose gate/up units
// all fit in one wave of one CTA per SM (small layers, latency-bound: each
// CTA streams one unit) take one CTA per SM with five stages instead, 200 KB
// in flight per unit rather than 80 KB: the 64-token 16-expert layer's FFN
// went from 28.5 to 25.2 us, while the V2-Lite-sized layer, with 900 gate/up
// units, ran 5% slower that way.
constexpr int kCtasPerSm = 2;
constexpr int kStages = 2;
constexpr int kDeepCtasPerSm = 1;
constexpr int kDeepStages = 5;
constexpr int kABytes = kBM * 128;                         // 16 KB weight box
constexpr int kBBytes = kBN * 128;                         // 4 KB: one K block of rows
constexpr int kStageBytes = 2 * kABytes + 2 * kBBytes;     // 40 KB
constexpr int smem_bytes(int stages) { return stages * kStageBytes + 1024; }   // + alignment slack
constexpr int kAccBufs = 4;
constexpr int kAccCols = 2 * kBN;                          // gate | up
constexpr int kTmemCols = kAccBufs * kAccCols;             // 256
constexpr int kRing = 4;                                   // claimed units in flight
constexpr int kMaxGroups = 1024;
static_assert(kBN == 32, "one activation row per lane");
static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte swizzle alignment");
static_assert(kTmemCols * kCtasPerSm <= 512, "TMEM columns");
constexpr int kStaticSmem = 2 * 4 * (kMaxGroups + 1) + 2 * 4 * 4 * kBN + 4 * 4 * 2 * 2 * kBN + 1024;
static_assert(smem_bytes(kStages) + kStaticSmem <= 228 * 1024 / kCtasPerSm - 1024,
              "shared memory for two CTAs per SM");
static_assert(smem_bytes(kDeepStages) + kStaticSmem <= 228 * 1024 / kDeepCtasPerSm - 1024,
              "shared memory of a deep-ring CTA");

struct FfnArgs {
    int groups, hidden, inter, rows;
    const int32_t *offsets;
    const float *x_scales;     // [rows, hidden/128]
    const float *w13_scales;   // [groups, 2*inter/128, hidden/128]
    const float *w2_scales;    // [groups, hidden/128, inter/128]
    uint8_t *h;                // [rows, inter] e4m3
    float *h_scales;           // [rows, inter/128]
    float *y;                  // [rows, hidden]
    int32_t *sched;            // [0] next unit; [1 + j] finished gate/up tiles of activation tile j
    int w_tiled;               // W13, W2 in MOE_LAYOUT_TILES (tiles read by 16 KB bulk copies)
    const uint8_t *w13, *w2;   // weight bytes
    int min_rows, max_rows;    // groups whose row count lies outside are skipped
    int32_t *status;
};

struct Unit {
    bool down;
    int g, mt, j, row0, nvalid;
};

// Units: the gate/up tiles of all groups (group-major, then weight tile,
// then activation tile), then the down tiles in the same order.  s_nt is the
// prefix count of activation tiles over groups.
__device__ __forceinline__ Unit decode_unit(int t, int n_gu, int MT1, int MT2, int G,
                                            const int *s_nt, const int *s_off) {
    Unit u;
    u.down = t >= n_gu;
    const int MT = u.down ? MT2 : MT1;
    const int local0 = u.down ? t - n_gu : t;
    const int q = local0 / MT;   // s_nt[g] <= q < s_nt[g + 1] for the unit's group g
    int lo = 0, hi = G;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_nt[mid] <= q) lo = mid;
        else hi = mid;
    }
    u.g = lo;
    const int ntn = s_nt[lo + 1] - s_nt[lo];
    const int local = local0 - MT * s_nt[lo];
    u.mt = local / ntn;
    const int nt = local - u.mt * ntn;
    u.j = s_nt[lo] + nt;
    u.row0 = s_off[lo] + nt * kBN;
    u.nvalid = min(kBN, s_off[lo + 1] - u.row0);
    return u;
}

// FP8: e4m3 operands with per-128-K-block promotion of the fp32 partial
// sums; BF16: bf16 operands, one tensor-memory accumulation over all of K
// per unit, h rounded to bf16.  K blocks are 128 bytes in both.
//
// EW epilogue warpgroups: warp 2 + 4h + j (h < EW) reads TMEM lane quarter
// warp & 3 of the CB = 32/EW activation columns [h CB, (h + 1) CB).
template <bool FP8, int EW, int ST, int CPS>
__global__ void __launch_bounds__(64 + 128 * EW, CPS)
    expert_ffn_kernel(const __grid_constant__ CUtensorMap tmW13,
                      const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmW2,
                      const __grid_constant__ CUtensorMap tmH,
                      const __grid_constant__ CUtensorMap tmX32,
                      const __grid_constant__ CUtensorMap tmH32, const FfnArgs args) {
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t full_bar[ST];
    __shared__ __align__(8) uint64_t empty_bar[ST];
    __shared__ __align__(8) uint64_t acc_full[kAccBufs];
    __shared__ __align__(8) uint64_t acc_empty[kAccBufs];
    __shared__ __align__(8) uint64_t unit_full[kRing];
    __shared__ __align__(8) uint64_t unit_empty[kRing];
    __shared__ __align__(8) uint64_t amax_bar[2];
    __shared__ __align__(8) uint64_t hdone_bar[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_abort, s_bad;
    __shared__ int s_ring[kRing];
    __shared__ int s_off[kMaxGroups + 1];
    __shared__ int s_nt[kMaxGroups + 1];
    __shared__ float s_amax[2][4 * kBN];   // per gate/up tile: each lane quarter's column maxima
    // per epilogue warp and K-block parity: every column's promotion factor
    // x_scale[n, kb] * w_scale[kb] (gate, then up), read as 16-byte broadcasts
    constexpr int CB = kBN / EW;   // activation columns per epilogue warp
    static_assert(CB % 16 == 0, "whole 16-column TMEM loads");
    __shared__ __align__(16) float s_sx[4 * EW][2][2 * CB];

    using namespace ptx;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem_base = (smem_u32(dsmem) + 1023u) & ~1023u;
    const int G = args.groups, H = args.hidden, I = args.inter;
    const int MT1 = I / kBM;    // gate/up tiles per activation tile
    const int MT2 = H / kBM;    // down tiles per activation tile
    constexpr int kKE = FP8 ? 128 : 64;   // elements per 128-byte K block
    const int KB1 = H / kKE;    // K blocks of the gate/up GEMM
    const int KB2 = I / kKE;    // K blocks of the down GEMM (an odd count ends on a 1-block stage)
    volatile int *abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 4 * EW);
        }
        for (int r = 0; r < kRing; ++r) {
            mbar_init(smem_u32(&unit_full[r]), 1);
            mbar_init(smem_u32(&unit_empty[r]), 1 + 4 * EW);   // the MMA thread + every epilogue warp
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&amax_bar[b]), 4 * EW);
            mbar_init(smem_u32(&hdone_bar[b]), 4 * EW);
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
        tma_prefetch_desc(&tmW13);
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW2);
        tma_prefetch_desc(&tmH);
        tma_prefetch_desc(&tmX32);
        tma_prefetch_desc(&tmH32);
    }
    pdl_wait();   // the set-up above overlaps the previous kernel's tail
    for (int i = threadIdx.x; i <= G; i += (int)blockDim.x) s_off[i] = args.offsets[i];
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += (int)blockDim.x) {
        const int a = s_off[g], b = s_off[g + 1];
        if (a < 0 || b < a || b > args.rows) s_bad = 1;
    }
    __syncthreads();
    // activation tiles of group g; none for groups outside the row window
    auto ntiles_of = [&](int g) {
        const int n = s_off[g + 1] - s_off[g];
        return (n < args.min_rows || n > args.max_rows) ? 0 : (n + kBN - 1) / kBN;
    };
    if (warp == 0) {   // activation-tile prefix over groups: lane L owns a contiguous run
        const int per = (G + 31) / 32;
        const int g0 = lane * per;
        int local = 0;
        for (int q = 0; q < per; ++q) {
            const int g = g0 + q;
            if (g < G) local += ntiles_of(g);
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
                s_nt[g] = run;
                run += ntiles_of(g);
            }
        }
        if (lane == 31) s_nt[G] = incl;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;
    const int NT = s_nt[G];
    const int n_gu = MT1 * NT;
    const int total = s_bad ? 0 : n_gu + MT2 * NT;
    if (s_bad && threadIdx.x == 0 && blockIdx.x == 0 && args.status)
        atomicOr(args.status, MOE_DEV_BAD_OFFSETS);

    if (warp == 0) {
        // ------------------------------ scheduler + TMA producer
        if (lane == 0) {
            // Weight boxes are read once unless their group spans several
            // activation tiles (then neighbouring units share the L2 copy);
            // activation and h rows are re-read by every weight tile.
            const uint64_t pol_w_once = policy_evict_first();
            const uint64_t pol_w_shared = policy_evict_normal();
            const uint64_t pol_a = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0, issued = 0, parity_bits = 0;
            bool ok = true;
            for (int i = 0; ok; ++i) {
                const int slot = i % kRing;
                if (!wait_bounded(smem_u32(&unit_empty[slot]), ((uint32_t)(i / kRing) & 1u) ^ 1u,
                                  abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                const int t = atomicAdd(args.sched, 1);
                s_ring[slot] = t;
                mbar_arrive(smem_u32(&unit_full[slot]));
                if (t >= total) {
                    pdl_launch_dependents();   // nothing left to claim
                    break;
                }
                const Unit u = decode_unit(t, n_gu, MT1, MT2, G, s_nt, s_off);
                if (u.down) {   // h rows of activation tile j complete?
                    if (!wait_flag_geq(args.sched + 1 + u.j, MT1, abort_flag, args.status,
                                       MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_global();
                }
                // the unit's activation (or h) rows as one TMA box per K block:
                // 16 rows, or all 32 when more than 16 are valid
                const bool box32 = u.nvalid > kBoxRows;
                const uint32_t abytes = (box32 ? kBN : kBoxRows) * 128;
                const CUtensorMap *tmA = box32 ? &tmX32 : &tmX;
                const CUtensorMap *tmHb = box32 ? &tmH32 : &tmH;
                const int nsteps = u.down ? (KB2 + 1) / 2 : KB1;
                const uint64_t pol_w =
                    (s_off[u.g + 1] - s_off[u.g] > kBN) ? pol_w_shared : pol_w_once;
                const int wrow = u.down ? u.g * H + u.mt * kBM : u.g * 2 * I + u.mt * kBM;
                // tiled weights: box (128-row block b, K block kb) at rows
                // (b * KB + kb) * 128 of a [tiles * 128, 128-byte] view
                const int tb_gate = (u.g * 2 * MT1 + u.mt) * KB1;
                const int tb_up = tb_gate + MT1 * KB1;
                const int tb_down = (u.g * MT2 + u.mt) * KB2;
                const bool tiled = args.w_tiled != 0;
                for (int ks = 0; ks < nsteps; ++ks) {
                    if (!wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1u, abort_flag,
                                      args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_base + stage * kStageBytes;
                    const uint32_t sb = sa + 2 * kABytes;
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    // a down stage holds K blocks 2ks and (if it exists) 2ks + 1
                    const bool two = 2 * ks + 1 < KB2;
                    const uint32_t bytes =
                        u.down ? (two ? 2u : 1u) * (kABytes + abytes) : 2 * kABytes + abytes;
                    mbar_arrive_expect_tx(fb, bytes);
                    if (!u.down) {
                        if (tiled) {   // pre-swizzled 16 KB tiles: plain bulk copies
                            bulk_load(sa, args.w13 + (size_t)(tb_gate + ks) * kABytes, kABytes, fb,
                                      pol_w);
                            bulk_load(sa + kABytes, args.w13 + (size_t)(tb_up + ks) * kABytes,
                                      kABytes, fb, pol_w);
                        } else {
                            tma_load_2d(sa, &tmW13, ks * kKE, wrow, fb, pol_w);            // gate
                            tma_load_2d(sa + kABytes, &tmW13, ks * kKE, wrow + I, fb, pol_w);   // up
                        }
                        tma_load_2d(sb, tmA, ks * kKE, u.row0, fb, pol_a);
                    } else {
#pragma unroll
                        for (int hk = 0; hk < 2; ++hk) {
                            if (hk == 1 && !two) break;
                            const int k0 = (2 * ks + hk) * kKE;
                            if (tiled)
                                bulk_load(sa + hk * kABytes,
                                          args.w2 + (size_t)(tb_down + 2 * ks + hk) * kABytes,
                                          kABytes, fb, pol_w);
                            else
                                tma_load_2d(sa + hk * kABytes, &tmW2, k0, wrow, fb, pol_w);
                            tma_load_2d(sb + hk * kBBytes, tmHb, k0, u.row0, fb, pol_a);
                        }
                    }
                    issued |= 1u << stage;
                    parity_bits = (parity_bits & ~(1u << stage)) | (phase << stage);
                    if (++stage == ST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {   // let every copy in flight land before the CTA exits
                for (int s = 0; s < ST; ++s)
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
            for (int i = 0; ok; ++i) {
                const int slot = i % kRing;
                if (!wait_bounded(smem_u32(&unit_full[slot]), (uint32_t)(i / kRing) & 1u,
                                  abort_flag, args.status, MOE_DEV_TIMEOUT)) {
                    ok = false;
                    break;
                }
                const int t = s_ring[slot];
                mbar_arrive(smem_u32(&unit_empty[slot]));
                if (t >= total) break;
                const Unit u = decode_unit(t, n_gu, MT1, MT2, G, s_nt, s_off);
                const int nmma = ((u.nvalid + 15) / 16) * 16;
                const uint32_t idesc = FP8 ? idesc_e4m3(kBM, nmma) : idesc_bf16(kBM, nmma);
                const int nsteps = u.down ? (KB2 + 1) / 2 : KB1;
                if (!FP8) {   // BF16: one accumulator for the whole unit
                    if (!wait_bounded(smem_u32(&acc_empty[ab]), aphase ^ 1u, abort_flag,
                                      args.status, MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                for (int ks = 0; ks < nsteps && ok; ++ks) {
                    if (!wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag, args.status,
                                      MOE_DEV_TIMEOUT)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_base + stage * kStageBytes;
                    const uint32_t sb = sa + 2 * kABytes;
                    const int nacc = (u.down && 2 * ks + 1 < KB2) ? 2 : 1;
                    for (int hk = 0; hk < nacc; ++hk) {
                        if (FP8) {   // one accumulator per K block
                            if (!wait_bounded(smem_u32(&acc_empty[ab]), aphase ^ 1u, abort_flag,
                                              args.status, MOE_DEV_TIMEOUT)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint32_t d = tmem_base + (uint32_t)(ab * kAccCols);
                        // FP8 starts every K block afresh; BF16 only the unit's first
                        const bool fresh = FP8 || (ks == 0 && hk == 0);
                        auto mma = [&](uint32_t dd, uint64_t a, uint64_t b, bool acc) {
                            if (FP8) mma_f8f6f4(dd, a, b, idesc, acc);
                            else mma_f16(dd, a, b, idesc, acc);
                        };
                        if (!u.down) {
                            const uint64_t dg = sdesc_k_sw128(sa);
                            const uint64_t du = sdesc_k_sw128(sa + kABytes);
                            const uint64_t db = sdesc_k_sw128(sb);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {   // 4 x 32 bytes of K
                                mma(d, dg + 2 * kk, db + 2 * kk, !(fresh && kk == 0));
                                mma(d + kBN, du + 2 * kk, db + 2 * kk, !(fresh && kk == 0));
                            }
                        } else {
                            const uint64_t da = sdesc_k_sw128(sa + hk * kABytes);
                            const uint64_t db = sdesc_k_sw128(sb + hk * kBBytes);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma(d, da + 2 * kk, db + 2 * kk, !(fresh && kk == 0));
                        }
                        if (FP8 || (ks == nsteps - 1 && hk == nacc - 1)) {
                            mma_commit(smem_u32(&acc_full[ab]));
                            if (++ab == kAccBufs) {
                                ab = 0;
                                aphase ^= 1u;
                            }
                        }
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&empty_bar[stage]));
                    if (++stage == ST) {
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
        const uint32_t lane_base = tmem_base + ((uint32_t)(q * 32) << 16);
        const int m_local = q * 32 + lane;
        // a wait's outcome is made warp-uniform: the tcgen05.ld that follow
        // are warp-collective
        auto wwait = [&](uint64_t *bar, uint32_t parity) {
            const bool r = wait_bounded(smem_u32(bar), parity, abort_flag, args.status,
                                        MOE_DEV_TIMEOUT);
            return __all_sync(0xffffffffu, r) != 0;
        };
        int ab = 0, n_done_gu = 0;
        uint32_t aphase = 0;
        bool ok = true;
        for (int i = 0; ok; ++i) {
            const int slot = i % kRing;
            if (!wwait(&unit_full[slot], (uint32_t)(i / kRing) & 1u)) break;
            const int t = s_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&unit_empty[slot]));
            if (t >= total) break;
            const Unit u = decode_unit(t, n_gu, MT1, MT2, G, s_nt, s_off);
            const int nch = (u.nvalid + 15) / 16 - n0 / 16;   // this warp's valid 16-column chunks
            // lane j < CB holds the scale of activation row n0 + j
            const bool row_ok = lane < CB && n0 + lane < u.nvalid;
            float acc[CB], accu[CB];   // columns n0 .. n0 + CB - 1
            if constexpr (FP8) {
                // columns (2p, 2p + 1) side by side for the paired FMA
                uint64_t acc2[CB / 2], accu2[CB / 2];
    #pragma unroll
                for (int p = 0; p < CB / 2; ++p) {
                    acc2[p] = 0ull;
                    accu2[p] = 0ull;
                }
                const int KB = u.down ? KB2 : KB1;
                const float *wsp, *wup = nullptr, *xsp;
                if (!u.down) {
                    wsp = args.w13_scales + ((size_t)u.g * (2 * MT1) + u.mt) * KB1;
                    wup = wsp + (size_t)MT1 * KB1;
                    xsp = args.x_scales + (size_t)(u.row0 + (row_ok ? n0 + lane : 0)) * KB1;
                } else {
                    // h and its scales are written by gate/up units of this launch:
                    // the unit id is published before its producer has seen them
                    // complete, so the epilogue acquires the completion count too
                    // before it reads a scale (lane 0 polls; after the warp
                    // barrier every lane's own acquire load reads the final count)
                    bool dep = true;
                    if (lane == 0)
                        dep = wait_flag_geq(args.sched + 1 + u.j, MT1, abort_flag, args.status,
                                            MOE_DEV_TIMEOUT);
                    if (!__shfl_sync(0xffffffffu, dep, 0)) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    (void)ld_acquire_gpu(args.sched + 1 + u.j);
                    wsp = args.w2_scales + ((size_t)u.g * MT2 + u.mt) * KB2;
                    xsp = args.h_scales + (size_t)(u.row0 + (row_ok ? n0 + lane : 0)) * KB2;
                }
                // scales of K block kb + 1 are fetched while block kb is reduced;
                // h_scales (written during this launch) take coherent loads, the
                // rest the read-only path
                auto xs_at = [&](int kb) {
                    if (!row_ok) return 0.0f;
                    return u.down ? ld_relaxed_gpu_f32(xsp + kb) : __ldg(xsp + kb);
                };
                float xs_n = xs_at(0), sw_n = __ldg(wsp), su_n = u.down ? 0.0f : __ldg(wup);
                for (int kb = 0; kb < KB; ++kb) {
                    const float xs = xs_n, sw = sw_n, su = su_n;
                    if (kb + 1 < KB) {
                        xs_n = xs_at(kb + 1);
                        sw_n = __ldg(wsp + kb + 1);
                        if (!u.down) su_n = __ldg(wup + kb + 1);
                    }
                    float *sxw = s_sx[ew][kb & 1];
                    if (lane < CB) {   // factors of columns n0 + lane: gate at [lane], up at [CB + lane]
                        sxw[lane] = __fmul_rn(xs, sw);
                        if (!u.down) sxw[CB + lane] = __fmul_rn(xs, su);
                    }
                    __syncwarp();
                    if (!wwait(&acc_full[ab], aphase)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t col = (uint32_t)(ab * kAccCols);
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
                    if (!u.down) {   // up rows: same activation scales, their own block scale
    #pragma unroll
                        for (int c = 0; c < CB / 16; ++c)
                            if (c < nch)
                                tmem_ld16(lane_base + col + (uint32_t)(kBN + n0 + c * 16), v[c]);
    #pragma unroll
                        for (int c = 0; c < CB / 16; ++c)
                            if (c < nch) tmem_wait_ld(v[c]);
    #pragma unroll
                        for (int c = 0; c < CB / 16; ++c)
                            if (c < nch) {
    #pragma unroll
                                for (int j4 = 0; j4 < 4; ++j4) {
                                    const uint4 f =
                                        reinterpret_cast<const uint4 *>(sxw + CB)[c * 4 + j4];
                                    const int p = (c * 16 + j4 * 4) / 2;
                                    accu2[p] = fma2(pack2(v[c][j4 * 4], v[c][j4 * 4 + 1]),
                                                    pack2(f.x, f.y), accu2[p]);
                                    accu2[p + 1] = fma2(pack2(v[c][j4 * 4 + 2], v[c][j4 * 4 + 3]),
                                                        pack2(f.z, f.w), accu2[p + 1]);
                                }
                            }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
                    if (++ab == kAccBufs) {
                        ab = 0;
                        aphase ^= 1u;
                    }
                }
                if (!ok) break;
    #pragma unroll
                for (int p = 0; p < CB / 2; ++p) {
                    acc[2 * p] = __uint_as_float((uint32_t)acc2[p]);
                    acc[2 * p + 1] = __uint_as_float((uint32_t)(acc2[p] >> 32));
                    accu[2 * p] = __uint_as_float((uint32_t)accu2[p]);
                    accu[2 * p + 1] = __uint_as_float((uint32_t)(accu2[p] >> 32));
                }
            } else {
                // BF16: the unit's accumulator holds the full sums; the h rows
                // a down unit reads arrive through TMA only (its producer
                // waited for them), so the epilogue reads no scales
                if (!wwait(&acc_full[ab], aphase)) break;
                tc_fence_after();
                const uint32_t col = (uint32_t)(ab * kAccCols);
                uint32_t v[CB / 16][16], vu[CB / 16][16];
#pragma unroll
                for (int c = 0; c < CB / 16; ++c)
                    if (c < nch) {
                        tmem_ld16(lane_base + col + (uint32_t)(n0 + c * 16), v[c]);
                        if (!u.down)
                            tmem_ld16(lane_base + col + (uint32_t)(kBN + n0 + c * 16), vu[c]);
                    }
#pragma unroll
                for (int c = 0; c < CB / 16; ++c)
                    if (c < nch) {
                        tmem_wait_ld(v[c]);
                        if (!u.down) tmem_wait_ld(vu[c]);
                    }
#pragma unroll
                for (int c = 0; c < CB / 16; ++c)
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        acc[c * 16 + jj] = c < nch ? __uint_as_float(v[c][jj]) : 0.0f;
                        accu[c * 16 + jj] = (c < nch && !u.down) ? __uint_as_float(vu[c][jj]) : 0.0f;
                    }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
                if (++ab == kAccBufs) {
                    ab = 0;
                    aphase ^= 1u;
                }
            }

            if (!u.down) {
                // h = silu(gate) * up; FP8: row n is quantised over the tile's
                // 128 features (one per thread): warp maxima, then the four
                // warps' maxima through shared memory; BF16: rounded to bf16
                const int b = n_done_gu & 1;
                const uint32_t par = (uint32_t)(n_done_gu >> 1) & 1u;
#pragma unroll
                for (int n = 0; n < CB; ++n) acc[n] = silu_mul(acc[n], accu[n]);
                if constexpr (!FP8) {
                    __nv_bfloat16 *hb = reinterpret_cast<__nv_bfloat16 *>(args.h);
#pragma unroll
                    for (int n = 0; n < CB; ++n)
                        if (n0 + n < u.nvalid)
                            hb[(size_t)(u.row0 + n0 + n) * I + u.mt * kBM + m_local] =
                                __float2bfloat16_rn(acc[n]);
                } else {
                    // s_amax[b][q' kBN + n]: lane quarter q's maximum of column n
                    float mine = 0.0f;
    #pragma unroll
                    for (int n = 0; n < CB; ++n) {
                        float m = fabsf(acc[n]);
    #pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                        if (n == lane) mine = m;
                    }
                    if (lane < CB) s_amax[b][q * kBN + n0 + lane] = mine;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&amax_bar[b]));
                    if (!wwait(&amax_bar[b], par)) break;
    #pragma unroll
                    for (int j = 0; j < CB; ++j)
                        if (n0 + j < u.nvalid) {
                            const int n = n0 + j;
                            const float amax = fmaxf(fmaxf(s_amax[b][n], s_amax[b][kBN + n]),
                                                     fmaxf(s_amax[b][2 * kBN + n], s_amax[b][3 * kBN + n]));
                            const float sc = fp8_group_scale(amax);
                            const size_t row = (size_t)(u.row0 + n);
                            args.h[row * I + u.mt * kBM + m_local] =
                                fp8_code(acc[j], fp8_group_inv(sc));
                            if (m_local == 0) args.h_scales[row * KB2 + u.mt] = sc;
                        }
                }
                // publish: every epilogue warp's h stores, then one release
                fence_proxy_async_global();
                __syncwarp();
                if constexpr (!FP8) {
                    // hdone_bar[b] served gate/up tile n_done_gu - 2 before: that
                    // phase must be complete before this arrival, or a warp two
                    // tiles ahead could finish it for a slower one (FP8 warps
                    // are held in step by the amax exchange)
                    if (!wwait(&hdone_bar[b], par ^ 1u)) break;
                }
                if (lane == 0) mbar_arrive(smem_u32(&hdone_bar[b]));
                if (ew == 0) {   // warp 2 publishes
                    if (!wwait(&hdone_bar[b], par)) break;
                    if (lane == 0) {
                        __threadfence();
                        fence_proxy_async_global();
                        red_release_gpu_add(args.sched + 1 + u.j, 1);
                    }
                    __syncwarp();
                }
                ++n_done_gu;
            } else {
#pragma unroll
                for (int n = 0; n < CB; ++n)
                    if (n0 + n < u.nvalid)
                        args.y[(size_t)(u.row0 + n0 + n) * H + u.mt * kBM + m_local] = acc[n];
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

size_t ffn_sched_bytes(int groups, int rows) {
    return (size_t)4 * (1 + (size_t)groups + (size_t)ceil_div(rows, kBN));
}

namespace {

struct FfnMaps {
    CUtensorMap w13, x, w2, h, x32, h32;
};

// two epilogue warpgroups: FP8 promotes every K block, and more warps per SM
// sub-partition hide those latencies (BF16: neutral to slightly faster)
constexpr int kEW = 2;

template <bool FP8, int ST, int CPS>
int launch_ffn_cfg(const FfnMaps &m, const FfnArgs &a, int64_t units_bound, cudaStream_t s) {
    constexpr int kSmem = smem_bytes(ST);
    auto kern = expert_ffn_kernel<FP8, kEW, ST, CPS>;
    static std::once_flag attr_once[64];
    static int attr_rc[64];
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return cuda_fail("device ordinal beyond 63");
    std::call_once(attr_once[dev], [&] {
        attr_rc[dev] = (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kSmem);
    });
    if (attr_rc[dev]) return cuda_fail("cudaFuncSetAttribute", (cudaError_t)attr_rc[dev]);
    const int grid = (int)std::min<int64_t>((int64_t)sm_count() * CPS, units_bound);
    if (launch_dependent(kern, dim3(grid), dim3(64 + 128 * kEW), kSmem, s, m.w13, m.x, m.w2,
                         m.h, m.x32, m.h32, a))
        return MOE_ERR_CUDA;
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

template <bool FP8>
int launch_ffn_impl(int groups, int hidden, int inter, int rows, const void *xp,
                    const float *xp_scales, const int32_t *offsets, const void *w13,
                    const float *w13_scales, const void *w2, const float *w2_scales,
                    bool w_tiled, void *h, float *h_scales, float *y, int32_t *sched,
                    bool sched_zeroed, int32_t *status, cudaStream_t s, int min_rows,
                    int max_rows) {
    if (rows == 0) return MOE_OK;
    constexpr int kKE = FP8 ? 128 : 64;
    FfnMaps m;
    const uint64_t w13_rows = (uint64_t)groups * 2 * inter, w2_rows = (uint64_t)groups * hidden;
    const bool w_ok =
        w_tiled ? encode_2d(&m.w13, w13, FP8, kKE, w13_rows * (hidden / kKE), kBM) &&
                      encode_2d(&m.w2, w2, FP8, kKE, w2_rows * (inter / kKE), kBM)
                : encode_2d(&m.w13, w13, FP8, (uint64_t)hidden, w13_rows, kBM) &&
                      encode_2d(&m.w2, w2, FP8, (uint64_t)inter, w2_rows, kBM);
    if (!w_ok ||
        !encode_2d(&m.x, xp, FP8, (uint64_t)hidden, (uint64_t)rows, kBoxRows) ||
        !encode_2d(&m.h, h, FP8, (uint64_t)inter, (uint64_t)rows, kBoxRows) ||
        !encode_2d(&m.x32, xp, FP8, (uint64_t)hidden, (uint64_t)rows, kBN) ||
        !encode_2d(&m.h32, h, FP8, (uint64_t)inter, (uint64_t)rows, kBN))
        return cuda_fail("cuTensorMapEncodeTiled");
    if (!sched_zeroed) MOE_CUDA_TRY(cudaMemsetAsync(sched, 0, ffn_sched_bytes(groups, rows), s));
    FfnArgs a;
    a.groups = groups;
    a.hidden = hidden;
    a.inter = inter;
    a.rows = rows;
    a.offsets = offsets;
    a.x_scales = xp_scales;
    a.w13_scales = w13_scales;
    a.w2_scales = w2_scales;
    a.h = static_cast<uint8_t *>(h);   // e4m3 or bf16 bytes
    a.h_scales = h_scales;
    a.y = y;
    a.sched = sched;
    a.w_tiled = w_tiled;
    a.w13 = static_cast<const uint8_t *>(w13);
    a.w2 = static_cast<const uint8_t *>(w2);
    a.min_rows = min_rows;
    a.max_rows = max_rows;
    a.status = status;
    // activation tiles are at most one per group plus one per 32 rows
    const int64_t tiles_bound = groups + ceil_div(rows, kBN);
    const int64_t units_bound = (int64_t)(inter / kBM + hidden / kBM) * tiles_bound;
    if constexpr (!FP8) {
        if ((int64_t)(inter / kBM) * tiles_bound <= (int64_t)sm_count() * kDeepCtasPerSm)
            return launch_ffn_cfg<FP8, kDeepStages, kDeepCtasPerSm>(m, a, units_bound, s);
    }
    return launch_ffn_cfg<FP8, kStages, kCtasPerSm>(m, a, units_bound, s);
}

}  // namespace

int launch_expert_ffn(bool fp8, int groups, int hidden, int inter, int rows, const void *xp,
                      const float *xp_scales, const int32_t *offsets, const void *w13,
                      const float *w13_scales, const void *w2, const float *w2_scales,
                      bool w_tiled, void *h, float *h_scales, float *y, int32_t *sched,
                      bool sched_zeroed, int32_t *status, cudaStream_t s, int min_rows,
                      int max_rows) {
    auto f = fp8 ? launch_ffn_impl<true> : launch_ffn_impl<false>;
    return f(groups, hidden, inter, rows, xp, xp_scales, offsets, w13, w13_scales, w2, w2_scales,
             w_tiled, h, h_scales, y, sched, sched_zeroed, status, s, min_rows, max_rows);
}

}  // namespace moe

// ---- self-test of the inter-CTA flag wait ------------------------------------
namespace moe {
namespace {

constexpr int kSelftestH = 128, kSelftestI = 256;

__global__ void ffn_selftest_init_kernel(int32_t *offsets, int32_t *sched, int n_gu) {
    if (threadIdx.x == 0) {
        offsets[0] = 0;
        offsets[1] = 1;
        sched[0] = n_gu;   // every gate/up unit counts as claimed; none will finish
    }
}

struct SelftestLayout {
    size_t xp, xs, off, w13, w13s, w2, w2s, h, hs, y, sched, total;
};

SelftestLayout selftest_layout() {
    SelftestLayout L;
    size_t o = 0;
    auto take = [&](size_t b) {
        const size_t r = o;
        o = align_up(o + b);
        return r;
    };
    L.xp = take(kSelftestH);
    L.xs = take(4 * (kSelftestH / 128));
    L.off = take(8);
    L.w13 = take((size_t)2 * kSelftestI * kSelftestH);
    L.w13s = take(4 * (2 * kSelftestI / 128) * (kSelftestH / 128));
    L.w2 = take((size_t)kSelftestH * kSelftestI);
    L.w2s = take(4 * (kSelftestH / 128) * (kSelftestI / 128));
    L.h = take(kSelftestI);
    L.hs = take(4 * (kSelftestI / 128));
    L.y = take(4 * kSelftestH);
    L.sched = take(ffn_sched_bytes(1, 1));
    L.total = o;
    return L;
}

}  // namespace
}  // namespace moe

extern "C" MOE_API size_t moe_selftest_ffn_flag_timeout_scratch_bytes(void) {
    return moe::selftest_layout().total;
}

extern "C" MOE_API int moe_selftest_ffn_flag_timeout(void *scratch, size_t scratch_bytes,
                                                     int32_t *dev_status, void *stream) {
    using namespace moe;
    const SelftestLayout L = selftest_layout();
    if (!scratch || !dev_status || !aligned16(scratch) || scratch_bytes < L.total)
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *b = static_cast<uint8_t *>(scratch);
    MOE_CUDA_TRY(cudaMemsetAsync(b, 0, L.total, s));
    int32_t *off = reinterpret_cast<int32_t *>(b + L.off);
    int32_t *sched = reinterpret_cast<int32_t *>(b + L.sched);
    const int n_gu = kSelftestI / 128;   // gate/up units of the one 32-row activation tile
    ffn_selftest_init_kernel<<<1, 32, 0, s>>>(off, sched, n_gu);
    MOE_LAUNCH_CHECK();
    return launch_expert_ffn(true, 1, kSelftestH, kSelftestI, 1, b + L.xp,
                             reinterpret_cast<const float *>(b + L.xs), off, b + L.w13,
                             reinterpret_cast<const float *>(b + L.w13s), b + L.w2,
                             reinterpret_cast<const float *>(b + L.w2s), false, b + L.h,
                             reinterpret_cast<float *>(b + L.hs), reinterpret_cast<float *>(b + L.y),
                             sched, true, dev_status, s);
}

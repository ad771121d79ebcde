// Dispatch on one GPU: every (token, choice) slot is given a row in its
// expert's contiguous block of rows, and the token's activations are copied
// there (Moreh report "21K output tokens/s DeepSeek inference on MI300X with
// Expert Parallelism", sections "Overview" and "Compute-communication
// overlap": the all-to-all dispatch that brings tokens to their experts).
//
// Row of routed slot i with expert e:
//   expert_offsets[e] + #{ i' < i : e_i' = e }
// so rows within an expert are in slot order and the result does not depend
// on the order threads run in.  Three kernels (the first two as one for
// batches of at most 1024 routed slots):
//   permute_count    1024 slots per CTA: warp-level __match_any_sync gives
//                    each slot its rank among equal ids of its warp, a
//                    shared-memory table of per-warp counts gives the rank
//                    inside the CTA, and the CTA's histogram goes to scratch.
//   permute_scan     one CTA: totals per expert, exclusive scan into
//                    expert_offsets (shared experts: T rows each), and the
//                    first row of every (chunk, expert).
//   permute_scatter  one warp per row: writes row_of_slot / src_of_row and
//                    copies the row (16-byte vectors) and its scales, unless
//                    the row's group has more rows than copy_max_rows (a
//                    GEMM that gathers the token rows itself reads them).
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kChunk = 1024;   // slots per permute_count CTA

struct PermArgs {
    int T, k, E, S, H, fp8;
    const int32_t *ids;
    const uint8_t *x;
    const float *xs;
    int32_t *offsets, *src_of_row, *row_of_slot;
    uint8_t *xp;
    float *xps;
    int32_t *chunk_counts;   // [chunks, E]
    int32_t *chunk_base;     // [chunks, E]
    int32_t *local_rank;     // [T*k]
    int copy_max_rows;       // rows of groups with more rows are not copied (tables only)
    int32_t *status;
};

// Counts of chunk `chunk` (1024 slots): ranks among equal ids, histogram.
__device__ __forceinline__ void count_chunk(const PermArgs &a, int chunk, int32_t *wc) {
    const int R = a.T * a.k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int i = chunk * kChunk + tid;
    for (int j = tid; j < 32 * a.E; j += kChunk) wc[j] = 0;
    int e = -1;
    if (i < R) {
        e = a.ids[i];
        if (e < 0 || e >= a.E) {
            if (a.status) atomicOr(a.status, MOE_DEV_BAD_EXPERT_ID);
            e = -1;
        }
    }
    __syncthreads();
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) wc[warp * a.E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
        int r = rank;
        for (int w = 0; w < warp; ++w) r += wc[w * a.E + e];
        a.local_rank[i] = r;
    }
    for (int ee = tid; ee < a.E; ee += kChunk) {
        int c = 0;
        for (int w = 0; w < 32; ++w) c += wc[w * a.E + ee];
        a.chunk_counts[(size_t)chunk * a.E + ee] = c;
    }
}

__global__ void __launch_bounds__(kChunk) permute_count_kernel(const PermArgs a) {
    extern __shared__ int32_t wc[];   // [32 warps][E]
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();   // routing ids
    count_chunk(a, blockIdx.x, wc);
}

// Exclusive scan of `v` over the CTA (1024 threads); returns the total too.
__device__ int block_exclusive_scan(int v, int *total, int *sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = sh[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        sh[lane] = wi - w;          // exclusive prefix of warp totals
        if (lane == 31) sh[32] = wi;
    }
    __syncthreads();
    const int res = sh[warp] + incl - v;
    *total = sh[32];
    __syncthreads();
    return res;
}

// Offsets of all groups and the first row of every (chunk, expert).
__device__ __forceinline__ void scan_chunks(const PermArgs &a, int chunks, int *sh) {
    const int G = a.E + a.S;
    const int per = (G + 1023) / 1024;   // consecutive groups per thread
    const int g0 = threadIdx.x * per;
    int local = 0;
    for (int q = 0; q < per; ++q) {
        const int g = g0 + q;
        if (g >= G) break;
        int n = 0;
        if (g < a.E) {
            for (int c = 0; c < chunks; ++c) n += a.chunk_counts[(size_t)c * a.E + g];
        } else {
            n = a.T;
        }
        local += n;
    }
    int total;
    int run = block_exclusive_scan(local, &total, sh);
    for (int q = 0; q < per; ++q) {
        const int g = g0 + q;
        if (g >= G) break;
        a.offsets[g] = run;
        if (g < a.E) {
            for (int c = 0; c < chunks; ++c) {
                a.chunk_base[(size_t)c * a.E + g] = run;
                run += a.chunk_counts[(size_t)c * a.E + g];
            }
        } else {
            run += a.T;
        }
    }
    if (threadIdx.x == 0) a.offsets[G] = total;
}

__global__ void __launch_bounds__(1024) permute_scan_kernel(const PermArgs a, int chunks) {
    __shared__ int sh[33];
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();   // per-chunk counts
    scan_chunks(a, chunks, sh);
}

// Decode batches (at most 1024 routed slots, one chunk): count and scan in
// one CTA, one launch fewer.  The CTA barrier orders the counts written to
// global memory before the scan reads them.
__global__ void __launch_bounds__(kChunk) permute_count_scan_kernel(const PermArgs a) {
    extern __shared__ int32_t wc[];   // [32 warps][E]
    __shared__ int sh[33];
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();   // routing ids
    count_chunk(a, 0, wc);
    __syncthreads();
    scan_chunks(a, 1, sh);
}

__global__ void __launch_bounds__(256) permute_scatter_kernel(const PermArgs a) {
    ptx::pdl_launch_dependents();
    ptx::pdl_wait();   // offsets and ranks
    const int lane = threadIdx.x & 31;
    const long w = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const long R = (long)a.T * a.k;
    const long Rtot = R + (long)a.S * a.T;
    if (w >= Rtot) return;
    long row;
    int t, group_rows;
    if (w < R) {
        const int e = a.ids[w];
        if (e < 0 || e >= a.E) {   // reported by permute_count
            if (lane == 0) a.row_of_slot[w] = -1;
            return;
        }
        row = a.chunk_base[(w / kChunk) * a.E + e] + a.local_rank[w];
        t = (int)(w / a.k);
        group_rows = a.offsets[e + 1] - a.offsets[e];
        if (lane == 0) {
            a.row_of_slot[w] = (int32_t)row;
            a.src_of_row[row] = (int32_t)w;
        }
    } else {
        const long ws = w - R;
        const int s = (int)(ws / a.T);
        t = (int)(ws % a.T);
        row = a.offsets[a.E + s] + t;
        group_rows = a.T;
        if (lane == 0) a.src_of_row[row] = (int32_t)w;
    }
    if (group_rows > a.copy_max_rows) return;   // its rows are gathered by the GEMM
    const long row_bytes = a.fp8 ? a.H : 2L * a.H;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (long)t * row_bytes);
    uint4 *dst = reinterpret_cast<uint4 *>(a.xp + row * row_bytes);
    // up to 8 loads per lane in flight before their stores (a 7168-byte row:
    // two rounds; same-box at 4096 tokens 68.6 -> 67.1 us)
    const long nvec = row_bytes / 16;
    for (long v0 = lane; v0 < nvec; v0 += 32 * 8) {
        uint4 buf[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (v0 + 32 * u < nvec) buf[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (v0 + 32 * u < nvec) dst[v0 + 32 * u] = buf[u];
    }
    if (a.fp8) {
        const int ng = a.H / 128;
        for (int g = lane; g < ng; g += 32) a.xps[row * ng + g] = __ldg(a.xs + (long)t * ng + g);
    }
}

}  // namespace

int permute_kernel_count(const moe_config *cfg, int T) {
    return (int64_t)T * cfg->top_k <= kChunk ? 2 : 3;
}

size_t permute_scratch_bytes(const moe_config *cfg, int T) {
    const int64_t R = (int64_t)T * cfg->top_k;
    const int64_t chunks = ceil_div(R, kChunk);
    return align_up(4 * (size_t)(chunks * cfg->num_experts)) * 2 + align_up(4 * (size_t)R);
}

int launch_permute(const moe_config *cfg, int T, const int32_t *topk_ids, const void *x_rows,
                   const float *x_scales, int32_t *offsets, int32_t *src_of_row,
                   int32_t *row_of_slot, void *xp, float *xp_scales, void *ws,
                   int32_t *status, cudaStream_t s, int copy_max_rows) {
    PermArgs a;
    a.T = T;
    a.k = cfg->top_k;
    a.E = cfg->num_experts;
    a.S = cfg->num_shared;
    a.H = cfg->hidden;
    a.fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    a.ids = topk_ids;
    a.x = static_cast<const uint8_t *>(x_rows);
    a.xs = x_scales;
    a.offsets = offsets;
    a.src_of_row = src_of_row;
    a.row_of_slot = row_of_slot;
    a.xp = static_cast<uint8_t *>(xp);
    a.xps = xp_scales;
    const int64_t R = (int64_t)T * a.k;
    const int chunks = (int)ceil_div(R, kChunk);
    uint8_t *p = static_cast<uint8_t *>(ws);
    const size_t cc = align_up(4 * (size_t)((int64_t)chunks * a.E));
    a.chunk_counts = reinterpret_cast<int32_t *>(p);
    a.chunk_base = reinterpret_cast<int32_t *>(p + cc);
    a.local_rank = reinterpret_cast<int32_t *>(p + 2 * cc);
    a.copy_max_rows = copy_max_rows;
    a.status = status;

    const size_t smem = 32 * sizeof(int32_t) * (size_t)a.E;
    if (chunks <= 1) {   // count (if any slot) and scan in one CTA
        if (smem > 48 * 1024)
            MOE_CUDA_TRY(cudaFuncSetAttribute(permute_count_scan_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)smem));
        if (launch_dependent(permute_count_scan_kernel, dim3(1), dim3(kChunk), smem, s, a))
            return MOE_ERR_CUDA;
        MOE_LAUNCH_CHECK();
    } else {
        if (smem > 48 * 1024)
            MOE_CUDA_TRY(cudaFuncSetAttribute(permute_count_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)smem));
        if (launch_dependent(permute_count_kernel, dim3(chunks), dim3(kChunk), smem, s, a))
            return MOE_ERR_CUDA;
        MOE_LAUNCH_CHECK();
        if (launch_dependent(permute_scan_kernel, dim3(1), dim3(1024), 0, s, a, chunks))
            return MOE_ERR_CUDA;
        MOE_LAUNCH_CHECK();
    }
    const int64_t rows = total_rows(cfg, T);
    if (rows > 0) {
        if (launch_dependent(permute_scatter_kernel, dim3((unsigned)ceil_div(rows, 8)), dim3(256),
                             0, s, a))
            return MOE_ERR_CUDA;
        MOE_LAUNCH_CHECK();
    }
    return MOE_OK;
}

}  // namespace moe

// moe_permute for callers that cannot allocate device memory.
//
// Some callers cannot hand this library a workspace: a plugin inside a host
// framework that owns every device allocation and exposes none to its
// extensions, or a runtime that works within a fixed, pre-reserved memory
// budget and forbids allocation once it is serving.  This entry point runs
// the same dispatch kernels as moe_permute, with their scratch (per-chunk
// expert counts, per-chunk first rows, per-slot ranks) in a file-scope
// device array instead of a caller buffer.  The array is part of the
// library image: every GPU that loads the library holds it until the
// process exits.
#include <cuda.h>

#include <mutex>

#include "internal.h"

namespace {

// Capacity of the static scratch, per device.
constexpr size_t kStaticScratchBytes = size_t(1) << 20;   // 1 MiB

static __device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

// Identity of the current CUDA context (driver entry points looked up at run
// time, so the library still loads where no driver is installed); 0 when it
// cannot be told.
unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// The array's device address for the current device.  In host code the
// symbol names a host-side stand-in, never the device memory, so the address
// is looked up (with the device current) the first time a device is used and
// again whenever that device's context has changed since (a device reset
// unloads the module that holds the array, and the old address would be
// stale); where the context cannot be identified it is looked up on every call.
int static_scratch_address(void **out) {
    static std::mutex mu;
    static void *addr[64];
    static unsigned long long ctx_of[64];
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return moe::cuda_fail("cudaGetDevice", e);
    if (dev < 0 || dev >= 64) return moe::cuda_fail("device ordinal beyond 63");
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (ctx == 0 || ctx_of[dev] != ctx || !addr[dev]) {
        void *p = nullptr;
        const cudaError_t es = cudaGetSymbolAddress(&p, g_permute_scratch);
        if (es != cudaSuccess || p == nullptr) return moe::cuda_fail("cudaGetSymbolAddress", es);
        addr[dev] = p;
        ctx_of[dev] = ctx;
    }
    *out = addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" MOE_API int moe_permute_static_scratch(
    const moe_config *cfg, int32_t T, const int32_t *topk_ids, const void *x_rows,
    const float *x_scales, int32_t *expert_offsets, int32_t *src_of_row, int32_t *row_of_slot,
    void *xp, float *xp_scales, int32_t *dev_status, void *stream) {
    int rc = moe::check_config(cfg);
    if (rc) return rc;
    if (T < 0 || !expert_offsets) return MOE_ERR_INVALID_ARG;
    const bool fp8 = cfg->dtype == MOE_DTYPE_FP8_BLOCK128;
    if (T > 0 && (!topk_ids || !x_rows || !src_of_row || !row_of_slot || !xp ||
                  (fp8 && (!x_scales || !xp_scales))))
        return MOE_ERR_INVALID_ARG;
    if ((x_rows && !moe::aligned16(x_rows)) || (xp && !moe::aligned16(xp)))
        return MOE_ERR_INVALID_ARG;
    if (moe::permute_scratch_bytes(cfg, T) > kStaticScratchBytes)
        return MOE_ERR_UNSUPPORTED_SHAPE;   // beyond the static scratch capacity
    void *scratch = nullptr;
    rc = static_scratch_address(&scratch);
    if (rc) return rc;
    return moe::launch_permute(cfg, T, topk_ids, x_rows, x_scales, expert_offsets, src_of_row,
                               row_of_slot, xp, xp_scales, scratch, dev_status,
                               static_cast<cudaStream_t>(stream));
}

extern "C" MOE_API size_t moe_permute_static_scratch_capacity(void) { return kStaticScratchBytes; }

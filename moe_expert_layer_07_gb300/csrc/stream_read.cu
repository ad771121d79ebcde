// Measurement utility: the rate at which this GPU reads HBM when nothing else
// is done with the data.  The layer's decode path is bound by streaming expert
// weights, and a copy (read + write) understates how fast a read-only stream
// can go, so a roofline for such a path wants a read-stream rate measured on
// the same device.  Persistent CTAs (one thread each, one per SM) move
// consecutive 64 KB chunks of the buffer into a 3-deep shared-memory ring with
// 1-D bulk copies (cp.async.bulk) and discard them.  Every wait is bounded:
// on a timeout the CTA records MOE_DEV_TIMEOUT, lets its other copies land
// (bounded) and returns.
#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kChunk = 64 * 1024;
constexpr int kRing = 3;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__global__ void __launch_bounds__(32, 1)
    stream_read_kernel(const uint8_t *__restrict__ src, size_t chunks, int32_t *status) {
    using namespace ptx;
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t bar[kRing];
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    for (int s = 0; s < kRing; ++s) mbar_init(smem_u32(&bar[s]), 1);
    abort_flag = 0;
    fence_mbar_init();
    const uint32_t base = (smem_u32(ring) + 127u) & ~127u;
    uint32_t parity = 0;   // bit s: parity of the next completion of slot s
    size_t issued = 0, waited = 0;
    bool ok = true;
    for (size_t c = blockIdx.x; c < chunks && ok; c += gridDim.x, ++issued) {
        const int slot = (int)(issued % kRing);
        if (issued >= (size_t)kRing) {   // the copy that last used this slot has landed
            if (!wait_bounded(smem_u32(&bar[slot]), (parity >> slot) & 1u, &abort_flag, status,
                              MOE_DEV_TIMEOUT)) {
                ok = false;
                break;
            }
            parity ^= 1u << slot;
            ++waited;
        }
        mbar_arrive_expect_tx(smem_u32(&bar[slot]), kChunk);
        bulk_load(base + slot * kChunk, src + c * (size_t)kChunk, kChunk, smem_u32(&bar[slot]));
    }
    for (size_t m = waited; m < issued; ++m) {   // drain, the late copy included (bounded)
        const int slot = (int)(m % kRing);
        if (!wait_drain(smem_u32(&bar[slot]), (parity >> slot) & 1u)) break;
        parity ^= 1u << slot;
    }
}

}  // namespace
}  // namespace moe

extern "C" MOE_API size_t moe_stream_read_granule(void) { return moe::kChunk; }

extern "C" MOE_API int moe_stream_read(const void *src, size_t bytes, int32_t *dev_status,
                                       void *stream) {
    using namespace moe;
    if (!src || !aligned16(src) || bytes % kChunk) return MOE_ERR_INVALID_ARG;
    if (bytes == 0) return MOE_OK;
    static std::once_flag attr_once[64];
    static int attr_rc[64];
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return cuda_fail("device ordinal beyond 63");
    const int smem = kRing * kChunk + 128;
    std::call_once(attr_once[dev], [&] {
        attr_rc[dev] = (int)cudaFuncSetAttribute(stream_read_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_rc[dev]) return cuda_fail("cudaFuncSetAttribute", (cudaError_t)attr_rc[dev]);
    const size_t chunks = bytes / kChunk;
    const int grid = (int)std::min<size_t>((size_t)sm_count(), chunks);
    stream_read_kernel<<<grid, 32, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(src), chunks, dev_status);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

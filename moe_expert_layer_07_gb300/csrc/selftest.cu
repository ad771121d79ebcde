// Self-test of the bounded pipeline wait that every tcgen05/TMA kernel of the
// library uses: one warp waits on an mbarrier that is completed (must pass)
// and on one that nothing ever arrives on (must give up after the limit and
// record MOE_DEV_TIMEOUT).  The kernel always returns; nothing faults.
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void bounded_wait_selftest_kernel(int32_t *status, uint64_t limit_ns,
                                             int32_t *passed) {
    __shared__ __align__(8) uint64_t done_bar, never_bar;
    __shared__ int abort_flag;
    using namespace ptx;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&done_bar), 1);
        mbar_init(smem_u32(&never_bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_arrive(smem_u32(&done_bar));
    __syncwarp();
    const bool ok = wait_bounded(smem_u32(&done_bar), 0, &abort_flag, status, MOE_DEV_TIMEOUT,
                                 limit_ns);
    const bool late = wait_bounded(smem_u32(&never_bar), 0, &abort_flag, status,
                                   MOE_DEV_TIMEOUT, limit_ns);
    if (threadIdx.x == 0 && passed) *passed = (ok ? 1 : 0) | (late ? 0 : 2);
}

}  // namespace
}  // namespace moe

extern "C" MOE_API int moe_selftest_bounded_wait(int32_t *dev_status, int64_t limit_ns,
                                                 int32_t *dev_result, void *stream) {
    if (!dev_status || !dev_result || limit_ns < 1000 || limit_ns > 100000000)
        return MOE_ERR_INVALID_ARG;
    moe::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        dev_status, (uint64_t)limit_ns, dev_result);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
}

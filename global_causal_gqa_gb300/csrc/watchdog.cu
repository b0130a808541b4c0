// watchdog.cu -- a self-test of the bounded-wait watchdog that every kernel relies on.
//
// One warp initialises an mbarrier that nothing ever arrives on and waits for it with the
// same bounded wait and the same error reporting as the attention kernels.  The wait must
// expire after the requested time; the kernel then records GQA_ERR_DEVICE_TIMEOUT and its
// diagnostic code in the status word and returns normally, leaving the context usable.
// No fault, trap or endless loop is involved.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {
namespace {

__global__ void __launch_bounds__(32, 1) watchdog_selftest_kernel(int *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // no thread arrives on `bar`, so its phase 0 never completes
    const bool done = __all_sync(0xffffffffu, mbar_wait_for(&bar, 0, limit_ns));
    if (!done && threadIdx.x == 0) set_timeout(status, kDiagWatchdog, 0, 0, 0);
}

}  // namespace

cudaError_t launch_watchdog_selftest(int64_t limit_ns, int *status, cudaStream_t s) {
    watchdog_selftest_kernel<<<1, 32, 0, s>>>(status, static_cast<uint64_t>(limit_ns));
    return cudaPeekAtLastError();
}

}  // namespace gqa

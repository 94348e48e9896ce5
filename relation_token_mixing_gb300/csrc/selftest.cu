// Self-test of the bounded device-side wait that every kernel of the library
// uses for failure detection: one warp waits on an mbarrier that nothing
// arrives on, so the wait runs out after its limit, records a timeout code in
// the device status word, raises the CTA's abort flag and returns.  Nothing
// faults, traps or hangs; the context stays usable.
#include "common.cuh"
#include "kernels.h"
#include "ptx_sm100.cuh"

namespace relation {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t limit_ns, unsigned int* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    (void)ptx::mbar_wait_for(&bar, 0, &abort_flag, status, kDevTimeoutFull, limit_ns);
    __syncwarp();
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, unsigned int* status, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, status);
    return cudaGetLastError();
}

}  // namespace relation

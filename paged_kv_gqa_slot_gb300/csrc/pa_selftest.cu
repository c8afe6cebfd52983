// pa_selftest.cu -- a check that the library's bounded waits end and report.
//
// Every wait on an mbarrier in the kernels gives up after a fixed number of SM cycles, sets
// PA_DEV_TIMEOUT in the device status word and lets the kernel return, so that a lost arrival
// becomes an error the host reads instead of a hung GPU.  This kernel makes one such wait run
// out on purpose -- an mbarrier nothing ever arrives on, waited for through the kernels' own
// helper with a short limit -- so that the path is exercised without any fault: no trap, no
// bad address, no unbounded loop.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(unsigned* status, long long limit_cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    // phase 0 of a barrier with one expected arrival and none coming: the wait gives up
    if (threadIdx.x == 0 && !mbar_wait_for(&bar, 0, limit_cycles)) atomicOr(status, kDevTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned* status, long long limit_cycles, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(status, limit_cycles);
    return cudaGetLastError();
}

}  // namespace pa

// k_selftest.cu -- a self-test of the device-side failure path.
//
// Every wait in the library's kernels is bounded: when it runs out the kernel
// latches DEV_ERR_TIMEOUT in the device error flag and unwinds, and
// qmm_check_device_error() reports QMM_ERR_DEVICE_TIMEOUT. This kernel makes
// such a wait run out on purpose -- an mbarrier that nothing ever arrives on --
// so a test can check that the status reaches the host and that the context
// stays usable. Nothing here traps or faults.
#include "qmm.h"
#include "qmm_internal.cuh"
#include "sm100_async.cuh"

namespace qmm {
namespace {

__global__ void k_wait_never(unsigned* err, long long limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    const long long t0 = clock64();
    while (!mbar_try_wait(&bar, 0)) {   // phase 0 never completes
        if (clock64() - t0 > limit) {
            atomicOr(err, DEV_ERR_TIMEOUT);
            break;
        }
    }
    // complete the phase so the barrier is left in a clean state
    mbar_arrive(&bar);
}

}  // namespace

cudaError_t launch_wait_never(unsigned* err, long long cycles, cudaStream_t s) {
    k_wait_never<<<1, 32, 0, s>>>(err, cycles);
    count_launch(1);
    return cudaGetLastError();
}

}  // namespace qmm

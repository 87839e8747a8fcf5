// selftest.cu -- a kernel that stalls one wait on purpose, so that a caller
// can see on the device at hand that the library's bounded waits end with an
// error status rather than a hang (sm_103a).
#include <cuda_runtime.h>
#include <stdint.h>

#include "shkv_device.cuh"

namespace shkv {

// One thread waits, through the same bounded wait every kernel of this
// library uses, for phase 0 of a fresh mbarrier that nothing arrives at.
// After kWaitLimitNs the wait gives up: it raises the CTA's abort flag, sets
// SHKV_ERRF_TIMEOUT in err and returns, and the kernel exits normally.  No
// copy or MMA is in flight, so nothing else needs draining.
__global__ void shkv_wait_selftest_kernel(uint32_t *err)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait_bounded(smem_u32(&bar), 0u, &abort_flag, err);
}

cudaError_t launch_wait_selftest(uint32_t *err, cudaStream_t stream)
{
    shkv_wait_selftest_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

}  // namespace shkv

// launch.cuh -- host-side kernel launch with programmatic stream
// serialization (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace shkv {

// kern<<<grid, block, smem, stream>>>(args...), allowed to start its CTAs
// while the previous kernel of the stream is still finishing.  The kernel
// must call pdl_wait_prior() before it touches global memory, and calls
// pdl_launch_dependents() only after that wait: so once a kernel of this
// library lets its dependent start, everything before it in the stream has
// completed.  The per-decoder tails unit kernel relies on this (it is the
// one exception to the first rule: it reads the page tables before its wait,
// see shkv_tails_unit_kernel).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int block, uint32_t smem, cudaStream_t stream,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace shkv

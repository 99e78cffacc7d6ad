// Kernel launches with programmatic dependent launch (sm_90 and later).
//
// A step is a chain of short dependent kernels on one stream (accumulate,
// norm partials, final reduction, AdamW).  Every kernel of the library is
// launched with programmatic stream serialisation and begins with
// pdl_enter(): it lets the next kernel in the stream be scheduled as soon as
// all of its own blocks have started, then waits until its predecessor has
// completed and that grid's memory operations are visible.  So consecutive
// kernels overlap only their launch and block ramp-up, never their memory
// accesses; the wait always ends, because the predecessor's blocks are all
// resident or done before any dependent block is placed.  After an ordinary
// (not programmatic) predecessor, such as a copy or another library's
// kernel, the launch is serialised as usual.
#pragma once

#include <cuda_runtime.h>

#include <utility>

#include "zero1_internal.h"

namespace zero1 {

__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// kernel<<<grid, block, 0, stream>>>(args...), launched as a programmatic
// dependent of the stream's previous kernel; counted and checked through
// after_launch().
template <typename... Params, typename... Args>
cudaError_t launch(void (*kernel)(Params...), dim3 grid, dim3 block, cudaStream_t stream, Args&&... args) {
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return after_launch(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

}  // namespace zero1

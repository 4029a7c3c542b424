// pdl.cuh -- programmatic dependent launch between the kernels of a stream:
// device-side trigger and wait, and the host-side launch with the attribute.
#pragma once

#include <cuda_runtime.h>

namespace rl {

// A kernel launched with launch_dependent may be scheduled before the kernel
// ahead of it on the stream has finished: once every block of that kernel has
// called pdl_trigger (or exited) the next one is launched, and it waits for its
// predecessor to complete, with that grid's memory operations visible, before
// it touches any of its data (pdl_wait).  Both are no-ops for a kernel launched
// the ordinary way.  Every block of such a kernel calls pdl_wait before it
// returns, so completion stays transitive down the chain.  (Triggering at the
// start of each kernel measured slower than not triggering at all: the early
// blocks hold SM resources while they wait.)
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace rl

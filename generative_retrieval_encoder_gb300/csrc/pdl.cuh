// Programmatic dependent launch.  A kernel launched by launch_pdl may be
// scheduled while the kernel before it in the stream is still running, which
// hides the launch latency between the layer's kernels.  Such a kernel calls
// pdl_wait() before its first access to global memory: it returns once the
// previous kernel has completed and its writes are visible.  pdl_trigger()
// lets the next kernel be scheduled in turn (the next kernel still waits for
// this one's completion in its own pdl_wait()).  Launched without the
// attribute, both are no-ops.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace gbla {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Kernel entry: wait for the previous kernel, then release the next launch.
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_trigger();
}

// The launch attribute that allows the overlap (used alone or with others).
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at.val.programmaticStreamSerializationAllowed = 1;
  return at;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace gbla

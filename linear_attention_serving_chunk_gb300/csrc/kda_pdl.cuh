// Programmatic dependent launch for the two-pass prefill's kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>

namespace kda {

// Programmatic dependent launch: a kernel launched with launch_pdl may be
// launched while the previous kernel on its stream is still running (once
// every CTA of that kernel has called grid_launch_dependents or exited).
// grid_dependency_wait() returns once the previous grids have completed and
// their writes are visible, so each kernel calls it before it touches
// anything earlier work on the stream wrote; what the chain saves is the
// launch latency between the kernels.  Both are no-ops for a kernel launched
// the ordinary way.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace kda

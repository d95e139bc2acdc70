// Programmatic dependent launch: a kernel may start while the one before it in the stream is
// still running (sm_90 and later).
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace spectree {

// ---- programmatic dependent launch -------------------------------------------------------------
// A kernel launched with launch_dependent (below) may start while the kernel before it in the
// stream is still running: it does its independent set-up, then pdl_wait() returns once that
// kernel has completed and its memory writes are visible (a no-op for an ordinary launch).  A
// kernel that calls pdl_launch_dependents() lets its dependent launch as soon as every one of
// its CTAs has made the call (or exited), instead of when the last one exits.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Host: launches `kernel` as a programmatic dependent of the previous kernel in `stream`.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace spectree

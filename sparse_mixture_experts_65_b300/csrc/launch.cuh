// launch.cuh -- programmatic dependent launch (PDL).  Every kernel of the
// layer is launched with programmatic stream serialisation: it may start
// while the previous kernel in the stream is finishing, runs its prologue
// (shared-memory carve-up, barrier set-up, tensor-memory allocation,
// descriptor prefetch), and then waits in griddepcontrol.wait until the
// previous grid has completed and its memory is visible.  Each kernel also
// allows its own dependents to launch early.  A kernel launched this way must
// call pdl_wait() before it touches anything an earlier kernel wrote.
#pragma once

#include <cuda_runtime.h>

namespace moe {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace moe

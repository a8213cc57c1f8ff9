// Kernel launch with programmatic dependent launch (PDL): the next kernel in
// the stream may be scheduled while this one runs; it waits in
// griddepcontrol.wait (pdl_enter) until this grid has completed and its
// writes are visible. Every kernel launched this way must call pdl_enter()
// before it reads or writes memory that an earlier kernel touches.
#pragma once

#include <cuda_runtime.h>

#include <utility>

#include "ptx.cuh"

namespace dfl {

// Let the following grid be scheduled (it can take free SM resources and
// start streaming its weights), then wait for the preceding grid.
__device__ __forceinline__ void pdl_enter() {
  pdl_launch_dependents();
  pdl_wait();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace dfl

// Kernel launch with programmatic dependent launch: the kernel may begin
// while the kernel before it on the stream is still running.  Every kernel
// launched this way calls grid_dep_wait() (ptx.cuh) before it touches memory
// that an earlier kernel writes or reads, and grid_dep_launch() only after
// that wait, so at most the immediately preceding kernel is still running
// when its prologue (barrier set-up, tensor-memory allocation, loads of
// constant weights) executes.
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace moe {

template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
               Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

}  // namespace moe

// Launch as a programmatic dependent of the previous kernel on the stream: the grid may be
// scheduled once every block of that kernel has executed griddepcontrol.launch_dependents (or
// exited), so its blocks are resident when the previous kernel finishes instead of being
// launched then. The kernel must execute griddepcontrol.wait (griddep_wait) before it reads
// anything written earlier in the same stream.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace skv {

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace skv

// launch.cuh -- host-side launch helper: every kernel of the library is
// launched with programmatic stream serialization, so a kernel's CTAs may be
// scheduled while its predecessor drains.  Each kernel executes
// griddepcontrol.wait (dfl::pdl_wait) before it touches anything the
// predecessor writes, and griddepcontrol.launch_dependents once it has
// started; work that depends on nothing upstream (weight prefetch, barrier
// and TMEM set-up) happens before the wait.
#pragma once
#include <cuda_runtime.h>

#include <utility>

#include "trace.h"

namespace dfl {

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  trace_kernel();
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace dfl

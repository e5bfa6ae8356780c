// Kernel launch helper: launches with the programmatic-dependent-launch
// attribute while a PdlScope is active on this host thread (the decode step),
// plainly otherwise.
#pragma once

#include <cuda_runtime.h>

namespace fk {

bool pdl_enabled();

struct PdlScope {
  bool prev;
  explicit PdlScope(bool on);
  ~PdlScope();
};

template <typename... KArgs, typename... Args>
inline cudaError_t fk_launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace fk

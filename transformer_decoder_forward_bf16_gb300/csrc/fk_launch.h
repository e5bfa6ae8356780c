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

// As fk_launch, with thread-block clusters of cluster_x x cluster_y CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t fk_launch_cluster2(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                      unsigned cluster_x, unsigned cluster_y, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = cluster_y;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t fk_launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     unsigned cluster_x, Args... args) {
  return fk_launch_cluster2(kernel, grid, block, smem, st, cluster_x, 1u, args...);
}

}  // namespace fk

// Kernel launch helper: programmatic dependent launch (PDL) and optional thread-block clusters.
//
// Every kernel of the library executes pdl_wait() and then pdl_trigger() (common.cuh): with
// the programmatic-stream-serialization attribute a kernel may be scheduled while its
// predecessor on the stream is still draining; it runs its prologue (barrier setup, TMEM
// allocation, the first weight TMA loads, which read no data produced upstream) and then
// waits in griddepcontrol.wait until the predecessor has completed and its writes are
// visible. Only after that wait does it let its own successor be scheduled, so a kernel's
// pre-wait reads overlap its immediate predecessor alone: every earlier kernel of the chain
// has completed by then. Without the attribute both instructions are no-ops. MXG_PDL=0 in
// the environment turns the attribute off (plain stream order).
#pragma once
#include <cuda_runtime.h>
#include <stdlib.h>

#include <utility>

namespace mxg {

inline bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("MXG_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kc(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, dim3 cluster,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster.x * cluster.y * cluster.z > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster.x;
    attr[n].val.clusterDim.y = cluster.y;
    attr[n].val.clusterDim.z = cluster.z;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Launch with PDL and, when cluster_z > 1, a cluster of cluster_z CTAs along z.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     unsigned cluster_z, Args&&... args) {
  return launch_kc(kernel, grid, block, smem, st, dim3(1, 1, cluster_z), std::forward<Args>(args)...);
}

}  // namespace mxg

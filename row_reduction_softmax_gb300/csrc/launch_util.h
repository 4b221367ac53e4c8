// Host-side launch helper: every kernel of the library is launched with
// programmatic stream serialization (programmatic dependent launch), so a
// launch can be scheduled while the previous kernel on the stream drains.
// Each kernel starts with pdl_entry(): it lets its own dependents launch and
// then waits (griddepcontrol.wait) until the previous grid on the stream has
// completed and its memory is visible, before it touches x or y.  When the
// previous work is not a programmatic launch the wait returns at once.
#pragma once

#include <cuda_runtime.h>

namespace rrs {

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace rrs

// spec_launch.h -- internal: launch helpers and the per-translation-unit launchers.
//
// Every call enqueues two kernels on the caller's stream: stream_kernel<E, MODE> (a plain
// launch) and its finishing kernel, launched with programmatic stream serialization so that it
// may start while the stream kernel drains and waits (griddepcontrol.wait) for its results.
#pragma once

#include <cuda_runtime.h>

#include "spec_device.cuh"

namespace specv {

// Launch shape of the finishing kernel chosen on the host.
struct FinishPlan {
  int grid;        // CTAs
  int cluster;     // CTAs per cluster (1 = no cluster)
  size_t smem;     // dynamic shared memory per CTA
  bool warp_tail;  // chain sampling with single-unit rows: one warp per batch row
};

template <typename Kernel>
inline cudaError_t launch_dependent(Kernel kernel, const Params &p, int grid, int cluster,
                                    size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(na);
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <typename E, int MODE>
inline cudaError_t launch_stream(const Params &p, int grid, cudaStream_t stream) {
  stream_kernel<E, MODE><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

// Launchers: each enqueues the stream kernel and the finishing kernel of its mode for the
// element type named by dtype and returns the first launch error.
cudaError_t launch_chain(int mode, int dtype, const Params &p, int grid, const FinishPlan &f,
                         cudaStream_t stream);
cudaError_t launch_tree(int dtype, const Params &p, int grid, const FinishPlan &f,
                        cudaStream_t stream);
cudaError_t launch_probs(int mode, int dtype, const Params &p, int grid, const FinishPlan &f,
                         cudaStream_t stream);

}  // namespace specv

// spec_launch.h -- internal: launch helpers and the per-translation-unit launchers.
//
// Every call enqueues two kernels on the caller's stream, both with programmatic stream
// serialization: stream_kernel<E, MODE>, then its finishing kernel. Each may be scheduled while
// the kernel ahead of it drains and waits (griddepcontrol.wait) for that kernel's completion
// before touching memory the other could write.
#pragma once

#include <cuda_runtime.h>

#include "spec_device.cuh"

namespace specv {

// Launch shape of the finishing kernel chosen on the host.
// Warps per CTA of the one-warp-per-batch-row chain finisher: small CTAs spread the batch rows
// over every SM, so fewer warps share each scheduler.
constexpr int kTailWarpsPerCta = 4;

struct FinishPlan {
  int grid;        // CTAs
  int cluster;     // CTAs per cluster (1 = no cluster)
  size_t smem;     // dynamic shared memory per CTA
  bool warp_tail;  // chain sampling with single-unit rows: one warp per batch row
  bool sample_warp;  // sampling (gamma = 0) with 16-byte aligned rows: one warp per row
  bool resident;   // one kernel holds every row in registers (no stream kernel)
};

template <typename Kernel>
inline cudaError_t launch_dependent(Kernel kernel, const Params &p, int grid, int cluster,
                                    size_t smem, cudaStream_t stream, int threads = kThreads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
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

// The stream kernel is itself a programmatic dependent of whatever precedes it on the stream:
// its launch may overlap the previous kernel's last CTAs, and it waits (griddepcontrol.wait)
// for that kernel to complete before reading anything.
template <typename E, int MODE>
inline cudaError_t launch_stream(const Params &p, int grid, cudaStream_t stream) {
  return launch_dependent(stream_kernel<E, MODE>, p, grid, 1, 0, stream);
}

// Launchers: each enqueues the stream kernel and the finishing kernel of its mode for the
// element type named by dtype and returns the first launch error.
cudaError_t launch_chain(int mode, int dtype, const Params &p, int grid, const FinishPlan &f,
                         cudaStream_t stream);
cudaError_t launch_tree(int dtype, const Params &p, int grid, const FinishPlan &f,
                        cudaStream_t stream);
// Chain verification fused with its logit producer: the tensor-core LM-head GEMMs with the
// softmax-partial epilogue, then the chain finisher (plan f).
cudaError_t launch_lmhead(const Params &p, const void *hidden_t, const void *head_t, int Kt,
                          const void *hidden_d, const void *head_d, int Kd, void *logits_t,
                          void *logits_d, const FinishPlan &f, cudaStream_t stream);
// Stochastic tree verification: the stream kernel over every target and draft row, then one
// finishing CTA per tree with `smem` bytes of dynamic shared memory.
cudaError_t launch_tree_sample(int dtype, const Params &p, int grid, size_t smem,
                               cudaStream_t stream);
cudaError_t launch_probs(int mode, int dtype, const Params &p, int grid, const FinishPlan &f,
                         cudaStream_t stream);
cudaError_t launch_topk(int dtype, const Params &p, int grid, cudaStream_t stream);
cudaError_t launch_tree_mask(const Params &p, cudaStream_t stream);

}  // namespace specv

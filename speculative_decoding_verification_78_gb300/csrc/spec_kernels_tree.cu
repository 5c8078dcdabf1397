// spec_kernels_tree.cu -- kernel instances for tree verification: greedy, and stochastic (the
// walk by per-sibling rejection sampling).
#include <mutex>

#include "spec_launch.h"

namespace specv {

namespace {

// The walk's finishing kernel needs more than the default 48 KB of shared memory for the largest
// trees and vocabularies. Its dynamic limit is raised only that far, to the largest size a call
// has needed so far on the device (a kernel launched right after one whose limit sat at the
// device maximum failed to launch in a measured experiment, so the limit is kept no higher than
// it must be).
template <typename E>
cudaError_t tree_sample(const Params &p, int grid, size_t smem, cudaStream_t stream) {
  static std::mutex mu;
  static size_t limit[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (smem + sizeof(TsShared) > 48 * 1024) {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 64 || smem > limit[dev]) {
      e = cudaFuncSetAttribute(finish_tree_sample<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      if (dev < 64) limit[dev] = smem;
    }
  }
  e = launch_stream<E, kProbs>(p, grid, stream);
  if (e != cudaSuccess) return e;
  return launch_dependent(finish_tree_sample<E>, p, p.B, 1, smem, stream);
}

template <typename E>
cudaError_t tree(const Params &p, int grid, const FinishPlan &f, cudaStream_t stream) {
  cudaError_t e = launch_stream<E, kTree>(p, grid, stream);
  if (e != cudaSuccess) return e;
  return launch_dependent(finish_cta<E, kTree>, p, f.grid, 1, f.smem, stream);
}

}  // namespace

cudaError_t launch_tree(int dtype, const Params &p, int grid, const FinishPlan &f,
                        cudaStream_t stream) {
  return dtype == SPEC_BF16 ? tree<uint16_t>(p, grid, f, stream) : tree<float>(p, grid, f, stream);
}

cudaError_t launch_tree_sample(int dtype, const Params &p, int grid, size_t smem,
                               cudaStream_t stream) {
  return dtype == SPEC_BF16 ? tree_sample<uint16_t>(p, grid, smem, stream)
                            : tree_sample<float>(p, grid, smem, stream);
}

}  // namespace specv

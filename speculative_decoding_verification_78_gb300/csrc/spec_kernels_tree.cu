// spec_kernels_tree.cu -- kernel instances for greedy tree verification.
#include "spec_launch.h"

namespace specv {

namespace {

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

}  // namespace specv

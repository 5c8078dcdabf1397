// spec_kernels_probs.cu -- kernel instances for the probability helper.
#include "spec_launch.h"

namespace specv {

namespace {

template <typename E, int MODE>
cudaError_t probs(const Params &p, int grid, const FinishPlan &f, cudaStream_t stream) {
  if (f.resident)
    return launch_dependent(probs_resident<E, MODE == kProbsGreedy>, p, f.grid, f.cluster, 0,
                            stream);
  cudaError_t e = launch_stream<E, MODE>(p, grid, stream);
  if (e != cudaSuccess) return e;
  return launch_dependent(finish_probs<E, MODE == kProbsGreedy>, p, f.grid, 1, 0, stream);
}

}  // namespace

cudaError_t launch_probs(int mode, int dtype, const Params &p, int grid, const FinishPlan &f,
                         cudaStream_t stream) {
  if (mode == kProbs)
    return dtype == SPEC_BF16 ? probs<uint16_t, kProbs>(p, grid, f, stream)
                              : probs<float, kProbs>(p, grid, f, stream);
  return dtype == SPEC_BF16 ? probs<uint16_t, kProbsGreedy>(p, grid, f, stream)
                            : probs<float, kProbsGreedy>(p, grid, f, stream);
}

}  // namespace specv

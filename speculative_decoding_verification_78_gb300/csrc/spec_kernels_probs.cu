// spec_kernels_probs.cu -- instances of the verify kernel for the probability helper.
#include "spec_launch.h"

namespace specv {

cudaError_t launch_probs(int mode, int dtype, const Params &p, int grid, size_t smem,
                         cudaStream_t stream) {
  if (mode == kProbs) {
    if (dtype == SPEC_BF16)
      verify_kernel<uint16_t, kProbs><<<grid, kThreads, smem, stream>>>(p);
    else
      verify_kernel<float, kProbs><<<grid, kThreads, smem, stream>>>(p);
  } else {
    if (dtype == SPEC_BF16)
      verify_kernel<uint16_t, kProbsGreedy><<<grid, kThreads, smem, stream>>>(p);
    else
      verify_kernel<float, kProbsGreedy><<<grid, kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace specv

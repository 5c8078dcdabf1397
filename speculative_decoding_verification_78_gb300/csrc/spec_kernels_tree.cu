// spec_kernels_tree.cu -- instances of the verify kernel for greedy tree verification.
#include "spec_launch.h"

namespace specv {

cudaError_t launch_tree(int dtype, const Params &p, int grid, size_t smem, cudaStream_t stream) {
  if (dtype == SPEC_BF16)
    verify_kernel<uint16_t, kTree><<<grid, kThreads, smem, stream>>>(p);
  else
    verify_kernel<float, kTree><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace specv

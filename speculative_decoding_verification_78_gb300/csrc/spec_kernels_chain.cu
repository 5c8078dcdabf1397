// spec_kernels_chain.cu -- instances of the verify kernel for chain verification.
#include "spec_launch.h"

namespace specv {

cudaError_t launch_chain(int mode, int dtype, const Params &p, int grid, size_t smem,
                         cudaStream_t stream) {
  if (mode == kChainSample) {
    if (dtype == SPEC_BF16)
      verify_kernel<uint16_t, kChainSample><<<grid, kThreads, smem, stream>>>(p);
    else
      verify_kernel<float, kChainSample><<<grid, kThreads, smem, stream>>>(p);
  } else {
    if (dtype == SPEC_BF16)
      verify_kernel<uint16_t, kChainGreedy><<<grid, kThreads, smem, stream>>>(p);
    else
      verify_kernel<float, kChainGreedy><<<grid, kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace specv

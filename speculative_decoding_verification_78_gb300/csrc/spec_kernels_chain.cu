// spec_kernels_chain.cu -- kernel instances for chain verification.
#include "spec_launch.h"

namespace specv {

namespace {

template <typename E>
cudaError_t chain_sample(const Params &p, int grid, const FinishPlan &f, cudaStream_t stream) {
  cudaError_t e = launch_stream<E, kChainSample>(p, grid, stream);
  if (e != cudaSuccess) return e;
  if (f.warp_tail)
    return launch_dependent(finish_chain_sample_warp<E>, p, f.grid, 1, 0, stream,
                            32 * kTailWarpsPerCta);
  if (f.sample_warp)
    return launch_dependent(finish_sample_warp<E>, p, f.grid, 1, f.smem, stream,
                            32 * kTailWarpsPerCta);
  return launch_dependent(finish_chain_sample<E>, p, f.grid, f.cluster, f.smem, stream);
}

template <typename E>
cudaError_t chain_greedy(const Params &p, int grid, const FinishPlan &f, cudaStream_t stream) {
  cudaError_t e = launch_stream<E, kChainGreedy>(p, grid, stream);
  if (e != cudaSuccess) return e;
  return launch_dependent(finish_cta<E, kChainGreedy>, p, f.grid, 1, f.smem, stream);
}

}  // namespace

cudaError_t launch_chain(int mode, int dtype, const Params &p, int grid, const FinishPlan &f,
                         cudaStream_t stream) {
  if (mode == kChainSample)
    return dtype == SPEC_BF16 ? chain_sample<uint16_t>(p, grid, f, stream)
                              : chain_sample<float>(p, grid, f, stream);
  return dtype == SPEC_BF16 ? chain_greedy<uint16_t>(p, grid, f, stream)
                            : chain_greedy<float>(p, grid, f, stream);
}

}  // namespace specv

// spec_kernels_next.cu -- kernel instances for the drafter-side helpers: top-n candidates per
// row (stream pass + merge) and the tree-attention mask. (Sampling reuses the chain kernels with
// gamma = 0.)
#include <atomic>

#include "spec_launch.h"

namespace specv {

namespace {

// Raises a kernel's dynamic shared-memory limit once per instance.
template <typename Kernel>
cudaError_t allow_smem(Kernel kernel, size_t bytes, std::atomic<bool> &done) {
  if (done.load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(bytes));
  if (e == cudaSuccess) done.store(true, std::memory_order_release);
  return e;
}

// the merge runs in CTAs of a few warps, so that the rows spread over every SM
template <typename E, int kK>
cudaError_t topk_k(const Params &p, int grid, cudaStream_t stream) {
  const cudaError_t e = launch_dependent(topk_stream_kernel<E, kK>, p, grid, 1, 0, stream);
  if (e != cudaSuccess) return e;
  return launch_dependent(topk_finish<kK>, p, (p.B + kTailWarpsPerCta - 1) / kTailWarpsPerCta, 1,
                          0, stream, 32 * kTailWarpsPerCta);
}

template <typename E>
cudaError_t topk_e(const Params &p, int grid, cudaStream_t stream) {
  if (p.topk <= 1) return topk_k<E, 1>(p, grid, stream);
  if (p.topk <= 2) return topk_k<E, 2>(p, grid, stream);
  if (p.topk <= 4) return topk_k<E, 4>(p, grid, stream);
  if (p.topk <= 8) return topk_k<E, 8>(p, grid, stream);
  return topk_k<E, 16>(p, grid, stream);
}

}  // namespace

cudaError_t launch_topk(int dtype, const Params &p, int grid, cudaStream_t stream) {
  return dtype == SPEC_BF16 ? topk_e<uint16_t>(p, grid, stream) : topk_e<float>(p, grid, stream);
}

cudaError_t launch_tree_mask(const Params &p, cudaStream_t stream) {
  static std::atomic<bool> done{false};
  const size_t max_smem =
      sizeof(int) * SPEC_MAX_NODES + sizeof(uint32_t) * kThreads * kMaskMaxWords;
  const cudaError_t e = allow_smem(tree_mask_kernel<0>, max_smem, done);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(int) * SPEC_MAX_NODES +
                      sizeof(uint32_t) * kThreads * ((static_cast<size_t>(p.N) + 31) / 32);
  return launch_dependent(tree_mask_kernel<0>, p, p.B, 1, smem, stream);
}

}  // namespace specv

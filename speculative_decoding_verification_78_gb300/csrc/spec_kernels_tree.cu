// spec_kernels_tree.cu -- kernel instances for tree verification: greedy, and stochastic (the
// walk by per-sibling rejection sampling).
#include <atomic>
#include <mutex>

#include "spec_launch.h"

namespace specv {

namespace {

// Raises a kernel's dynamic shared-memory limit to `smem` when it needs more than the default,
// only as far as the largest size a call has needed so far on the device: a kernel launched
// right after one whose limit sat at the device maximum failed to launch in a measured
// experiment, so no limit is kept higher than it must be.
template <typename Kernel>
cudaError_t raise_smem(Kernel kernel, size_t smem, size_t static_smem, int dev, std::mutex &mu,
                       size_t (&limit)[64]) {
  if (smem + static_smem <= 48 * 1024) return cudaSuccess;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && smem <= limit[dev]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
  if (e == cudaSuccess && dev < 64) limit[dev] = smem;
  return e;
}

// The stochastic walk's finishing kernel: a cluster of S CTAs per tree, each holding p and q of
// its vocabulary slice in shared memory, when that fits (S from 1 to 8: the most that keeps the
// grid within one CTA per SM, raised further when the slice does not fit otherwise); else one
// CTA per tree reading the rows from L2 on every pass. `smem` is the single-CTA kernel's size.
template <typename E>
cudaError_t tree_sample(const Params &p, int grid, size_t smem, cudaStream_t stream) {
  static std::mutex mu_one, mu_cl;
  static size_t lim_one[64], lim_cl[64];
  static std::atomic<int> optin_of[64], sms_of[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int optin = dev < 64 ? optin_of[dev].load(std::memory_order_acquire) : 0;
  int n_sm = dev < 64 ? sms_of[dev].load(std::memory_order_acquire) : 0;
  if (optin <= 0 || n_sm <= 0) {
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) {
      optin_of[dev].store(optin, std::memory_order_release);
      sms_of[dev].store(n_sm, std::memory_order_release);
    }
  }
  const size_t nseg = static_cast<size_t>((p.V + kSeg - 1) / kSeg);
  const size_t fixed = sizeof(float) * 2 * static_cast<size_t>(p.R) +
                       sizeof(int) * 3 * static_cast<size_t>(p.N);
  const size_t stat_cl = sizeof(TsShared) + sizeof(TsClusterShared);
  auto cl_smem = [&](int S) {
    const size_t nsl = (nseg + S - 1) / S;
    return fixed + sizeof(float) * nsl + 16 + 2 * sizeof(float) * nsl * kSeg;
  };
  int S = 1;
  while (S < kMaxCluster && static_cast<long long>(p.B) * 2 * S <= n_sm) S *= 2;
  while (S < kMaxCluster && cl_smem(S) + stat_cl > static_cast<size_t>(optin)) S *= 2;
  const bool cluster = cl_smem(S) + stat_cl <= static_cast<size_t>(optin);
  if (cluster) {
    e = raise_smem(finish_tree_sample_cluster<E>, cl_smem(S), stat_cl, dev, mu_cl, lim_cl);
  } else {
    e = raise_smem(finish_tree_sample<E>, smem, sizeof(TsShared), dev, mu_one, lim_one);
  }
  if (e != cudaSuccess) return e;
  e = launch_stream<E, kProbs>(p, grid, stream);
  if (e != cudaSuccess) return e;
  if (cluster)
    return launch_dependent(finish_tree_sample_cluster<E>, p, p.B * S, S, cl_smem(S), stream);
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

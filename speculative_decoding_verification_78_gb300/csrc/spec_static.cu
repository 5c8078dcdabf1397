// spec_static.cu -- spec_verify_chain_static: chain verification whose scratch lives in a
// file-scope device array instead of a caller-provided workspace.
//
// Some callers cannot hand the library a workspace: a host process whose device memory is
// entirely owned by another framework's caching allocator, or a per-step decode path that must
// not allocate (an allocation can synchronise the device and fragment memory over a long run).
// For them this entry point uses one statically sized device array, reserved when the library
// is loaded, and never allocates or frees anything itself.
#include <atomic>

#include <cuda_runtime.h>

#include "spec_verify.h"

namespace specv {
int chain_args_check(const void *target_logits, const void *draft_logits, int dtype,
                     const int32_t *draft_tokens, const float *uniforms, int B, int gamma, int V,
                     float temperature, const int32_t *accept_len, const int32_t *out_tokens,
                     const int32_t *status, const void *workspace, bool need_workspace);
int launch_result(cudaError_t e);   // SPEC_ERR_LAUNCH, recording e for spec_last_cuda_error
}  // namespace specv

namespace {

constexpr size_t kStaticScratchBytes = SPEC_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself: the same contents a workspace would hold, none of which needs to start
// at any particular value.
static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

// Its device address, looked up once per device (with that device current) and cached.
std::atomic<void *> g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" int spec_verify_chain_static(const void *target_logits, const void *draft_logits,
                                        int dtype, const int32_t *draft_tokens,
                                        const float *uniforms, int B, int gamma, int V,
                                        float temperature, int32_t *accept_len,
                                        int32_t *out_tokens, int32_t *status, void *stream) {
  // the argument and size checks need no device: bad arguments, and a call larger than the
  // array, are refused up front
  const int chk = specv::chain_args_check(target_logits, draft_logits, dtype, draft_tokens,
                                          uniforms, B, gamma, V, temperature, accept_len,
                                          out_tokens, status, nullptr, false);
  if (chk != SPEC_OK) return chk;
  if (B == 0) return SPEC_OK;
  if (spec_workspace_bytes(B, 2 * gamma + 1, V, dtype) > kStaticScratchBytes)
    return SPEC_ERR_WORKSPACE;
  int dev = -1;
  const cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return specv::launch_result(de);
  if (dev < 0) return SPEC_ERR_LAUNCH;
  // devices beyond the cache table look the address up on every call (same result, slower)
  const bool cached = dev < kMaxDevices;
  void *addr = cached ? g_scratch_addr[dev].load(std::memory_order_acquire) : nullptr;
  if (!addr) {
    const cudaError_t se = cudaGetSymbolAddress(&addr, g_scratch);
    if (se != cudaSuccess) return specv::launch_result(se);
    if (!addr) return SPEC_ERR_LAUNCH;
    if (cached) g_scratch_addr[dev].store(addr, std::memory_order_release);
  }
  return spec_verify_chain(target_logits, draft_logits, dtype, draft_tokens, uniforms, B, gamma,
                           V, temperature, accept_len, out_tokens, status, addr,
                           kStaticScratchBytes, stream);
}

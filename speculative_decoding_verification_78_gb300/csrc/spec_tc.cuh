// spec_tc.cuh -- the tensor-core building blocks of the fused LM-head producer: tensor-map (TMA)
// loads, mbarriers with bounded waits, 5th-generation MMA (tcgen05) with its operands in shared
// memory and its accumulator in tensor memory, and tensor-memory loads.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {
namespace tc {

constexpr unsigned long long kWaitNs = 2000000000ull;   // a bounded wait gives up after 2 s

__device__ __forceinline__ uint32_t saddr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
// the initialised barriers visible to the async proxy (TMA, tcgen05.commit) and the cluster
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::
                   : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits until the phase of parity `parity` has completed, for at most limit_ns; false if it gave
// up. (A fresh barrier is in phase 0, so waiting on parity 1 returns at once.)
static __device__ __noinline__ bool mbar_wait(uint64_t *b, uint32_t parity,
                                              unsigned long long limit_ns = kWaitNs) {
  if (mbar_try(b, parity)) return true;
  const unsigned long long t0 = now_ns();
  while (!mbar_try(b, parity))
    if (now_ns() - t0 > limit_ns) return false;
  return true;
}

// Shared-memory matrix descriptor of a K-major operand tile written by a TMA load with 128-byte
// swizzling: rows of 128 bytes (64 bf16), 8-row atoms of 1024 bytes (the stride between atoms),
// the tile 1024-byte aligned. Fields: start address / 16 (bits 0-13), leading byte offset / 16
// (16-29; not used by this layout), stride byte offset / 16 (32-45), descriptor version 1 (46),
// swizzle mode 2 = 128 bytes (61-63). Advancing K by 16 elements adds 32 bytes (2 units) to the
// start address.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of a dense bf16 x bf16 -> fp32 MMA with both operands K-major: D format
// f32 (bits 4-5 = 1), A and B format bf16 (bits 7-9, 10-12 = 1), N / 8 (bits 17-22), M / 16
// (bits 24-28).
__host__ __device__ constexpr uint32_t bf16_f32_idesc(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// 16 consecutive fp32 columns of this thread's lane (warp w reads lanes 32 (w % 4) .. + 31)
__device__ __forceinline__ void tmem_load16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- CTA pairs (cta_group::2): one MMA over the tensor cores of two SMs of a cluster

// This CTA's rank in its cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of every CTA of the cluster arrive and wait (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// The shared::cluster address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t saddr_local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr_local), "r"(rank));
  return r;
}
// One arrival, with release semantics at cluster scope, on a barrier anywhere in the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_cluster(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], "
      "%2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for a barrier that threads of other CTAs of the cluster arrive on (acquire at cluster
// scope), at most limit_ns; false if it gave up.
static __device__ __noinline__ bool mbar_wait_cluster(uint64_t *b, uint32_t parity,
                                                      unsigned long long limit_ns = kWaitNs) {
  if (mbar_try_cluster(b, parity)) return true;
  const unsigned long long t0 = now_ns();
  while (!mbar_try_cluster(b, parity))
    if (now_ns() - t0 > limit_ns) return false;
  return true;
}
// A 2-D tile of a tensor map into this CTA's shared memory whose completion is counted on a
// barrier of the pair's even CTA (`bar_cluster`: its shared::cluster address, from mapa).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, int c0, int c1,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(saddr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}
// tma_load_2d_pair with an L2 cache-policy hint (a policy from l2_policy_evict_last).
__device__ __forceinline__ void tma_load_2d_pair_hint(void *dst, const CUtensorMap *map, int c0,
                                                      int c1, uint32_t bar_cluster,
                                                      uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(saddr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Tensor memory of a CTA pair: one warp of each of the two CTAs executes these together; both
// CTAs get the same columns of their own SM's tensor memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   saddr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[tmem of both CTAs] (+)= A * B^T over the pair, issued by one thread of the even CTA: A's M
// rows are split between the CTAs (M/2 each, at the same shared-memory offset), B's N rows too
// (N/2 each); each CTA's tensor memory receives its M/2 rows x N columns.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc));
}
// The barrier at `bar`'s offset in every CTA of `cta_mask` receives one arrival once every pair
// MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(saddr(bar)),
      "h"(cta_mask)
      : "memory");
}

}  // namespace tc
}  // namespace specv

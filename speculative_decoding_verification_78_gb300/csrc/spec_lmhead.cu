// spec_lmhead.cu -- chain verification fused with its logit producer: the target's and the
// drafter's LM-head GEMMs (logits = hidden states x head^T, bf16 in, fp32 accumulation) on the
// 5th-generation tensor cores, whose epilogue turns each accumulator tile straight into the
// softmax partials that verification needs, so that no pass reads the logits back to reduce
// them. The speculative-decoding review ("Fast Inference from Transformers via Speculative
// Decoding", pith.science, "The pith") has the target score every drafted position in one
// parallel pass; this is that pass's last layer, with the verify step's first reduction fused in.
//
// Persistent: one CTA per SM walks the output tiles blockIdx.x, blockIdx.x + G, ... (128 rows x
// 256 vocabulary columns each, row tiles fastest so that the CTAs running at one time share
// their head tiles in L2). Warp 0 streams the hidden-state and head tiles of every K block (64
// wide) of every tile through a 4-stage TMA ring (128-byte swizzle) without draining it between
// tiles; warp 1 owns 512 tensor-memory columns, two accumulators, and one of its threads issues
// the MMAs (4 x K=16 per block) of tile i into accumulator i mod 2; warps 2-5 read tile i's
// accumulator (one row per thread) while the MMAs of tile i+1 run in the other one: each fp32
// value is rounded to bf16 (the stored logit), the row's 256 stored values give one (max, sum
// of 2^((l - max) log2(e)/T)) partial, the drafted token's logit is kept when it falls in the
// tile, and the bf16 logits are written out (the finishing kernel re-reads the two rows where
// each step stopped). The finishing kernel is the chain finisher, with 256-column tiles as its
// units.
#include <limits.h>

#include <atomic>

#include <cudaTypedefs.h>

#include "spec_launch.h"
#include "spec_tc.cuh"

namespace specv {

namespace {

constexpr int kLmBM = 128, kLmBN = 256, kLmBK = 64, kLmStages = 4, kLmAcc = 2;
constexpr int kLmABytes = kLmBM * kLmBK * 2;
constexpr int kLmBBytes = kLmBN * kLmBK * 2;
constexpr int kLmStageBytes = kLmABytes + kLmBBytes;
constexpr int kLmEpiWarps = 4;
constexpr int kLmThreads = 32 * (2 + kLmEpiWarps);
constexpr int kLmSmem = kLmStages * kLmStageBytes + 1024;   // + alignment of the ring to 1 KB
constexpr uint32_t kLmTmemCols = kLmAcc * kLmBN;            // 512: all of an SM's tensor memory

struct LmArgs {
  uint16_t *logits_t;   // [Mt, V] bf16 out
  uint16_t *logits_d;   // [Md, V] bf16 out
  int Mt, Md;           // B * (gamma + 1), B * gamma
  int Kt, Kd;           // hidden sizes of the target and of the drafter
  int rt_t, rt;         // row tiles of the target GEMM; of both (the draft's follow)
  int tiles;            // rt * (V / 256)
};

// Tile t: row tile t mod rt (the target's first, then the drafter's), column tile t / rt.
struct LmTile {
  bool draft;
  int m0, M, ctile, KB;
};

__device__ __forceinline__ LmTile lm_tile(const LmArgs &a, int t) {
  LmTile x;
  const int r = t % a.rt;
  x.ctile = t / a.rt;
  x.draft = r >= a.rt_t;
  x.m0 = (x.draft ? r - a.rt_t : r) * kLmBM;
  x.M = x.draft ? a.Md : a.Mt;
  x.KB = (x.draft ? a.Kd : a.Kt) / kLmBK;
  return x;
}

// The epilogue of one accumulator row: thread `row` of the tile (tensor-memory lane q*32+lane).
__device__ __forceinline__ void lm_epilogue_row(const Params &p, const LmArgs &a, const LmTile &x,
                                                uint32_t tacc, int q, int lane) {
  const int j = x.m0 + q * 32 + lane;
  const bool valid = j < x.M;
  const int g1 = p.gamma + 1;
  int b = 0, r = 0, tok = -1;
  if (valid) {
    if (x.draft) {
      b = j / p.gamma;
      const int i = j - b * p.gamma;
      r = g1 + i;
      tok = __ldg(p.tokens + static_cast<long long>(b) * p.gamma + i);
    } else {
      b = j / g1;
      const int i = j - b * g1;
      r = i;
      tok = i < p.gamma ? __ldg(p.tokens + static_cast<long long>(b) * p.gamma + i) : -1;
    }
  }
  const int n0 = x.ctile * kLmBN;
  const float c2 = p.c2;
  uint16_t *out = (x.draft ? a.logits_d : a.logits_t) + static_cast<long long>(j) * p.V + n0;
  float m = -INFINITY, s = 0.f, xval = 0.f;
  bool has_x = false;
#pragma unroll 1
  for (int c = 0; c < kLmBN / 32; ++c) {
    uint32_t v[32];
    tc::tmem_load32(tacc + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c * 32),
                    v);
    // round to the stored bf16 logits; the statistics are taken on those values
    uint32_t h[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[2 * e])));
      const uint32_t hi =
          __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[2 * e + 1])));
      h[e] = lo | (hi << 16);
    }
    if (valid) {
      uint4 *o = reinterpret_cast<uint4 *>(out + c * 32);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        o[t] = make_uint4(h[4 * t], h[4 * t + 1], h[4 * t + 2], h[4 * t + 3]);
    }
    float cm = -INFINITY;
#pragma unroll
    for (int e = 0; e < 16; ++e) cm = fmax_nan(cm, fmax_nan(bf_lo(h[e]), bf_hi(h[e])));
    float cs = 0.f;
    if (cm != -INFINITY) {
      f32x2 acc = pk2(0.f, 0.f);
      const f32x2 m2 = pk2(cm, cm), c22 = pk2(c2, c2);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        acc = add2(acc, ex2_shift2(pk2(bf_lo(h[e]), bf_hi(h[e])), m2, c22));
      float a0, a1;
      up2(acc, a0, a1);
      cs = __fadd_rn(a0, a1);
    }
    stat_merge(m, s, cm, cs, c2);
    const int rel = tok - (n0 + c * 32);
    if (rel >= 0 && rel < 32) {
      uint32_t w = h[0];
#pragma unroll
      for (int e = 1; e < 16; ++e)
        if (e == (rel >> 1)) w = h[e];
      xval = (rel & 1) ? bf_hi(w) : bf_lo(w);
      has_x = true;
    }
  }
  if (valid) {
    const long long row = static_cast<long long>(b) * p.R + r;
    p.ws_part[row * p.C + x.ctile] = make_uint2(__float_as_uint(m), __float_as_uint(s));
    if (has_x) p.ws_xlogit[row] = xval;
  }
}

__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_stats_kernel(const __grid_constant__ CUtensorMap map_ht,
                        const __grid_constant__ CUtensorMap map_wt,
                        const __grid_constant__ CUtensorMap map_hd,
                        const __grid_constant__ CUtensorMap map_wd, Params p, LmArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[kLmStages], empty[kLmStages];
  __shared__ __align__(8) uint64_t acc_full[kLmAcc], acc_empty[kLmAcc], mma_done;
  __shared__ uint32_t tmem_slot;
  // the finishing kernel may be scheduled once every CTA of this grid has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = static_cast<int>(gridDim.x);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kLmStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kLmAcc; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], kLmEpiWarps);
    }
    tc::mbar_init(&mma_done, 1);
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, kLmTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = tmem_slot;
  // launched in stream order, so the kernel ahead has completed: this wait returns at once; it
  // keeps the kernel correct if it is ever launched as a programmatic dependent
  asm volatile("griddepcontrol.wait;" ::: "memory");
  bool timed_out = false;
  if (warp == 0 && lane == 0) {   // producer: TMA loads of every K block of every tile
    int it = 0;   // K blocks issued so far (all tiles)
    for (int t = blockIdx.x; t < a.tiles && !timed_out; t += G) {
      const LmTile x = lm_tile(a, t);
      const CUtensorMap *mh = x.draft ? &map_hd : &map_ht;
      const CUtensorMap *mw = x.draft ? &map_wd : &map_wt;
      for (int kb = 0; kb < x.KB; ++kb, ++it) {
        const int s = it % kLmStages;
        if (!tc::mbar_wait(&empty[s], ((it / kLmStages) & 1) ^ 1)) {
          timed_out = true;
          break;
        }
        uint8_t *st = ring + s * kLmStageBytes;
        tc::mbar_expect_tx(&full[s], kLmStageBytes);
        tc::tma_load_2d(st, mh, kb * kLmBK, x.m0, &full[s]);
        tc::tma_load_2d(st + kLmABytes, mw, kb * kLmBK, x.ctile * kLmBN, &full[s]);
      }
    }
    // no copy may still be landing in shared memory when the CTA exits: only the last load of
    // each stage can be (an earlier one was consumed before the stage was refilled)
    for (int q = it > kLmStages ? it - kLmStages : 0; q < it; ++q)
      if (!tc::mbar_wait(&full[q % kLmStages], (q / kLmStages) & 1)) timed_out = true;
  } else if (warp == 1 && lane == 0) {   // the MMA thread
    constexpr uint32_t idesc = tc::bf16_f32_idesc(kLmBM, kLmBN);
    int it = 0, i = 0;   // K blocks consumed; tiles done
    for (int t = blockIdx.x; t < a.tiles && !timed_out; t += G, ++i) {
      const LmTile x = lm_tile(a, t);
      const int buf = i & 1;
      // the epilogue has read this accumulator's previous tile
      if (!tc::mbar_wait(&acc_empty[buf], ((i >> 1) & 1) ^ 1)) {
        timed_out = true;
        break;
      }
      tc::fence_after_sync();
      const uint32_t d = taddr + static_cast<uint32_t>(buf * kLmBN);
      for (int kb = 0; kb < x.KB; ++kb, ++it) {
        const int s = it % kLmStages;
        if (!tc::mbar_wait(&full[s], (it / kLmStages) & 1)) {
          timed_out = true;
          break;
        }
        tc::fence_after_sync();
        const uint32_t sa = tc::saddr(ring + s * kLmStageBytes);
        const uint64_t ad = tc::sw128_kmajor_desc(sa), bd = tc::sw128_kmajor_desc(sa + kLmABytes);
#pragma unroll
        for (int k = 0; k < kLmBK / 16; ++k)
          tc::mma_bf16(d, ad + static_cast<uint64_t>(2 * k), bd + static_cast<uint64_t>(2 * k),
                       idesc, (kb | k) != 0);
        tc::mma_commit(&empty[s]);   // the stage is free once these MMAs have read it
      }
      if (timed_out) break;
      tc::mma_commit(&acc_full[buf]);   // the tile's accumulator is complete
    }
    // every MMA issued has completed before tensor memory is freed (also after a timeout)
    tc::mma_commit(&mma_done);
    if (!tc::mbar_wait(&mma_done, 0)) timed_out = true;
  } else if (warp >= 2) {   // epilogue: one accumulator row per thread
    const int q = warp & 3;   // this warp's tensor-memory lanes: 32 q .. 32 q + 31
    int i = 0;
    for (int t = blockIdx.x; t < a.tiles; t += G, ++i) {
      const LmTile x = lm_tile(a, t);
      const int buf = i & 1;
      const bool ok = tc::mbar_wait(&acc_full[buf], (i >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        timed_out = true;
        break;
      }
      tc::fence_after_sync();
      lm_epilogue_row(p, a, x, taddr + static_cast<uint32_t>(buf * kLmBN), q, lane);
      // this warp's reads of the accumulator are complete: the MMAs may overwrite it
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
    }
  }
  if (timed_out) set_status(p.status, SPEC_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_free(taddr, kLmTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (!f) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !ptr)
      return nullptr;
    f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    fn.store(f, std::memory_order_release);
  }
  return f;
}

// a [rows, K] bf16 row-major matrix, boxes of box_rows x 64 with 128-byte swizzle
bool make_map(CUtensorMap *m, const void *base, int rows, int K, int box_rows) {
  const auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {kLmBK, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_lmhead(const Params &p, const void *hidden_t, const void *head_t, int Kt,
                          const void *hidden_d, const void *head_d, int Kd, void *logits_t,
                          void *logits_d, const FinishPlan &f, cudaStream_t stream) {
  static std::atomic<int> raised[64];
  static std::atomic<int> sms[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !raised[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(lmhead_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kLmSmem);
    if (e != cudaSuccess) return e;
    if (dev < 64) raised[dev].store(1, std::memory_order_release);
  }
  int n_sm = dev < 64 ? sms[dev].load(std::memory_order_acquire) : 0;
  if (n_sm <= 0) {
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev < 64) sms[dev].store(n_sm, std::memory_order_release);
  }
  const int Mt = p.B * (p.gamma + 1), Md = p.B * p.gamma;
  CUtensorMap mht, mwt, mhd, mwd;
  if (!make_map(&mht, hidden_t, Mt, Kt, kLmBM) || !make_map(&mwt, head_t, p.V, Kt, kLmBN) ||
      !make_map(&mhd, hidden_d, Md, Kd, kLmBM) || !make_map(&mwd, head_d, p.V, Kd, kLmBN))
    return cudaErrorInvalidValue;
  LmArgs a;
  a.logits_t = static_cast<uint16_t *>(logits_t);
  a.logits_d = static_cast<uint16_t *>(logits_d);
  a.Mt = Mt;
  a.Md = Md;
  a.Kt = Kt;
  a.Kd = Kd;
  a.rt_t = (Mt + kLmBM - 1) / kLmBM;
  a.rt = a.rt_t + (Md + kLmBM - 1) / kLmBM;
  const long long tiles = static_cast<long long>(a.rt) * (p.V / kLmBN);
  if (tiles > INT_MAX) return cudaErrorInvalidValue;
  a.tiles = static_cast<int>(tiles);
  // One persistent CTA per SM. A plain stream-ordered launch (not a programmatic dependent of
  // the kernel before it): the GEMM is long, and a 193 KB kernel launched early beside a
  // predecessor whose shared-memory limit had been raised to the device maximum failed to
  // launch in a measured experiment.
  const int grid = a.tiles < n_sm ? a.tiles : n_sm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid < 1 ? 1 : grid), 1, 1);
  cfg.blockDim = dim3(kLmThreads, 1, 1);
  cfg.dynamicSmemBytes = kLmSmem;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  e = cudaLaunchKernelEx(&cfg, lmhead_stats_kernel, mht, mwt, mhd, mwd, p, a);
  if (e != cudaSuccess) return e;
  if (f.warp_tail)
    return launch_dependent(finish_chain_sample_warp<uint16_t>, p, f.grid, 1, 0, stream,
                            32 * kTailWarpsPerCta);
  return launch_dependent(finish_chain_sample<uint16_t>, p, f.grid, f.cluster, f.smem, stream);
}

}  // namespace specv

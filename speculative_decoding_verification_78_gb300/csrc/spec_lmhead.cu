// spec_lmhead.cu -- chain verification fused with its logit producer: the target's and the
// drafter's LM-head GEMMs (logits = hidden states x head^T, bf16 in, fp32 accumulation) on the
// 5th-generation tensor cores, whose epilogue turns each accumulator tile straight into the
// softmax partials that verification needs, so that no pass reads the logits back to reduce
// them. The speculative-decoding review ("Fast Inference from Transformers via Speculative
// Decoding", pith.science, "The pith") has the target score every drafted position in one
// parallel pass; this is that pass's last layer, with the verify step's first reduction fused in.
//
// Persistent CTA pairs. A cluster of two CTAs (on two SMs) walks the output tiles c, c + NC, ...
// (NC clusters), each tile 256 rows x 512 vocabulary columns, row tiles fastest so that the
// clusters running at one time share their head tiles in L2. A tile is two 5th-generation MMAs per
// K step (tcgen05.mma.cta_group::2, M = 256, N = 256, K = 16), one per 256-column half, both on the
// same hidden-state operand: each CTA holds its own 128 hidden-state rows and, of each half, 128 of
// the head's rows in shared memory, so an SM loads 48 KB per 64-wide K block for 128 x 512 outputs
// (a 256-column tile needs 32 KB for half as many). Each K block is one 48 KB stage (three TMA
// boxes, 128-byte swizzle: the hidden-state box and one head box per half) behind one barrier, in a
// ring of four stages that runs across tile boundaries. On GB300 the number of stage barriers per
// byte decides the streaming rate more than the bytes in flight (B = 256, gamma = 8, V = 128256,
// hidden 4096 / 2048, per fused call: about 1740 us like this; 2700 us with the same boxes behind
// one barrier each, fourteen 16 KB slots; 2060 us for 256-column tiles in seven 32 KB stages, 1810
// us in three 64 KB ones). Per CTA: warp 0 issues this CTA's copies; warp 1 allocates all 512
// tensor-memory columns with the other CTA (the two halves' accumulators), and in the even CTA one
// of its threads issues the pair's MMAs once both CTAs' copies of a stage have landed (the odd
// CTA's copies count their bytes on the even CTA's stage barrier); warps 2-9 (one per 32
// tensor-memory lanes and half) first copy their rows of the finished accumulator into registers,
// rounded to bf16 (the stored logits), and hand the tensor memory back to the next tile's MMAs,
// then reduce each row's 256 values of the half to one (max, sum of 2^((l - max) log2(e)/T))
// partial, keep the drafted token's logit when it falls in the half and write the bf16 logits out
// (the finishing kernel re-reads the two rows where each step stopped). The finishing kernel is the
// chain finisher, with 256-column halves as its units.
#include <limits.h>

#include <atomic>

#include <cudaTypedefs.h>

#include "spec_launch.h"
#include "spec_tc.cuh"

namespace specv {

namespace {

constexpr int kLmBM = 128;     // rows of a CTA (the pair's tile: 256)
constexpr int kLmHalf = 256;   // vocabulary columns of one MMA (each CTA loads 128 head rows)
constexpr int kLmBN = 2 * kLmHalf;   // vocabulary columns of a tile
constexpr int kLmBK = 64;       // K of a stage: one TMA box wide (the 128-byte swizzle span)
constexpr int kLmStages = 4;
constexpr int kLmBoxBytes = kLmBM * kLmBK * 2;   // one 128-row box: 16 KB
constexpr int kLmStageBytes = 3 * kLmBoxBytes;   // hidden rows, head half 0, head half 1
constexpr int kLmEpiWarps = 8;
constexpr int kLmThreads = 32 * (2 + kLmEpiWarps);
constexpr int kLmSmem = kLmStages * kLmStageBytes + 1024;   // + alignment of the ring to 1 KB
constexpr uint32_t kLmTmemCols = kLmBN;                   // 512: all of an SM's tensor memory
constexpr uint16_t kLmPairMask = 3;                       // both CTAs of the cluster
static_assert(kLmBM * 2 == kLmHalf, "each CTA loads half of an MMA's head rows");

struct LmArgs {
  uint16_t *logits_t;   // [Mt, V] bf16 out
  uint16_t *logits_d;   // [Md, V] bf16 out
  int Mt, Md;           // B * (gamma + 1), B * gamma
  int Kt, Kd;           // hidden sizes of the target and of the drafter
  int rt_t, rt_d;       // 256-row tiles of the target GEMM and of the drafter's
  int ct;               // 512-column tiles: ceil(V / 512) (the last one may hold one half)
  int tiles_t;          // rt_t * ct: the target's tiles come first
  int tiles;            // (rt_t + rt_d) * ct
  int even;             // drafter tiles a cluster with one target tile fewer takes first (see
                        // lm_sched): Kt / Kd rounded down, 0 when the drafter's K is larger
};

// Tile t: the target GEMM's tiles first, then the drafter's; within each, column tile-major with
// the row tiles fastest. All tiles of one GEMM cost the same (one K), so the clusters walking
// t = c, c + NC, ... stay in step within a GEMM, and the tiles they run at one time are a
// contiguous window: each head tile is read by its row tiles' clusters together, from L2 after
// the first. m0 is this CTA's first row (the pair's tile starts 128 rows earlier in the odd CTA);
// nh is the number of 256-column halves the tile holds (1 for the last tile when V / 256 is odd).
struct LmTile {
  bool draft;
  int m0, M, ctile, nh, KB;
};

__device__ __forceinline__ LmTile lm_tile(const Params &p, const LmArgs &a, int t, int rank) {
  LmTile x;
  x.draft = t >= a.tiles_t;
  const int u = x.draft ? t - a.tiles_t : t;
  const int rt = x.draft ? a.rt_d : a.rt_t;
  x.ctile = u / rt;
  const int r = u - x.ctile * rt;
  x.m0 = r * (2 * kLmBM) + rank * kLmBM;
  x.M = x.draft ? a.Md : a.Mt;
  x.nh = p.C - 2 * x.ctile < 2 ? 1 : 2;
  x.KB = (x.draft ? a.Kd : a.Kt) / kLmBK;   // hidden sizes are multiples of 64
  return x;
}

// The i-th tile of cluster c of NC, or -1 when it has no more. The target's tiles go round robin
// (cluster c takes c, c + NC, ...), so the clusters c >= T mod NC hold one target tile fewer; they
// first take `even` drafter tiles each (round robin among them), which the drafter's shorter K
// makes worth about one target tile, and the remaining drafter tiles go round robin over all
// clusters. Every thread of both CTAs of a cluster computes the same sequence.
__device__ __forceinline__ int lm_sched(const LmArgs &a, int c, int NC, int i) {
  const int T = a.tiles_t, D = a.tiles - a.tiles_t;
  const int h = T % NC;
  const int nT = T / NC + (c < h ? 1 : 0);
  if (i < nT) return c + i * NC;
  i -= nT;
  const int light = NC - h;
  // drafter tiles of the first round (the product in 64 bits: even can be large)
  const int p1 = h > 0 ? static_cast<int>(min(static_cast<long long>(D),
                                              static_cast<long long>(light) * a.even))
                       : 0;
  if (h > 0 && c >= h) {
    const int first = c - h;   // this cluster's first tile of that round
    const int n1 = p1 > first ? (p1 - first + light - 1) / light : 0;
    if (i < n1) return T + first + i * light;
    i -= n1;
  }
  const int j = p1 + c + i * NC;
  return j < D ? T + j : -1;
}

// Chunk C (columns 32 C .. 32 C + 31 of the half, bf16 pairs h[16 C ..]) merged into the row's
// (m, s), in the stream kernel's paired arithmetic; the drafted token's logit kept if it is there.
template <int C>
__device__ __forceinline__ void lm_chunk_stats(const uint32_t (&h)[kLmHalf / 2], int n0, int tok,
                                               float c2, float &m, float &s, float &xval,
                                               bool &has_x) {
  static_assert(C >= 0 && C < kLmHalf / 32, "chunk index");
  float cm = -INFINITY;
#pragma unroll
  for (int e = 0; e < 16; ++e)
    cm = fmax_nan(cm, fmax_nan(bf_lo(h[16 * C + e]), bf_hi(h[16 * C + e])));
  float cs = 0.f;
  if (cm != -INFINITY) {
    f32x2 acc = pk2(0.f, 0.f);
    const f32x2 m2 = pk2(cm, cm), c22 = pk2(c2, c2);
#pragma unroll
    for (int e = 0; e < 16; ++e)
      acc = add2(acc, ex2_shift2(pk2(bf_lo(h[16 * C + e]), bf_hi(h[16 * C + e])), m2, c22));
    float a0, a1;
    up2(acc, a0, a1);
    cs = __fadd_rn(a0, a1);
  }
  stat_merge(m, s, cm, cs, c2);
  const int rel = tok - (n0 + C * 32);
  if (rel >= 0 && rel < 32) {
    // word rel / 2 of the chunk by a tree of selects (a dynamic index would put h in memory)
    const int k = rel >> 1;
    uint32_t t8[8], t4[4], t2[2];
#pragma unroll
    for (int e = 0; e < 8; ++e) t8[e] = (k & 8) ? h[16 * C + 8 + e] : h[16 * C + e];
#pragma unroll
    for (int e = 0; e < 4; ++e) t4[e] = (k & 4) ? t8[4 + e] : t8[e];
#pragma unroll
    for (int e = 0; e < 2; ++e) t2[e] = (k & 2) ? t4[2 + e] : t4[e];
    const uint32_t w = (k & 1) ? t2[1] : t2[0];
    xval = (rel & 1) ? bf_hi(w) : bf_lo(w);
    has_x = true;
  }
}

// The epilogue of one accumulator row of one half: thread `row` of the tile (tensor-memory lane
// q*32+lane), columns hc*256 .. hc*256+255 of the vocabulary (hc: the row's 256-column unit).
// First every value is read from tensor memory and rounded to bf16 (the stored logit, two per
// register); then the warp hands the accumulator back (an arrival on `release`, a barrier of the
// even CTA), and only then reduces and stores, while the next tile's MMAs already run.
__device__ __forceinline__ void lm_epilogue_row(const Params &p, const LmArgs &a, const LmTile &x,
                                                int hc, uint32_t tacc, int q, int lane,
                                                uint32_t release) {
  uint32_t h[kLmHalf / 2];
#pragma unroll
  for (int c = 0; c < kLmHalf / 16; ++c) {
    uint32_t v[16];
    tc::tmem_load16(tacc + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c * 16),
                    v);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const __nv_bfloat162 w =
          __floats2bfloat162_rn(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
      h[8 * c + e] = *reinterpret_cast<const uint32_t *>(&w);
    }
  }
  // this warp's reads of the accumulator are complete: the MMAs may overwrite it
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) tc::mbar_arrive_cluster(release);

  const int j = x.m0 + q * 32 + lane;
  const bool valid = j < x.M && SPEC_CHECK(p, j >= 0 && hc >= 0 && hc < p.C);
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
  const int n0 = hc * kLmHalf;
  const float c2 = p.c2;
  if (valid) {
    uint4 *o = reinterpret_cast<uint4 *>((x.draft ? a.logits_d : a.logits_t) +
                                         static_cast<long long>(j) * p.V + n0);
#pragma unroll
    for (int t = 0; t < kLmHalf / 8; ++t)
      o[t] = make_uint4(h[4 * t], h[4 * t + 1], h[4 * t + 2], h[4 * t + 3]);
  }
  float m = -INFINITY, s = 0.f, xval = 0.f;
  bool has_x = false;
  // the 32-column chunks in order, each index a compile-time constant so that h stays in
  // registers
  lm_chunk_stats<0>(h, n0, tok, c2, m, s, xval, has_x);
  lm_chunk_stats<1>(h, n0, tok, c2, m, s, xval, has_x);
  lm_chunk_stats<2>(h, n0, tok, c2, m, s, xval, has_x);
  lm_chunk_stats<3>(h, n0, tok, c2, m, s, xval, has_x);
  lm_chunk_stats<4>(h, n0, tok, c2, m, s, xval, has_x);
  lm_chunk_stats<5>(h, n0, tok, c2, m, s, xval, has_x);
  lm_chunk_stats<6>(h, n0, tok, c2, m, s, xval, has_x);
  lm_chunk_stats<7>(h, n0, tok, c2, m, s, xval, has_x);
  if (valid && SPEC_CHECK(p, b < p.B && r < p.R)) {
    const long long row = static_cast<long long>(b) * p.R + r;
    p.ws_part[row * p.C + hc] = make_uint2(__float_as_uint(m), __float_as_uint(s));
    if (has_x) p.ws_xlogit[row] = xval;
  }
}

// Ten warps: three share an SM sub-partition's 16 K registers, so at most 168 per thread; the
// epilogue keeps a half row of bf16 logits (128 registers) live
__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_stats_kernel(const __grid_constant__ CUtensorMap map_ht,
                        const __grid_constant__ CUtensorMap map_wt,
                        const __grid_constant__ CUtensorMap map_hd,
                        const __grid_constant__ CUtensorMap map_wd, Params p, LmArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[kLmStages], empty[kLmStages];
  __shared__ __align__(8) uint64_t acc_full, acc_empty, mma_done;
  __shared__ uint32_t tmem_slot;
  // the finishing kernel may be scheduled once every CTA of this grid has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(tc::cluster_rank());
  const bool leader = rank == 0;
  const int NC = static_cast<int>(gridDim.x) / 2, c = static_cast<int>(blockIdx.x) / 2;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kLmStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(&acc_full, 1);
    tc::mbar_init(&acc_empty, 2 * kLmEpiWarps);   // the epilogue warps of both CTAs
    tc::mbar_init(&mma_done, 1);
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc_pair(&tmem_slot, kLmTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  // both CTAs' barriers are initialised and the pair's tensor memory allocated before any
  // thread touches the other CTA
  tc::cluster_sync_all();
  tc::fence_after_sync();
  const uint32_t taddr = tmem_slot;
  // launched in stream order, so the kernel ahead has completed: this wait returns at once; it
  // keeps the kernel correct if it is ever launched as a programmatic dependent
  asm volatile("griddepcontrol.wait;" ::: "memory");
  bool timed_out = false;
  if (warp == 0 && lane == 0) {   // producer: this CTA's boxes of every K block of every tile
    // both CTAs' copies into a stage count their bytes on the even CTA's barrier of that stage,
    // which expects the pair's bytes
    const uint32_t full0 = tc::mapa(tc::saddr(&full[0]), 0);
    // the hidden states are read by every column tile: keep them in L2
    const uint64_t keep = tc::l2_policy_evict_last();
    int it = 0;   // stages filled so far (all tiles)
    for (int i = 0, t; !timed_out && (t = lm_sched(a, c, NC, i)) >= 0; ++i) {
      const LmTile x = lm_tile(p, a, t, rank);
      const CUtensorMap *mh = x.draft ? &map_hd : &map_ht;
      const CUtensorMap *mw = x.draft ? &map_wd : &map_wt;
      const int n0 = x.ctile * kLmBN + rank * kLmBM;
      for (int kb = 0; kb < x.KB; ++kb, ++it) {
        const int s = it % kLmStages;
        if (!tc::mbar_wait(&empty[s], ((it / kLmStages) & 1) ^ 1)) {
          timed_out = true;
          break;
        }
        // the hidden-state box and the head box of each half the tile holds
        if (leader) tc::mbar_expect_tx(&full[s], 2 * (1 + x.nh) * kLmBoxBytes);
        const uint32_t bar = full0 + static_cast<uint32_t>(s * sizeof(uint64_t));
        uint8_t *st = ring + s * kLmStageBytes;
        tc::tma_load_2d_pair_hint(st, mh, kb * kLmBK, x.m0, bar, keep);
        for (int hf = 0; hf < x.nh; ++hf)
          tc::tma_load_2d_pair(st + (1 + hf) * kLmBoxBytes, mw, kb * kLmBK, n0 + hf * kLmHalf,
                               bar);
      }
    }
    // no copy may still be landing in shared memory when either CTA exits. The even CTA waits
    // for the last phase of each stage (the pair's copies); only the last copy of each stage can
    // be in flight (an earlier one was consumed before the stage was refilled). The odd CTA
    // cannot wait on those barriers: it stays until the even CTA has (the final cluster barrier),
    // and after a timeout it also lets any copy it issued past the even CTA's land.
    if (leader) {
      for (int q = it > kLmStages ? it - kLmStages : 0; q < it; ++q)
        if (!tc::mbar_wait(&full[q % kLmStages], (q / kLmStages) & 1)) timed_out = true;
    } else if (timed_out) {
      const unsigned long long t0 = tc::now_ns();
      while (tc::now_ns() - t0 < 100000ull) {
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {   // the pair's MMA thread
    constexpr uint32_t idesc = tc::bf16_f32_idesc(2 * kLmBM, kLmHalf);
    int it = 0, i = 0;   // stages consumed; tiles done
    for (int t; !timed_out && (t = lm_sched(a, c, NC, i)) >= 0; ++i) {
      const LmTile x = lm_tile(p, a, t, rank);
      // both CTAs' epilogues have read the previous tile's accumulators
      if (!tc::mbar_wait_cluster(&acc_empty, (i & 1) ^ 1)) {
        timed_out = true;
        break;
      }
      tc::fence_after_sync();
      for (int kb = 0; kb < x.KB; ++kb, ++it) {
        const int s = it % kLmStages;
        // both CTAs' boxes of the stage have landed
        if (!tc::mbar_wait(&full[s], (it / kLmStages) & 1)) {
          timed_out = true;
          break;
        }
        tc::fence_after_sync();
        const uint32_t sa = tc::saddr(ring + s * kLmStageBytes);
        const uint64_t ad = tc::sw128_kmajor_desc(sa);
        for (int hf = 0; hf < x.nh; ++hf) {
          const uint64_t bd = tc::sw128_kmajor_desc(sa + (1 + hf) * kLmBoxBytes);
          const uint32_t d = taddr + static_cast<uint32_t>(hf * kLmHalf);
#pragma unroll
          for (int k = 0; k < kLmBK / 16; ++k)
            tc::mma_bf16_pair(d, ad + static_cast<uint64_t>(2 * k),
                              bd + static_cast<uint64_t>(2 * k), idesc, (kb | k) != 0);
        }
        // both CTAs' stages are free once these MMAs have read them
        tc::mma_commit_pair(&empty[s], kLmPairMask);
      }
      if (timed_out) break;
      tc::mma_commit_pair(&acc_full, kLmPairMask);   // the tile's accumulators are complete
    }
    // every MMA issued has completed before either CTA frees its tensor memory or exits (also
    // after a timeout)
    tc::mma_commit_pair(&mma_done, kLmPairMask);
    if (!tc::mbar_wait(&mma_done, 0)) timed_out = true;
  } else if (warp == 1 && lane == 0) {
    // odd CTA: the pair's MMAs (which read this CTA's shared memory and write its tensor memory)
    // are complete before it frees its tensor memory or exits
    if (!tc::mbar_wait(&mma_done, 0)) timed_out = true;
  } else if (warp >= 2) {   // epilogue: one accumulator row of one half per thread
    const int q = warp & 3;            // this warp's tensor-memory lanes: 32 q .. 32 q + 31
    const int hf = (warp - 2) >> 2;    // warps 2-5 read the first half, 6-9 the second
    const uint32_t release = tc::mapa(tc::saddr(&acc_empty), 0);
    int i = 0;
    for (int t; (t = lm_sched(a, c, NC, i)) >= 0; ++i) {
      const LmTile x = lm_tile(p, a, t, rank);
      // the arrival is the MMA unit's (a commit from the even CTA); this CTA then reads only its
      // own tensor memory, so a CTA-scope wait suffices (and polls far more cheaply)
      const bool ok = tc::mbar_wait(&acc_full, i & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        timed_out = true;
        break;
      }
      tc::fence_after_sync();
      if (hf < x.nh)
        lm_epilogue_row(p, a, x, 2 * x.ctile + hf, taddr + static_cast<uint32_t>(hf * kLmHalf),
                        q, lane, release);
      else if (lane == 0)   // a tile with one half: nothing to read
        tc::mbar_arrive_cluster(release);
    }
  }
  if (timed_out) set_status(p.status, SPEC_ERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  // neither CTA leaves while the other may still arrive on its barriers
  tc::cluster_sync_all();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_free_pair(taddr, kLmTmemCols);
  }
}

// Self-check of the bounded waits: a cluster of two CTAs whose first threads wait, through the
// same routines the GEMM's roles use, on barriers that nothing ever arrives on (a CTA-scope wait in
// each CTA, then a cluster-scope one in the even CTA). Each wait must give up after limit_ns and
// report SPEC_ERR_TIMEOUT; the kernel then returns normally.
__global__ void __cluster_dims__(2, 1, 1)
    wait_selftest_kernel(int32_t *status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t never[2];
  if (threadIdx.x == 0) {
    tc::mbar_init(&never[0], 1);
    tc::mbar_init(&never[1], 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  tc::cluster_sync_all();
  if (threadIdx.x == 0) {
    if (!tc::mbar_wait(&never[0], 0, limit_ns)) set_status(status, SPEC_ERR_TIMEOUT);
    if (tc::cluster_rank() == 0 && !tc::mbar_wait_cluster(&never[1], 0, limit_ns))
      set_status(status, SPEC_ERR_TIMEOUT);
  }
  __syncthreads();
  tc::cluster_sync_all();
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
  static std::atomic<int> clusters[64];   // co-resident CTA pairs per device (0: not known yet)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int Mt = p.B * (p.gamma + 1), Md = p.B * p.gamma;
  CUtensorMap mht, mwt, mhd, mwd;
  if (!make_map(&mht, hidden_t, Mt, Kt, kLmBM) || !make_map(&mwt, head_t, p.V, Kt, kLmBM) ||
      !make_map(&mhd, hidden_d, Md, Kd, kLmBM) || !make_map(&mwd, head_d, p.V, Kd, kLmBM))
    return cudaErrorInvalidValue;
  LmArgs a;
  a.logits_t = static_cast<uint16_t *>(logits_t);
  a.logits_d = static_cast<uint16_t *>(logits_d);
  a.Mt = Mt;
  a.Md = Md;
  a.Kt = Kt;
  a.Kd = Kd;
  a.rt_t = (Mt + 2 * kLmBM - 1) / (2 * kLmBM);
  a.rt_d = (Md + 2 * kLmBM - 1) / (2 * kLmBM);
  a.ct = (p.C + 1) / 2;
  a.tiles_t = a.rt_t * a.ct;
  const long long tiles = static_cast<long long>(a.rt_t + a.rt_d) * a.ct;
  if (tiles > INT_MAX) return cudaErrorInvalidValue;
  a.tiles = static_cast<int>(tiles);
  a.even = Kd > 0 && Kt >= Kd ? Kt / Kd : 0;

  // Clusters of two CTAs, as many as can be resident at once (a persistent grid must not wait
  // for a slot). A plain stream-ordered launch (not a programmatic dependent of the kernel before
  // it): the GEMM is long, and a 193 KB kernel launched early beside a predecessor whose
  // shared-memory limit had been raised to the device maximum failed to launch in a measured
  // experiment.
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kLmThreads, 1, 1);
  cfg.dynamicSmemBytes = kLmSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int ncl = dev < 64 ? clusters[dev].load(std::memory_order_acquire) : 0;
  if (ncl <= 0) {
    e = cudaFuncSetAttribute(lmhead_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kLmSmem);
    if (e != cudaSuccess) return e;
    int n_sm = 0;
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (n_sm / 2)), 1, 1);
    e = cudaOccupancyMaxActiveClusters(&ncl, lmhead_stats_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (ncl <= 0) return cudaErrorInvalidConfiguration;
    if (dev < 64) clusters[dev].store(ncl, std::memory_order_release);
  }
  const int npair = a.tiles < ncl ? a.tiles : ncl;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (npair < 1 ? 1 : npair)), 1, 1);
  e = cudaLaunchKernelEx(&cfg, lmhead_stats_kernel, mht, mwt, mhd, mwd, p, a);
  if (e != cudaSuccess) return e;
  if (f.warp_tail)
    return launch_dependent(finish_chain_sample_warp<uint16_t>, p, f.grid, 1, 0, stream,
                            32 * kTailWarpsPerCta);
  return launch_dependent(finish_chain_sample<uint16_t>, p, f.grid, f.cluster, f.smem, stream);
}

cudaError_t launch_wait_selftest(int32_t *status, unsigned long long limit_ns,
                                 cudaStream_t stream) {
  wait_selftest_kernel<<<2, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace specv

// spec_helpers.cuh -- the drafter-side kernels: top-n candidates per row and the tree-attention
// mask.
#pragma once

#include "spec_kernels.cuh"

namespace specv {

// ------------------------------------------------------------------ top-n candidates
//
// The k largest logits of each row (value descending, equal values by increasing index), for
// expanding a draft tree. Two kernels, as for verification: the stream pass reduces every unit
// (4 KB of one row, one warp) to that unit's own top k -- each lane keeps a sorted list of its
// kK >= k best (value, index) pairs in registers, then k rounds of a warp maximum over the
// lists' heads -- and writes the k candidates to the workspace; the finishing kernel (one warp
// per row, a programmatic dependent) merges the row's C*k candidates the same way. Exact: every
// element of the row's top k is in its own unit's top k. A NaN or +inf poisons the row.

// (v, i) ranks before (w, j)
__device__ __forceinline__ bool ranks_before(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

template <int kK>
__device__ __forceinline__ void topk_insert(float (&lv)[kK], int (&li)[kK], float v, int i) {
  if (!ranks_before(v, i, lv[kK - 1], li[kK - 1])) return;
  lv[kK - 1] = v;
  li[kK - 1] = i;
#pragma unroll
  for (int j = kK - 1; j > 0; --j) {   // one bubble pass: the rest of the list is sorted
    if (ranks_before(lv[j], li[j], lv[j - 1], li[j - 1])) {
      const float tv = lv[j];
      lv[j] = lv[j - 1];
      lv[j - 1] = tv;
      const int ti = li[j];
      li[j] = li[j - 1];
      li[j - 1] = ti;
    }
  }
}

// k rounds of a warp maximum over the lanes' sorted lists: round r's winner goes to
// (out_v[r], out_i[r]) on lane 0. Lists are consumed. Each round is two redux.sync: the largest
// value (through its order-preserving integer image, -0 folded into +0 so that equal values tie;
// the lists hold no NaN), then the smallest index among the lanes holding it.
template <int kK>
__device__ __forceinline__ void warp_take_topk(float (&lv)[kK], int (&li)[kK], int k, int lane,
                                               uint2 *out) {
  for (int r = 0; r < k; ++r) {
    const unsigned key = float_key(__fadd_rn(lv[0], 0.f));
    const unsigned kmax = __reduce_max_sync(0xffffffffu, key);
    const int i = __reduce_min_sync(0xffffffffu, key == kmax ? li[0] : 0x7fffffff);
    const float v = key_float(kmax);
    if (li[0] == i) {   // indices are unique: exactly the winning lane pops its head
#pragma unroll
      for (int j = 0; j < kK - 1; ++j) { lv[j] = lv[j + 1]; li[j] = li[j + 1]; }
      lv[kK - 1] = -INFINITY;
      li[kK - 1] = 0x7fffffff;
    }
    if (lane == 0) out[r] = make_uint2(__float_as_uint(v), static_cast<uint32_t>(i));
  }
}

// Per unit: if T is the k-th largest of the 32 lanes' maxima, every element of the unit's top k
// is >= T (the k largest lane maxima are k distinct elements, all >= T). The elements >= T --
// usually about k of them -- go to a per-warp candidate buffer in shared memory, ranked there.
// When more than kTopkCand qualify (heavy ties), the unit falls back to sorted per-lane lists.
constexpr int kTopkCand = 64;

// One CTA per SM: up to 128 registers per thread for the per-lane lists. (Two CTAs per SM at
// 64 registers, for k <= 4, measured slower: 19.6 vs 18.9 us for 384 x 32000 bf16, k = 4.)
template <typename E, int kK>
__global__ void __launch_bounds__(kThreads, 1) topk_stream_kernel(Params p) {
  constexpr int kEPV = Elem<E>::kPerVec;
  __shared__ uint2 cbuf[kWarps][kTopkCand];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int W = gridDim.x * kWarps;
  const int k = p.topk;
  uint2 *cand = cbuf[warp];
  // Short lists (k <= 4) leave room for a second unit's registers: the next unit's loads are
  // issued before this unit is ranked, so two units per warp are in flight.
  constexpr bool kAhead = kK <= 4;
  auto fetch = [&](int un, uint4 (&b)[kVPL], float &h, float &t) {
    const UnitId uu = unit_id(p, un);
    const E *rr = static_cast<const E *>(p.tgt) + static_cast<long long>(uu.b) * p.V;
    load_unit<E>(rr, row_geom<E>(rr, p.V), uu.chunk, lane, b, h, t);
  };
  uint4 nbuf[kAhead ? kVPL : 1];
  float neh = -INFINITY, net = -INFINITY;
  if constexpr (kAhead) {
    const int first = blockIdx.x * kWarps + warp;
    if (first < p.units) fetch(first, nbuf, neh, net);
  }
  for (int unit = blockIdx.x * kWarps + warp; unit < p.units; unit += W) {
    const UnitId u = unit_id(p, unit);
    if (!SPEC_CHECK(p, u.b < p.B && u.chunk < p.C)) continue;
    const E *row = static_cast<const E *>(p.tgt) + static_cast<long long>(u.b) * p.V;
    const RowGeom g = row_geom<E>(row, p.V);
    uint4 buf[kVPL];
    float eh, et;
    if constexpr (kAhead) {
#pragma unroll
      for (int j = 0; j < kVPL; ++j) buf[j] = nbuf[j];
      eh = neh;
      et = net;
      if (unit + W < p.units) fetch(unit + W, nbuf, neh, net);
    } else {
      load_unit<E>(row, g, u.chunk, lane, buf, eh, et);
    }
    const bool has_h = u.chunk == 0 && lane < g.h, has_t = u.chunk == 0 && lane < g.tl;
    const int v0 = u.chunk * kUnitVecs + lane;
    // this lane's maximum (NaN-propagating); +inf and NaN poison the row
    float lm = fmax_nan(has_h ? eh : -INFINITY, has_t ? et : -INFINITY);
#pragma unroll
    for (int j = 0; j < kVPL; ++j)
      if (v0 + j * 32 < g.nv) lm = fmax_nan(lm, vec_max<E>(buf[j]));
    const bool any_elem = has_h || has_t || v0 < g.nv;
    const bool bad = (lm != lm) || lm == INFINITY;
    uint2 *out = p.ws_part + static_cast<long long>(unit) * k;
    if (__any_sync(0xffffffffu, bad)) {   // poison the unit: its first candidate NaN
      if (lane == 0) out[0] = make_uint2(0x7fc00000u, 0u);
      continue;
    }
    // T: the k-th largest lane maximum (-inf if fewer lanes hold elements). Each round one
    // redux.sync over the order-preserving integer images (0 for lanes already taken, below
    // every real value) and a ballot that retires the lowest lane holding the maximum.
    float T = -INFINITY;
    {
      bool taken = !any_elem;
      for (int r = 0; r < k; ++r) {
        const unsigned key = taken ? 0u : float_key(__fadd_rn(lm, 0.f));   // -0 -> +0
        const unsigned kmax = __reduce_max_sync(0xffffffffu, key);
        const unsigned holders = __ballot_sync(0xffffffffu, !taken && key == kmax);
        if (holders && lane == __ffs(holders) - 1) taken = true;
        T = holders ? key_float(kmax) : -INFINITY;
      }
    }
    // count, then gather, this lane's elements >= T
    int cnt = 0;
    if (has_h && eh >= T) ++cnt;
    if (has_t && et >= T) ++cnt;
#pragma unroll
    for (int j = 0; j < kVPL; ++j)
      if (v0 + j * 32 < g.nv)
#pragma unroll
        for (int e = 0; e < kEPV; ++e) cnt += (vec_elem<E>(buf[j], e) >= T) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total <= kTopkCand && T != -INFINITY) {
      int pos = incl - cnt;
      auto put = [&](float v, int i) {
        cand[pos++] = make_uint2(__float_as_uint(v), static_cast<uint32_t>(i));
      };
      if (has_h && eh >= T) put(eh, lane);
#pragma unroll
      for (int j = 0; j < kVPL; ++j)
        if (v0 + j * 32 < g.nv)
#pragma unroll
          for (int e = 0; e < kEPV; ++e) {
            const float v = vec_elem<E>(buf[j], e);
            if (v >= T) put(v, g.h + (v0 + j * 32) * kEPV + e);
          }
      if (has_t && et >= T) put(et, g.h + g.nv * kEPV + lane);
      __syncwarp();
      // two candidates per lane, ranked; k rounds of a warp maximum
      float lv[2];
      int li[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c = lane + 32 * q;
        const uint2 w = (c < total) ? cand[c] : make_uint2(0xff800000u, 0x7fffffffu);
        lv[q] = __uint_as_float(w.x);
        li[q] = (c < total) ? static_cast<int>(w.y) : 0x7fffffff;
      }
      if (ranks_before(lv[1], li[1], lv[0], li[0])) {
        const float tv = lv[0]; lv[0] = lv[1]; lv[1] = tv;
        const int ti = li[0]; li[0] = li[1]; li[1] = ti;
      }
      __syncwarp();   // the buffer is reused by this warp's next unit
      warp_take_topk<2>(lv, li, k, lane, out);
      continue;
    }
    // fallback: sorted per-lane lists of kK (value, index) pairs
    float lv[kK];
    int li[kK];
#pragma unroll
    for (int j = 0; j < kK; ++j) { lv[j] = -INFINITY; li[j] = 0x7fffffff; }
    if (has_h) topk_insert<kK>(lv, li, eh, lane);
    if (has_t) topk_insert<kK>(lv, li, et, g.h + g.nv * kEPV + lane);
#pragma unroll
    for (int j = 0; j < kVPL; ++j) {
      const int v = v0 + j * 32;
      if (v < g.nv) {
#pragma unroll
        for (int e = 0; e < kEPV; ++e) topk_insert<kK>(lv, li, vec_elem<E>(buf[j], e), g.h + v * kEPV + e);
      }
    }
    warp_take_topk<kK>(lv, li, k, lane, out);
  }
}

// One warp per row: the row's C*k unit candidates, merged. Launched in small CTAs (any number
// of warps) so that the rows spread over every SM.
template <int kK>
__global__ void __launch_bounds__(kThreads, 1) topk_finish(Params p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int row_i = blockIdx.x * static_cast<int>(blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row_i >= p.B) return;
  const int k = p.topk, n = p.C * k;
  const uint2 *cand = p.ws_part + static_cast<long long>(row_i) * n;
  float lv[kK];
  int li[kK];
#pragma unroll
  for (int j = 0; j < kK; ++j) { lv[j] = -INFINITY; li[j] = 0x7fffffff; }
  bool bad = false;
  for (int c = lane; c < n; c += 32) {
    const uint2 w = ldcg_u2(cand + c);
    const float v = __uint_as_float(w.x);
    if (v != v) bad = true;
    else topk_insert<kK>(lv, li, v, static_cast<int>(w.y));
  }
  __shared__ uint2 sel[kWarps][SPEC_MAX_TOPK];
  uint2 *mine = sel[threadIdx.x >> 5];
  const bool row_bad = __any_sync(0xffffffffu, bad);
  warp_take_topk<kK>(lv, li, k, lane, mine);
  __syncwarp();
  int32_t *out = p.out_tokens + static_cast<long long>(row_i) * k;
  // no element above -inf: no finite value in the row
  const bool invalid = row_bad || __uint_as_float(mine[0].x) == -INFINITY;
  if (invalid && lane == 0) set_status(p.status, SPEC_ERR_NONFINITE);
  for (int r = lane; r < k; r += 32) {
    const int idx = invalid ? -1 : static_cast<int>(mine[r].y);
    if (SPEC_CHECK(p, idx >= -1 && idx < p.V)) out[r] = idx;
  }
}

// ------------------------------------------------------------------ tree-attention mask
//
// Bit j of word j / 32 of row i is set iff node j is node i or one of its ancestors: the mask
// with which every node of a decoding tree attends to its own root path. One CTA per tree; the
// parents go to shared memory and are checked; thread t builds the rows of nodes t, t + 512, ...
// in its own shared-memory row by walking parent pointers, then writes them out.
constexpr int kMaskMaxWords = (SPEC_MAX_NODES + 31) / 32;

// (A template only so that the header can define it in every translation unit.)
template <int kUnused = 0>
__global__ void __launch_bounds__(kThreads, 1) tree_mask_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  int *par = reinterpret_cast<int *>(smem_raw);                          // [N]
  uint32_t *rows = reinterpret_cast<uint32_t *>(par + SPEC_MAX_NODES);   // [kThreads][W]
  __shared__ int bad;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x, tid = threadIdx.x;
  const int N = p.N, W = (N + 31) / 32;
  const long long base = static_cast<long long>(b) * N;
  if (tid == 0) bad = 0;
  __syncthreads();
  for (int i = tid; i < N; i += kThreads) {
    const int q = p.parents[base + i];
    par[i] = q;
    if (i == 0 ? (q != -1) : (q < 0 || q >= i)) atomicOr(&bad, 1);
  }
  __syncthreads();
  uint32_t *out = p.mask_words + base * W;
  if (bad) {
    for (long long q = tid; q < static_cast<long long>(N) * W; q += kThreads) out[q] = 0u;
    if (tid == 0) set_status(p.status, SPEC_ERR_PARENT);
    return;
  }
  uint32_t *mine = rows + tid * W;
  for (int i = tid; i < N; i += kThreads) {
    for (int w = 0; w < W; ++w) mine[w] = 0u;
    for (int j = i; j >= 0; j = par[j]) {   // par[0] = -1 ends it
      if (!SPEC_CHECK(p, j < N && (j >> 5) < W)) break;
      mine[j >> 5] |= 1u << (j & 31);
    }
    for (int w = 0; w < W; ++w) out[static_cast<long long>(i) * W + w] = mine[w];
  }
}

}  // namespace specv

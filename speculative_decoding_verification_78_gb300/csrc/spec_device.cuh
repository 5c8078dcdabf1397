// spec_device.cuh -- device code of the GB300 verify kernels (sm_103a).
//
// One persistent kernel template serves every entry point. The logits of a call are cut into
// work units: one unit = one warp's share of one logits row, 32 lanes x 8 x 16-byte vectors
// (4 KB), read once from HBM with coalesced, L1-bypassing 128-bit loads. A unit reduces to one
// 8-byte partial: (row max, sum of exp2((l - max) * log2(e)/T)) for the softmax statistics, or
// (max value, lowest index) for greedy argmax. CTAs of 16 warps take groups of 16 consecutive
// units (batch-row-major order) from a global counter; the CTA that completes the last unit of
// a batch row (an atomic per-row arrival count) runs that row's tail with all 512 threads:
//
//   chain, T > 0  acceptance test of every draft with one warp ballot, then the correction /
//                 bonus draw as a block-wide prefix scan over the one target (and draft) row
//                 the step stopped at, re-read from L2 right after it was streamed;
//   chain, T = 0  argmax comparison of every draft token, then the greedy correction token;
//   tree          accepted flags and depths of all nodes by pointer jumping, deepest node,
//                 path and bonus token;
//   probs         one write pass of the normalised probabilities of the row.
//
// No CTA ever waits for another: completion is detected with atomics, so any grid size is
// safe. Partials written by other SMs are read with ld.global.cg (L2), never through L1.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "spec_verify.h"

namespace specv {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kVPL = 8;                   // 16-byte vectors per lane in one unit
constexpr int kUnitVecs = 32 * kVPL;      // vectors per unit (4 KB)
constexpr int kSeg = 256;                 // residual segment: 32 lanes x 8 elements
constexpr int kSegIter = 2;               // segments per warp per pass-A iteration

enum Mode : int { kChainSample = 0, kChainGreedy = 1, kTree = 2, kProbs = 3, kProbsGreedy = 4 };

struct Params {
  const void *tgt;           // [B, Rt, V]
  const void *drf;           // [B, Rd, V] (chain sampling only)
  const int32_t *tokens;     // chain: [B, gamma]; tree: [B, N]
  const int32_t *parents;    // tree: [B, N]
  const float *uniforms;     // chain sampling: [B, gamma+1]
  int32_t *accept_len;       // [B]
  int32_t *out_tokens;       // chain: [B, gamma+1]; tree: [B, N]
  int32_t *path_nodes;       // tree: [B, N]
  float *out_probs;          // probs: [B, V]
  int32_t *status;
  unsigned *ws_ctl;          // [0] next group to hand out, [1] CTAs finished
  unsigned *ws_count;        // [B] units finished per batch row
  uint2 *ws_part;            // [B*R*C] one partial per unit
  float *ws_xlogit;          // [B*R] logit at the row's draft token (chain sampling)
  long long units;           // B*R*C
  long long groups;          // ceil(units / kWarps)
  int B, gamma, N, V;
  int Rt, Rd, R, C;          // rows per batch row: target, draft, total; units per row
  float c2;                  // log2(e) / T
};

// ------------------------------------------------------------------ element access

template <typename E> struct Elem;
template <> struct Elem<float> {
  static constexpr int kPerVec = 4;
  static constexpr uint32_t kNegInfWord = 0xff800000u;
};
template <> struct Elem<uint16_t> {   // bf16 bit patterns
  static constexpr int kPerVec = 8;
  static constexpr uint32_t kNegInfWord = 0xff80ff80u;
};

// volatile: the load sits behind a bounds guard and must never be speculated past it
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_vec(const void *p) {   // L1-cached (tail re-reads)
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

template <typename E> __device__ __forceinline__ float ld_elem(const E *p);
template <> __device__ __forceinline__ float ld_elem<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld_elem<uint16_t>(const uint16_t *p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// element e (0..kPerVec-1) of a 16-byte vector, as fp32
template <typename E> __device__ __forceinline__ float vec_elem(const uint4 &v, int e);
template <> __device__ __forceinline__ float vec_elem<float>(const uint4 &v, int e) {
  const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
  return __uint_as_float(w);
}
template <> __device__ __forceinline__ float vec_elem<uint16_t>(const uint4 &v, int e) {
  const int k = e >> 1;
  const uint32_t w = k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
  return (e & 1) ? bf_hi(w) : bf_lo(w);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t y;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
  return y;
}

// exp2((x - m) * c2) with no contraction, so every call site rounds identically
__device__ __forceinline__ float ex2_shift(float x, float m, float c2) {
  return ex2(__fmul_rn(__fsub_rn(x, m), c2));
}

__device__ __forceinline__ uint2 ldcg_u2(const uint2 *p) { return __ldcg(p); }
__device__ __forceinline__ float ldcg_f(const float *p) { return __ldcg(p); }

__device__ __forceinline__ void set_status(int32_t *status, int code) {
  atomicCAS(reinterpret_cast<int *>(status), 0, code);
}

// ------------------------------------------------------------------ row geometry

// A row's 16-byte aligned interior: `h` head elements before it, `nv` full vectors, `tl` tail
// elements after it. Chunk c of the row covers vectors [c*kUnitVecs, (c+1)*kUnitVecs); the
// head and tail elements belong to chunk 0.
struct RowGeom {
  const uint4 *vecs;
  int h, nv, tl;
};

template <typename E>
__device__ __forceinline__ RowGeom row_geom(const E *row, int V) {
  constexpr int kEPV = Elem<E>::kPerVec;
  const unsigned mis = static_cast<unsigned>(reinterpret_cast<uintptr_t>(row) & 15u);
  int h = static_cast<int>(((16u - mis) & 15u) / sizeof(E));
  if (h > V) h = V;
  RowGeom g;
  g.h = h;
  g.nv = (V - h) / kEPV;
  g.tl = V - h - g.nv * kEPV;
  g.vecs = reinterpret_cast<const uint4 *>(row + h);
  return g;
}

template <typename E>
__device__ __forceinline__ const E *row_ptr(const Params &p, long long b, int r) {
  if (r < p.Rt)
    return static_cast<const E *>(p.tgt) + (static_cast<long long>(b) * p.Rt + r) * p.V;
  return static_cast<const E *>(p.drf) + (static_cast<long long>(b) * p.Rd + (r - p.Rt)) * p.V;
}

// Loads one unit into registers: kVPL vectors per lane (out-of-row slots hold -inf), plus the
// row's head/tail scalar for this lane when the unit is chunk 0 (else -inf).
template <typename E>
__device__ __forceinline__ void load_unit(const E *row, const RowGeom &g, int chunk, int lane,
                                          uint4 (&buf)[kVPL], float &ex_head, float &ex_tail) {
  const int v0 = chunk * kUnitVecs + lane;
  const uint32_t ni = Elem<E>::kNegInfWord;
#pragma unroll
  for (int j = 0; j < kVPL; ++j) {
    const int v = v0 + j * 32;
    buf[j] = (v < g.nv) ? ld_stream(g.vecs + v) : make_uint4(ni, ni, ni, ni);
  }
  ex_head = -INFINITY;
  ex_tail = -INFINITY;
  if (chunk == 0) {
    if (lane < g.h) ex_head = ld_elem<E>(row + lane);
    if (lane < g.tl) ex_tail = ld_elem<E>(row + g.h + g.nv * Elem<E>::kPerVec + lane);
  }
}

// NaN-propagating maximum of a lane's unit values.
template <typename E>
__device__ __forceinline__ float unit_lane_max(const uint4 (&buf)[kVPL], float a, float b);

template <>
__device__ __forceinline__ float unit_lane_max<float>(const uint4 (&buf)[kVPL], float a,
                                                      float b) {
  float m = fmax_nan(a, b);
#pragma unroll
  for (int j = 0; j < kVPL; ++j) {
    m = fmax_nan(m, fmax_nan(fmax_nan(__uint_as_float(buf[j].x), __uint_as_float(buf[j].y)),
                             fmax_nan(__uint_as_float(buf[j].z), __uint_as_float(buf[j].w))));
  }
  return m;
}

template <>
__device__ __forceinline__ float unit_lane_max<uint16_t>(const uint4 (&buf)[kVPL], float a,
                                                         float b) {
  uint32_t w[kVPL];
#pragma unroll
  for (int j = 0; j < kVPL; ++j)
    w[j] = bmax2_nan(bmax2_nan(buf[j].x, buf[j].y), bmax2_nan(buf[j].z, buf[j].w));
#pragma unroll
  for (int s = kVPL / 2; s > 0; s >>= 1)
#pragma unroll
    for (int j = 0; j < s; ++j) w[j] = bmax2_nan(w[j], w[j + s]);
  return fmax_nan(fmax_nan(bf_lo(w[0]), bf_hi(w[0])), fmax_nan(a, b));
}

// ------------------------------------------------------------------ softmax statistics

// (m, s) <- (m, s) (+) (m2, s2): the pair for the union of two element sets, where s is the
// sum of exp2((x - m) * c2). An empty set is (-inf, 0). NaN or +inf poison the result.
__device__ __forceinline__ void stat_merge(float &m, float &s, float m2, float s2, float c2) {
  const float M = fmax_nan(m, m2);
  if (M == -INFINITY) {
    m = M;
    s = 0.f;
    return;
  }
  const float a = __fmul_rn(s, ex2_shift(m, M, c2));
  const float b = __fmul_rn(s2, ex2_shift(m2, M, c2));
  m = M;
  s = __fadd_rn(a, b);
}

__device__ __forceinline__ void warp_stat_merge(float &m, float &s, float c2) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    stat_merge(m, s, m2, s2, c2);
  }
}

template <typename E>
__device__ __forceinline__ void unit_stats(const E *row, const RowGeom &g, int chunk, int lane,
                                           float c2, float &m_out, float &s_out) {
  constexpr int kEPV = Elem<E>::kPerVec;
  uint4 buf[kVPL];
  float eh, et;
  load_unit<E>(row, g, chunk, lane, buf, eh, et);
  const float m = unit_lane_max<E>(buf, eh, et);
  float s = 0.f;
  if (m != -INFINITY) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < kVPL; ++j)
#pragma unroll
      for (int e = 0; e < kEPV; ++e)
        acc[e & 3] = __fadd_rn(acc[e & 3], ex2_shift(vec_elem<E>(buf[j], e), m, c2));
    s = __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3]));
    s = __fadd_rn(s, __fadd_rn(ex2_shift(eh, m, c2), ex2_shift(et, m, c2)));
  }
  float mm = m;
  warp_stat_merge(mm, s, c2);
  m_out = mm;
  s_out = s;
}

// ------------------------------------------------------------------ greedy argmax

// (v, i) <- the larger value, the smaller index on equal values. NaN marks a bad row.
__device__ __forceinline__ void arg_merge(float &v, int &i, float v2, int i2) {
  if (v2 != v2 || v != v) {
    v = __int_as_float(0x7fc00000);
    return;
  }
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// Unit argmax: (value, lowest index) over the unit's elements; value NaN when the unit holds
// NaN or +inf; value -inf (index INT_MAX) when it holds no element above -inf.
template <typename E>
__device__ __forceinline__ void unit_argmax(const E *row, const RowGeom &g, int chunk, int lane,
                                            float &v_out, int &i_out) {
  constexpr int kEPV = Elem<E>::kPerVec;
  uint4 buf[kVPL];
  float eh, et;
  load_unit<E>(row, g, chunk, lane, buf, eh, et);
  float wm = unit_lane_max<E>(buf, eh, et);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wm = fmax_nan(wm, __shfl_xor_sync(0xffffffffu, wm, off));
  int idx = 0x7fffffff;
  if (wm != wm || wm == INFINITY) {
    wm = __int_as_float(0x7fc00000);
  } else if (wm != -INFINITY) {
    // smallest index in this lane holding wm: scan from the highest index down
    if (et == wm) idx = g.h + g.nv * kEPV + lane;
    const int v0 = chunk * kUnitVecs + lane;
#pragma unroll
    for (int j = kVPL - 1; j >= 0; --j)
#pragma unroll
      for (int e = kEPV - 1; e >= 0; --e)
        if (vec_elem<E>(buf[j], e) == wm) idx = g.h + (v0 + j * 32) * kEPV + e;
    if (eh == wm) idx = lane;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, off));
  }
  v_out = wm;
  i_out = idx;
}

// ------------------------------------------------------------------ block helpers

struct TailShared {
  int n;
  int err;
  int seg;
  int mode;        // 0 = find the CDF crossing, 1 = take the last positive element
  float base;
  float total;
  float target;
  int token;
  float warp_tot[kWarps];
  float off[kWarps + 1];
  int red_i[kWarps];
};

__device__ __forceinline__ int block_max_int(int v, int *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, off));
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int r = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = max(r, red[w]);
  __syncthreads();
  return r;
}

// ------------------------------------------------------------------ residual / bonus draw

// r(k) for the draw: max(0, p(k) - q(k)) when Q is given, else p(k); every operation rounded
// explicitly so that pass A and pass C produce identical values.
__device__ __forceinline__ float resid(float pt, float qd, bool hasq, float Mt, float iZt,
                                      float Md, float iZd, float c2) {
  const float p = __fmul_rn(ex2_shift(pt, Mt, c2), iZt);
  if (!hasq) return p;
  const float q = __fmul_rn(ex2_shift(qd, Md, c2), iZd);
  return fmaxf(__fsub_rn(p, q), 0.f);
}

// The 8 elements [k0, k0+8) of a row as fp32 (-inf beyond V).
template <typename E>
__device__ __forceinline__ void load8(const E *row, int k0, int V, bool vec_ok, float (&x)[8]) {
  if (vec_ok && k0 + 8 <= V) {
    if constexpr (sizeof(E) == 2) {
      const uint4 v = ld_vec(row + k0);
      x[0] = bf_lo(v.x); x[1] = bf_hi(v.x); x[2] = bf_lo(v.y); x[3] = bf_hi(v.y);
      x[4] = bf_lo(v.z); x[5] = bf_hi(v.z); x[6] = bf_lo(v.w); x[7] = bf_hi(v.w);
    } else {
      const uint4 a = ld_vec(row + k0);
      const uint4 b = ld_vec(row + k0 + 4);
      x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
      x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
      x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
      x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (k0 + e < V) ? ld_elem<E>(row + k0 + e) : -INFINITY;
  }
}

// Inverse-CDF draw over r (see resid) with uniform u: the first k whose running sum strictly
// exceeds u * S. Returns -1 when Q is given and S == 0 (the caller then retries without Q).
// All threads of the CTA call it; the result is returned to every thread.
template <typename E>
__device__ int draw_token(const E *P, const E *Q, float Mt, float iZt, float Md, float iZd,
                          float c2, int V, float u, float *segsum, TailShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool hasq = Q != nullptr;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(P) & 15u) == 0) &&
                      (!hasq || (reinterpret_cast<uintptr_t>(Q) & 15u) == 0);
  const int nseg = (V + kSeg - 1) / kSeg;

  // pass A: per-segment sums of r (each warp takes kSegIter segments per iteration)
  for (int s0 = warp * kSegIter; s0 < nseg; s0 += kWarps * kSegIter) {
    float pt[kSegIter][8], qd[kSegIter][8];
#pragma unroll
    for (int t = 0; t < kSegIter; ++t) {
      const int k0 = (s0 + t) * kSeg + lane * 8;
      load8<E>(P, k0, V, vec_ok, pt[t]);
      if (hasq) load8<E>(Q, k0, V, vec_ok, qd[t]);
      else
#pragma unroll
        for (int e = 0; e < 8; ++e) qd[t][e] = -INFINITY;
    }
#pragma unroll
    for (int t = 0; t < kSegIter; ++t) {
      float ls = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ls = __fadd_rn(ls, resid(pt[t][e], qd[t][e], hasq, Mt, iZt, Md, iZd, c2));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ls = __fadd_rn(ls, __shfl_xor_sync(0xffffffffu, ls, off));
      if (lane == 0 && s0 + t < nseg) segsum[s0 + t] = ls;
    }
  }
  __syncthreads();

  // pass B: exclusive scan of the segment sums over the CTA (fixed association)
  const int K = (nseg + kThreads - 1) / kThreads;
  const int lo = threadIdx.x * K, hi = min(nseg, lo + K);
  float local = 0.f;
  for (int j = lo; j < hi; ++j) local = __fadd_rn(local, segsum[j]);
  float incl_w = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl_w, off);
    if (lane >= off) incl_w = __fadd_rn(incl_w, y);
  }
  if (lane == 31) sh.warp_tot[warp] = incl_w;
  __syncthreads();
  if (threadIdx.x == 0) {
    float o = 0.f;
    sh.off[0] = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      o = __fadd_rn(o, sh.warp_tot[w]);
      sh.off[w + 1] = o;
    }
    sh.total = o;
    sh.target = __fmul_rn(u, o);
    sh.seg = -1;
    sh.mode = 0;
  }
  __syncthreads();
  const float S = sh.total;
  if (hasq && S == 0.f) return -1;    // uniform across the CTA
  const float t_target = sh.target;
  const float up = __shfl_up_sync(0xffffffffu, incl_w, 1);
  const float excl = (lane == 0) ? sh.off[warp] : __fadd_rn(sh.off[warp], up);
  const float incl = __fadd_rn(sh.off[warp], incl_w);
  if (lo < hi && excl <= t_target && t_target < incl) {
    float acc = excl;
    int found = -1, lastpos = -1;
    float lastbase = excl;
    for (int j = lo; j < hi; ++j) {
      const float nxt = __fadd_rn(acc, segsum[j]);
      if (segsum[j] > 0.f) { lastpos = j; lastbase = acc; }
      if (nxt > t_target) { found = j; break; }
      acc = nxt;
    }
    if (found >= 0) { sh.seg = found; sh.base = acc; sh.mode = 0; }
    else { sh.seg = lastpos; sh.base = lastbase; sh.mode = 1; }
  }
  __syncthreads();
  if (sh.seg < 0) {
    // t_target >= S after rounding: the last segment holding mass, its last positive element
    int last = -1;
    for (int j = lo; j < hi; ++j)
      if (segsum[j] > 0.f) last = j;
    last = block_max_int(last, sh.red_i);
    if (threadIdx.x == 0) { sh.seg = last; sh.mode = 1; sh.base = 0.f; }
    __syncthreads();
  }

  // pass C: warp 0 rescans the chosen segment
  if (warp == 0) {
    const int seg = max(sh.seg, 0);   // sh.seg >= 0 whenever S > 0; never index before the row
    const int k0 = seg * kSeg + lane * 8;
    float pt[8], qd[8], r[8];
    load8<E>(P, k0, V, vec_ok, pt);
    if (hasq) load8<E>(Q, k0, V, vec_ok, qd);
    else
#pragma unroll
      for (int e = 0; e < 8; ++e) qd[e] = -INFINITY;
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      r[e] = resid(pt[e], qd[e], hasq, Mt, iZt, Md, iZd, c2);
      ls = __fadd_rn(ls, r[e]);
    }
    int lastpos = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (r[e] > 0.f) lastpos = k0 + e;
    int tok = -1;
    if (sh.mode == 0) {
      float li = ls;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, li, off);
        if (lane >= off) li = __fadd_rn(li, y);
      }
      const float lup = __shfl_up_sync(0xffffffffu, li, 1);
      const float lex = (lane == 0) ? sh.base : __fadd_rn(sh.base, lup);
      const float lin = __fadd_rn(sh.base, li);
      const unsigned cross = __ballot_sync(0xffffffffu, lin > t_target);
      if (cross) {
        const int cl = __ffs(cross) - 1;
        if (lane == cl) {
          float acc = lex;
          for (int e = 0; e < 8; ++e) {
            const float nxt = __fadd_rn(acc, r[e]);
            if (nxt > t_target) { tok = k0 + e; break; }
            acc = nxt;
          }
          if (tok < 0) tok = lastpos;
        }
        tok = __shfl_sync(0xffffffffu, tok, cl);
      }
    }
    if (tok < 0) {
      const unsigned has = __ballot_sync(0xffffffffu, lastpos >= 0);
      const int hl = has ? 31 - __clz(has) : 0;
      tok = __shfl_sync(0xffffffffu, lastpos, hl);
      if (tok < 0) tok = V - 1;   // unreachable when S > 0
    }
    if (lane == 0) sh.token = tok;
  }
  __syncthreads();
  return sh.token;
}

// ------------------------------------------------------------------ tails

template <typename E>
__device__ void fail_chain_row(const Params &p, int b) {
  const int g1 = p.gamma + 1;
  for (int j = threadIdx.x; j < g1; j += kThreads) p.out_tokens[(long long)b * g1 + j] = -1;
  if (threadIdx.x == 0) p.accept_len[b] = -1;
}

template <typename E>
__device__ void tail_chain_sample(const Params &p, int b, float *smem, TailShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = p.R, gamma = p.gamma;
  float *rowM = smem;
  float *rowZ = smem + R;
  float *segsum = smem + 2 * R;
  const float c2 = p.c2;

  // combine the unit partials of every row of this step
  for (int r = warp; r < R; r += kWarps) {
    const uint2 *part = p.ws_part + (static_cast<long long>(b) * R + r) * p.C;
    float m = -INFINITY, s = 0.f;
    for (int c = lane; c < p.C; c += 32) {
      const uint2 v = ldcg_u2(part + c);
      stat_merge(m, s, __uint_as_float(v.x), __uint_as_float(v.y), c2);
    }
    warp_stat_merge(m, s, c2);
    if (lane == 0) { rowM[r] = m; rowZ[r] = s; }
  }
  __syncthreads();

  // acceptance: one lane per draft position, first rejection by ballot
  if (warp == 0) {
    int err = 0;
    for (int r = lane; r < R; r += 32) {
      const float m = rowM[r], z = rowZ[r];
      if (!(isfinite(m) && isfinite(z) && z > 0.f)) err = SPEC_ERR_NONFINITE;
    }
    const int32_t *x = p.tokens + static_cast<long long>(b) * gamma;
    for (int i = lane; i < gamma; i += 32)
      if (x[i] < 0 || x[i] >= p.V) err = err ? err : SPEC_ERR_TOKEN;
    const unsigned any_err = __ballot_sync(0xffffffffu, err != 0);
    int n = gamma;
    if (any_err) {
      err = __shfl_sync(0xffffffffu, err, __ffs(any_err) - 1);
    } else {
      const float *u = p.uniforms + static_cast<long long>(b) * (gamma + 1);
      const float *xl = p.ws_xlogit + static_cast<long long>(b) * R;
      for (int i0 = 0; i0 < gamma; i0 += 32) {
        const int i = i0 + lane;
        bool rej = false;
        if (i < gamma) {
          const int rd = gamma + 1 + i;
          const float lt = ldcg_f(xl + i), ld = ldcg_f(xl + rd);
          // p_i(x)/q_i(x) = 2^(((lt - ld) + (Md - Mt)) * c2) * Zd / Zt
          const float d = __fadd_rn(__fsub_rn(lt, ld), __fsub_rn(rowM[rd], rowM[i]));
          const float ratio = __fmul_rn(ex2(__fmul_rn(d, c2)), __fdiv_rn(rowZ[rd], rowZ[i]));
          rej = !(u[i] <= ratio);
        }
        const unsigned rb = __ballot_sync(0xffffffffu, rej);
        if (rb) { n = i0 + __ffs(rb) - 1; break; }
      }
    }
    if (lane == 0) { sh.n = n; sh.err = err; }
  }
  __syncthreads();
  if (sh.err) {
    if (threadIdx.x == 0) set_status(p.status, sh.err);
    fail_chain_row<E>(p, b);
    return;
  }
  const int n = sh.n;
  const E *P = row_ptr<E>(p, b, n);
  const E *Q = (n < gamma) ? row_ptr<E>(p, b, gamma + 1 + n) : nullptr;
  const float Mt = rowM[n], iZt = __frcp_rn(rowZ[n]);
  const float Md = Q ? rowM[gamma + 1 + n] : 0.f, iZd = Q ? __frcp_rn(rowZ[gamma + 1 + n]) : 0.f;
  const float u = p.uniforms[static_cast<long long>(b) * (gamma + 1) + gamma];
  int tok = draw_token<E>(P, Q, Mt, iZt, Md, iZd, c2, p.V, u, segsum, sh);
  if (tok < 0) tok = draw_token<E>(P, nullptr, Mt, iZt, 0.f, 0.f, c2, p.V, u, segsum, sh);

  const int g1 = gamma + 1;
  int32_t *o = p.out_tokens + static_cast<long long>(b) * g1;
  const int32_t *x = p.tokens + static_cast<long long>(b) * gamma;
  for (int j = threadIdx.x; j < g1; j += kThreads) o[j] = (j < n) ? x[j] : (j == n ? tok : -1);
  if (threadIdx.x == 0) p.accept_len[b] = n;
}

// combine argmax partials of row (b, r) with one warp; returns (value, index) on all lanes
__device__ __forceinline__ void warp_row_argmax(const Params &p, long long b, int r, float &v,
                                                int &i) {
  const int lane = threadIdx.x & 31;
  const uint2 *part = p.ws_part + (b * p.R + r) * p.C;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = lane; c < p.C; c += 32) {
    const uint2 w = ldcg_u2(part + c);
    arg_merge(bv, bi, __uint_as_float(w.x), static_cast<int>(w.y));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, bv, off);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, off);
    arg_merge(bv, bi, v2, i2);
  }
  v = bv;
  i = bi;
}

// argmax of a row is usable when it is finite (no NaN/+inf seen, some element above -inf)
__device__ __forceinline__ bool arg_ok(float v) { return v == v && v != -INFINITY; }

template <typename E>
__device__ void tail_chain_greedy(const Params &p, int b, float *smem, TailShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = p.R, gamma = p.gamma;
  int *g = reinterpret_cast<int *>(smem);
  int *gok = g + R;
  for (int r = warp; r < R; r += kWarps) {
    float v;
    int i;
    warp_row_argmax(p, b, r, v, i);
    if (lane == 0) { g[r] = i; gok[r] = arg_ok(v); }
  }
  __syncthreads();
  if (warp == 0) {
    int err = 0;
    for (int r = lane; r < R; r += 32)
      if (!gok[r]) err = SPEC_ERR_NONFINITE;
    const int32_t *x = p.tokens + static_cast<long long>(b) * gamma;
    for (int i = lane; i < gamma; i += 32)
      if (x[i] < 0 || x[i] >= p.V) err = err ? err : SPEC_ERR_TOKEN;
    const unsigned any_err = __ballot_sync(0xffffffffu, err != 0);
    int n = gamma;
    if (any_err) {
      err = __shfl_sync(0xffffffffu, err, __ffs(any_err) - 1);
    } else {
      for (int i0 = 0; i0 < gamma; i0 += 32) {
        const int i = i0 + lane;
        const bool rej = (i < gamma) && (x[i] != g[i]);
        const unsigned rb = __ballot_sync(0xffffffffu, rej);
        if (rb) { n = i0 + __ffs(rb) - 1; break; }
      }
    }
    if (lane == 0) { sh.n = n; sh.err = err; }
  }
  __syncthreads();
  if (sh.err) {
    if (threadIdx.x == 0) set_status(p.status, sh.err);
    fail_chain_row<E>(p, b);
    return;
  }
  const int n = sh.n, g1 = gamma + 1;
  int32_t *o = p.out_tokens + static_cast<long long>(b) * g1;
  const int32_t *x = p.tokens + static_cast<long long>(b) * gamma;
  for (int j = threadIdx.x; j < g1; j += kThreads) o[j] = (j < n) ? x[j] : (j == n ? g[n] : -1);
  if (threadIdx.x == 0) p.accept_len[b] = n;
}

template <typename E>
__device__ void tail_tree(const Params &p, int b, float *smem, TailShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int N = p.N;
  int *g = reinterpret_cast<int *>(smem);
  int *par = g + N;
  int *tok = par + N;
  int *anc = tok + N;      // [2][N]
  int *acc = anc + 2 * N;  // [2][N]
  int *dep = acc + 2 * N;  // [2][N]
  const long long bN = static_cast<long long>(b) * N;
  if (threadIdx.x == 0) sh.err = 0;
  __syncthreads();
  for (int r = warp; r < N; r += kWarps) {
    float v;
    int i;
    warp_row_argmax(p, b, r, v, i);
    if (lane == 0) {
      g[r] = i;
      if (!arg_ok(v)) atomicCAS(&sh.err, 0, SPEC_ERR_NONFINITE);
    }
  }
  for (int j = threadIdx.x; j < N; j += kThreads) {
    const int pj = p.parents[bN + j];
    const int tj = (j == 0) ? 0 : p.tokens[bN + j];
    par[j] = pj;
    tok[j] = tj;
    if (j == 0 ? (pj != -1) : (pj < 0 || pj >= j)) atomicCAS(&sh.err, 0, SPEC_ERR_PARENT);
    else if (j > 0 && (tj < 0 || tj >= p.V)) atomicCAS(&sh.err, 0, SPEC_ERR_TOKEN);
  }
  __syncthreads();
  const int err = sh.err;
  int32_t *pn = p.path_nodes + bN;
  int32_t *ot = p.out_tokens + bN;
  if (err) {
    for (int j = threadIdx.x; j < N; j += kThreads) { pn[j] = -1; ot[j] = -1; }
    if (threadIdx.x == 0) { set_status(p.status, err); p.accept_len[b] = -1; }
    return;
  }
  // pointer jumping: acc[j] = all matches on the path j .. anc[j] (exclusive); dep[j] = hops
  for (int j = threadIdx.x; j < N; j += kThreads) {
    anc[j] = (j == 0) ? 0 : par[j];
    acc[j] = (j == 0) ? 1 : (tok[j] == g[par[j]]);
    dep[j] = (j == 0) ? 0 : 1;
  }
  __syncthreads();
  int cur = 0;
  for (int span = 1; span < N; span <<= 1) {
    const int nxt = cur ^ 1;
    for (int j = threadIdx.x; j < N; j += kThreads) {
      const int a = anc[cur * N + j];
      anc[nxt * N + j] = anc[cur * N + a];
      acc[nxt * N + j] = acc[cur * N + j] & acc[cur * N + a];
      dep[nxt * N + j] = dep[cur * N + j] + dep[cur * N + a];
    }
    __syncthreads();
    cur = nxt;
  }
  // deepest accepted node, smallest index among equals
  int key = -1;
  for (int j = threadIdx.x; j < N; j += kThreads)
    if (acc[cur * N + j]) key = max(key, (dep[cur * N + j] << 11) | (2047 - j));
  key = block_max_int(key, sh.red_i);
  const int best = 2047 - (key & 2047);
  const int D = key >> 11;
  for (int j = threadIdx.x; j < N; j += kThreads) {
    if (j > D) pn[j] = -1;
    if (j > D) ot[j] = -1;
  }
  if (threadIdx.x == 0) {
    int v = best;
    for (int d = D; d >= 0; --d) {
      pn[d] = v;
      if (d > 0) ot[d - 1] = tok[v];
      v = par[v];
    }
    ot[D] = g[best];
    p.accept_len[b] = D;
  }
}

// probabilities of one row (b = row index): one write pass
template <typename E, bool kGreedy>
__device__ void tail_probs(const Params &p, int b, float *smem, TailShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int V = p.V;
  const float c2 = p.c2;
  if (warp == 0) {
    if (kGreedy) {
      float v;
      int i;
      warp_row_argmax(p, b, 0, v, i);
      if (lane == 0) { sh.err = arg_ok(v) ? 0 : SPEC_ERR_NONFINITE; sh.token = i; }
    } else {
      const uint2 *part = p.ws_part + static_cast<long long>(b) * p.C;
      float m = -INFINITY, s = 0.f;
      for (int c = lane; c < p.C; c += 32) {
        const uint2 v = ldcg_u2(part + c);
        stat_merge(m, s, __uint_as_float(v.x), __uint_as_float(v.y), c2);
      }
      warp_stat_merge(m, s, c2);
      if (lane == 0) {
        sh.err = (isfinite(m) && isfinite(s) && s > 0.f) ? 0 : SPEC_ERR_NONFINITE;
        sh.base = m;
        sh.total = s;
      }
    }
  }
  __syncthreads();
  const int err = sh.err;
  const float M = sh.base, iZ = __frcp_rn(sh.total);
  const int g = sh.token;
  float *out = p.out_probs + static_cast<long long>(b) * V;
  const E *row = static_cast<const E *>(p.tgt) + static_cast<long long>(b) * V;
  if (err && threadIdx.x == 0) set_status(p.status, err);
  // 4-element groups aligned to 16 bytes of the output row
  const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(out) >> 2) & 3u);
  const int h = min(V, (4 - mis) & 3);
  const int ng = (V - h) / 4;
  auto val = [&](int k) -> float {
    if (err) return __int_as_float(0x7fc00000);
    if (kGreedy) return (k == g) ? 1.f : 0.f;
    return __fmul_rn(ex2_shift(ld_elem<E>(row + k), M, c2), iZ);
  };
  for (int k = threadIdx.x; k < h; k += kThreads) out[k] = val(k);
  float4 *o4 = reinterpret_cast<float4 *>(out + h);
  for (int q = threadIdx.x; q < ng; q += kThreads) {
    const int k = h + 4 * q;
    o4[q] = make_float4(val(k), val(k + 1), val(k + 2), val(k + 3));
  }
  for (int k = h + 4 * ng + threadIdx.x; k < V; k += kThreads) out[k] = val(k);
}

// ------------------------------------------------------------------ the kernel

template <typename E, int MODE>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(Params p) {
  extern __shared__ float smem[];
  __shared__ TailShared sh;
  __shared__ int s_tail[kWarps];
  __shared__ int s_ntail;
  __shared__ long long s_group;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long upb = static_cast<long long>(p.R) * p.C;   // units per batch row
  constexpr bool kStats = (MODE == kChainSample || MODE == kProbs);

  long long group = blockIdx.x;
  while (group < p.groups) {
    const long long unit = group * kWarps + warp;
    if (unit < p.units) {
      const long long b = unit / upb;
      const long long rem = unit - b * upb;
      const int r = static_cast<int>(rem / p.C);
      const int chunk = static_cast<int>(rem - static_cast<long long>(r) * p.C);
      const E *row = row_ptr<E>(p, b, r);
      const RowGeom geo = row_geom<E>(row, p.V);
      if constexpr (MODE == kChainSample) {
        // chunk 0 also fetches the logit at this row's draft token (target rows < gamma and
        // every draft row), so the tail does not wait on a scattered load
        if (chunk == 0 && lane == 0 && r != p.gamma) {
          const int i = (r < p.Rt) ? r : r - p.Rt;
          const int x = p.tokens[b * p.gamma + i];
          const float xl = (x >= 0 && x < p.V) ? ld_elem<E>(row + x) : 0.f;
          p.ws_xlogit[b * p.R + r] = xl;
        }
      }
      uint2 part;
      if constexpr (kStats) {
        float m, s;
        unit_stats<E>(row, geo, chunk, lane, p.c2, m, s);
        part = make_uint2(__float_as_uint(m), __float_as_uint(s));
      } else {
        float v;
        int i;
        unit_argmax<E>(row, geo, chunk, lane, v, i);
        part = make_uint2(__float_as_uint(v), static_cast<uint32_t>(i));
      }
      if (lane == 0) p.ws_part[unit] = part;
      __threadfence();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const long long u0 = group * kWarps;
      const long long u1 = min(u0 + kWarps, p.units);
      int nt = 0;
      for (long long b = u0 / upb; b <= (u1 - 1) / upb; ++b) {
        const long long lo = max(u0, b * upb), hi = min(u1, (b + 1) * upb);
        const unsigned add = static_cast<unsigned>(hi - lo);
        const unsigned old = atomicAdd(p.ws_count + b, add);
        if (old + add == static_cast<unsigned>(upb)) s_tail[nt++] = static_cast<int>(b);
      }
      s_ntail = nt;
      __threadfence();
    }
    __syncthreads();
    const int ntail = s_ntail;
    for (int t = 0; t < ntail; ++t) {
      const int b = s_tail[t];
      if constexpr (MODE == kChainSample) tail_chain_sample<E>(p, b, smem, sh);
      else if constexpr (MODE == kChainGreedy) tail_chain_greedy<E>(p, b, smem, sh);
      else if constexpr (MODE == kTree) tail_tree<E>(p, b, smem, sh);
      else if constexpr (MODE == kProbs) tail_probs<E, false>(p, b, smem, sh);
      else tail_probs<E, true>(p, b, smem, sh);
      __syncthreads();
      if (threadIdx.x == 0) p.ws_count[b] = 0;   // leave the workspace zeroed
    }
    if (threadIdx.x == 0) s_group = static_cast<long long>(atomicAdd(p.ws_ctl, 1u)) + gridDim.x;
    __syncthreads();
    group = s_group;
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned done = atomicAdd(p.ws_ctl + 1, 1u);
    if (done == gridDim.x - 1) {
      p.ws_ctl[0] = 0u;
      p.ws_ctl[1] = 0u;
    }
  }
}

}  // namespace specv

// spec_device.cuh -- device code of the GB300 verify kernels (sm_103a).
//
// Each call runs two kernels. The stream kernel cuts the call's logits into units (one warp's
// share of one row: up to 32 lanes x 8 x 16-byte vectors = 4 KB of the row's 16-byte aligned
// interior), reads every unit exactly once with coalesced, L1-bypassing 128-bit loads and
// reduces it to one 8-byte partial: (max, sum of exp2((l - max) * log2(e)/T)) for softmax
// statistics, or (max value, lowest index) for greedy argmax. The finishing kernel, a
// programmatic dependent launch, combines the partials of each batch row and produces the
// outputs:
//
//   chain, T > 0  acceptance of every draft with one warp ballot, then the correction / bonus
//                 draw: an inverse CDF over max(0, p_n - q_n) (or p_gamma) as a prefix scan
//                 over segment sums of the one target and draft row the step stopped at,
//                 re-read from L2 and split over the CTAs of a thread-block cluster;
//   chain, T = 0  argmax comparison of every draft token, then the greedy correction token;
//   tree          accepted flags and depths of all nodes by pointer jumping, deepest node,
//                 path and bonus token;
//   probs         one write pass of the normalised probabilities, unit by unit.
//
// No CTA ever waits for another CTA of its own grid except through the hardware cluster
// barrier. Data written by other CTAs is read with ld.global.cg (L2), never through L1.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "spec_verify.h"

namespace specv {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kVPL = 8;                     // 16-byte vectors per lane in one unit
constexpr int kUnitVecs = 32 * kVPL;        // vectors per unit (4 KB)
constexpr int kSeg = 256;                   // residual segment: 32 lanes x 8 elements
constexpr int kWarpTailMaxV = 2048;         // rows this short get warp-level chain finishing
constexpr int kMaxCluster = 8;              // CTAs per batch row in the chain finisher
template <typename E>
constexpr int kSegIterOf = (sizeof(E) == 2) ? 4 : 2;   // residual segments per warp and pass
constexpr int kRegSegs = 2;   // residual segments a warp keeps in registers for the one-pass draw
static_assert(SPEC_MAX_GAMMA < kThreads, "one draft token per thread");
static_assert(kMaxCluster <= 32, "one cluster rank per lane");

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
  uint2 *ws_part;            // [B*R*C] one partial per unit
  float *ws_xlogit;          // [B*R] logit at the row's draft token (chain sampling)
  int units;                 // B*R*C (< 2^31, checked on the host)
  int upb;                   // units per batch row, R*C
  int B, gamma, N, V;
  int Rt, Rd, R, C;          // rows per batch row: target, draft, total; units per row
  int topk;                  // top-n: candidates per row (1..SPEC_MAX_TOPK)
  uint32_t *mask_words;      // tree mask output: [B, N, ceil(N / 32)] words
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

// 128-bit streaming load that does not allocate in L1 (every logit is read once). volatile:
// the load sits behind a bounds guard and must never be speculated past it.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint4 ld_vec(const void *p) {   // L1-cached (re-reads)
  return __ldg(reinterpret_cast<const uint4 *>(p));
}

template <typename E> __device__ __forceinline__ float ld_elem(const E *p);
template <> __device__ __forceinline__ float ld_elem<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld_elem<uint16_t>(const uint16_t *p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(p)) << 16);
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The same widening, as volatile statements: each use is computed where it stands, so the
// compiler cannot keep dozens of widened copies alive across a reduction to reuse them later.
__device__ __forceinline__ float bf_lo_v(uint32_t w) {
  float f;
  asm volatile("shl.b32 %0, %1, 16;" : "=f"(f) : "r"(w));
  return f;
}
__device__ __forceinline__ float bf_hi_v(uint32_t w) {
  float f;
  asm volatile("and.b32 %0, %1, 0xffff0000;" : "=f"(f) : "r"(w));
  return f;
}

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

// Cluster barrier whose arrival publishes this CTA's earlier shared-memory writes to the other
// CTAs of the cluster (release / acquire), and one that only orders execution: after it no CTA
// still needs a peer's shared memory, so a peer may leave or reuse it.
__device__ __forceinline__ void cluster_sync_publish() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ void cluster_sync_exec() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;"
               ::: "memory");
}

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
__device__ __forceinline__ const E *row_ptr(const Params &p, int b, int r) {
  if (r < p.Rt)
    return static_cast<const E *>(p.tgt) + (static_cast<long long>(b) * p.Rt + r) * p.V;
  return static_cast<const E *>(p.drf) + (static_cast<long long>(b) * p.Rd + (r - p.Rt)) * p.V;
}

struct UnitId {
  int b, r, chunk;
};

// unit -> (batch row, row, chunk), 32-bit unsigned division only
__device__ __forceinline__ UnitId unit_id(const Params &p, int unit) {
  UnitId u;
  const unsigned uu = static_cast<unsigned>(unit);
  u.b = static_cast<int>(uu / static_cast<unsigned>(p.upb));
  const unsigned rem = uu - static_cast<unsigned>(u.b) * static_cast<unsigned>(p.upb);
  u.r = static_cast<int>(rem / static_cast<unsigned>(p.C));
  u.chunk = static_cast<int>(rem - static_cast<unsigned>(u.r) * static_cast<unsigned>(p.C));
  return u;
}

// Loads one span of a row straight into registers: interior vectors vb + j*32 + lane below ve
// (at most kUnitVecs of them; -inf beyond), plus this lane's head/tail scalar when `scalars`.
template <typename E>
__device__ __forceinline__ void load_span(const E *row, const RowGeom &g, int vb, int ve,
                                          bool scalars, int lane, uint4 (&buf)[kVPL],
                                          float &ex_head, float &ex_tail) {
  const int v0 = vb + lane;
  const uint32_t ni = Elem<E>::kNegInfWord;
#pragma unroll
  for (int j = 0; j < kVPL; ++j) {
    const int v = v0 + j * 32;
    buf[j] = (v < ve) ? ld_stream(g.vecs + v) : make_uint4(ni, ni, ni, ni);
  }
  ex_head = -INFINITY;
  ex_tail = -INFINITY;
  if (scalars) {
    if (lane < g.h) ex_head = ld_elem<E>(row + lane);
    if (lane < g.tl) ex_tail = ld_elem<E>(row + g.h + g.nv * Elem<E>::kPerVec + lane);
  }
}

// One unit of the stream kernel: chunk `chunk` of the row (its head/tail scalars with chunk 0).
template <typename E>
__device__ __forceinline__ void load_unit(const E *row, const RowGeom &g, int chunk, int lane,
                                          uint4 (&buf)[kVPL], float &ex_head, float &ex_tail) {
  load_span<E>(row, g, chunk * kUnitVecs, g.nv, chunk == 0, lane, buf, ex_head, ex_tail);
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
__device__ __forceinline__ void unit_stats(const uint4 (&buf)[kVPL], float eh, float et,
                                           float c2, float &m_out, float &s_out) {
  constexpr int kEPV = Elem<E>::kPerVec;
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

// NaN-propagating maximum of one vector.
template <typename E>
__device__ __forceinline__ float vec_max(const uint4 &v) {
  if constexpr (sizeof(E) == 2) {
    const uint32_t w = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
    return fmax_nan(bf_lo(w), bf_hi(w));
  } else {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
}

// Unit argmax: (value, lowest index) over the unit's elements; value NaN when the unit holds
// NaN or +inf; value -inf (index INT_MAX) when it holds no element above -inf. Lanes holding
// the warp maximum locate it through their per-vector maxima: first vector, then element.
template <typename E>
__device__ __forceinline__ void unit_argmax(const uint4 (&buf)[kVPL], float eh, float et,
                                            const RowGeom &g, int vb, int lane, float &v_out,
                                            int &i_out) {
  constexpr int kEPV = Elem<E>::kPerVec;
  float vm[kVPL];
#pragma unroll
  for (int j = 0; j < kVPL; ++j) vm[j] = vec_max<E>(buf[j]);
  float lm = fmax_nan(eh, et);
#pragma unroll
  for (int j = 0; j < kVPL; ++j) lm = fmax_nan(lm, vm[j]);
  float wm = lm;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wm = fmax_nan(wm, __shfl_xor_sync(0xffffffffu, wm, off));
  int idx = 0x7fffffff;
  if (wm != wm || wm == INFINITY) {
    wm = __int_as_float(0x7fc00000);
  } else if (wm != -INFINITY) {
    if (lm == wm) {
      if (eh == wm) {
        idx = lane;                                   // head elements precede every vector
      } else {
        int js = kVPL;
#pragma unroll
        for (int j = kVPL - 1; j >= 0; --j)
          if (vm[j] == wm) js = j;
        if (js < kVPL) {
          uint4 t = buf[0];
#pragma unroll
          for (int j = 1; j < kVPL; ++j)
            if (j == js) t = buf[j];
          int e0 = kEPV - 1;
#pragma unroll
          for (int e = kEPV - 1; e >= 0; --e)
            if (vec_elem<E>(t, e) == wm) e0 = e;
          idx = g.h + (vb + js * 32 + lane) * kEPV + e0;
        } else {
          idx = g.h + g.nv * kEPV + lane;             // the tail element
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) idx = min(idx, __shfl_xor_sync(0xffffffffu, idx, off));
  }
  v_out = wm;
  i_out = idx;
}

// The logit at token x (0 <= x < V) if the span [vb, ve) of interior vectors (or, with
// `scalars`, the row's head/tail elements) holds it: taken from the register of the lane that
// loaded it (a shuffle), or re-read for a head/tail element. Returns whether this span holds x
// (the same on every lane); *val is valid on lane 0.
template <typename E>
__device__ __forceinline__ bool span_logit(const E *row, const RowGeom &g, int vb, int ve,
                                           bool scalars, int x, int lane,
                                           const uint4 (&buf)[kVPL], float *val) {
  constexpr int kEPV = Elem<E>::kPerVec;
  const int rel = x - g.h;
  const int vx = rel >= 0 ? rel / kEPV : -1;
  if (rel >= 0 && vx < g.nv) {
    if (vx < vb || vx >= ve) return false;
    // slot (vx - vb) = j*32 + owner lane: pick vector j, then element e
    const int js = (vx - vb) >> 5, owner = (vx - vb) & 31, e = rel - vx * kEPV;
    uint4 t = buf[0];
#pragma unroll
    for (int j = 1; j < kVPL; ++j)
      if (j == js) t = buf[j];
    *val = __shfl_sync(0xffffffffu, vec_elem<E>(t, e), owner);
    return true;
  }
  if (!scalars) return false;
  if (lane == 0) *val = ld_elem<E>(row + x);
  return true;
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
// explicitly so that every pass produces identical values.
__device__ __forceinline__ float resid(float pt, float qd, bool hasq, float Mt, float iZt,
                                      float Md, float iZd, float c2) {
  const float p = __fmul_rn(ex2_shift(pt, Mt, c2), iZt);
  if (!hasq) return p;
  const float q = __fmul_rn(ex2_shift(qd, Md, c2), iZd);
  return fmaxf(__fsub_rn(p, q), 0.f);
}

// The 8 elements [k0, k0+8) of a row, still encoded (bf16: w[0] holds 8 halves; fp32: w[0],
// w[1] hold 4 words each); -inf beyond V.
template <typename E>
__device__ __forceinline__ void load8_raw(const E *row, int k0, int V, bool vec_ok,
                                          uint4 (&w)[2]) {
  if (vec_ok && k0 + 8 <= V) {
    w[0] = ld_vec(row + k0);
    if constexpr (sizeof(E) == 4) w[1] = ld_vec(row + k0 + 4);
  } else {
    uint32_t h[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if constexpr (sizeof(E) == 2)
        h[e] = (k0 + e < V) ? static_cast<uint32_t>(__ldg(row + k0 + e)) : 0xff80u;
      else
        h[e] = (k0 + e < V) ? __float_as_uint(__ldg(row + k0 + e)) : 0xff800000u;
    }
    if constexpr (sizeof(E) == 2) {
      w[0] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                        h[6] | (h[7] << 16));
    } else {
      w[0] = make_uint4(h[0], h[1], h[2], h[3]);
      w[1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

template <typename E>
__device__ __forceinline__ float raw8_elem(const uint4 (&w)[2], int e) {
  if constexpr (sizeof(E) == 2) return vec_elem<uint16_t>(w[0], e);
  else return vec_elem<float>(e < 4 ? w[0] : w[1], e & 3);
}

// Segment sum over this lane's 8 elements of segment `seg` (sequential), and the 8 values.
template <typename E>
__device__ __forceinline__ float lane_resid(const E *P, const E *Q, int seg, int lane, int V,
                                            bool vec_ok, float Mt, float iZt, float Md,
                                            float iZd, float c2, float (&r)[8]) {
  const int k0 = seg * kSeg + lane * 8;
  uint4 wp[2], wq[2];
  load8_raw<E>(P, k0, V, vec_ok, wp);
  if (Q) load8_raw<E>(Q, k0, V, vec_ok, wq);
  float ls = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    r[e] = resid(raw8_elem<E>(wp, e), Q ? raw8_elem<E>(wq, e) : -INFINITY, Q != nullptr, Mt,
                 iZt, Md, iZd, c2);
    ls = __fadd_rn(ls, r[e]);
  }
  return ls;
}

// Within one segment whose exclusive prefix is `base`: the first element whose running sum
// strictly exceeds t, or (mode 1 / no crossing) the last element with r > 0. One warp; the
// token is returned to every lane.
__device__ __forceinline__ int segment_pick(const float (&r)[8], float ls, int k0, float base,
                                            float t, int mode, int lane) {
  int lastpos = -1;
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (r[e] > 0.f) lastpos = k0 + e;
  int tok = -1;
  if (mode == 0) {
    float li = ls;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, li, off);
      if (lane >= off) li = __fadd_rn(li, y);
    }
    const float lup = __shfl_up_sync(0xffffffffu, li, 1);
    const float lex = (lane == 0) ? base : __fadd_rn(base, lup);
    const float lin = __fadd_rn(base, li);
    const unsigned cross = __ballot_sync(0xffffffffu, lin > t);
    if (cross) {
      const int cl = __ffs(cross) - 1;
      if (lane == cl) {
        float acc = lex;
        for (int e = 0; e < 8; ++e) {
          const float nxt = __fadd_rn(acc, r[e]);
          if (nxt > t) { tok = k0 + e; break; }
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
  }
  return tok;
}

// Pass A of the CTA-wide draw: the sum of r over each segment in [lo, hi) (kSeg elements,
// 8 per lane, sequential within a lane, then a fixed xor tree over the warp) into
// out[seg - out_base]. Each warp takes kSegIter segments per iteration with all their loads
// in flight together.
template <typename E>
__device__ __noinline__ void segment_sums(const E *P, const E *Q, float Mt, float iZt, float Md, float iZd,
                             float c2, int V, int lo, int hi, float *out, int out_base) {
  constexpr int kSegIter = kSegIterOf<E>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(P) & 15u) == 0) &&
                      (!Q || (reinterpret_cast<uintptr_t>(Q) & 15u) == 0);
  for (int s0 = lo + warp * kSegIter; s0 < hi; s0 += kWarps * kSegIter) {
    uint4 wp[kSegIter][2], wq[kSegIter][2];
#pragma unroll
    for (int t = 0; t < kSegIter; ++t) {
      const int k0 = (s0 + t < hi) ? (s0 + t) * kSeg + lane * 8 : V;
      load8_raw<E>(P, k0, V, vec_ok, wp[t]);
      if (Q) load8_raw<E>(Q, k0, V, vec_ok, wq[t]);
    }
#pragma unroll
    for (int t = 0; t < kSegIter; ++t) {
      float ls = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        ls = __fadd_rn(ls, resid(raw8_elem<E>(wp[t], e), Q ? raw8_elem<E>(wq[t], e) : -INFINITY,
                                 Q != nullptr, Mt, iZt, Md, iZd, c2));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ls = __fadd_rn(ls, __shfl_xor_sync(0xffffffffu, ls, off));
      if (lane == 0 && s0 + t < hi) out[s0 + t - out_base] = ls;
    }
  }
}

// Passes B and C of the draw within one vocabulary slice [lo*kSeg, (lo+nl)*kSeg): segsum[0..nl)
// holds the slice's segment sums (shared memory), `base` the running sum before the slice and
// `t` the target u*S. An exclusive scan of the segment sums (fixed association) finds the
// segment where the running sum first exceeds t; warp 0 rescans it. mode 0: that element (or,
// if rounding leaves no crossing in the slice, the slice's last element with r > 0); mode 1:
// the last element with r > 0. All threads call it; every thread gets the token.
template <typename E>
__device__ __noinline__ int pick_in_slice(const E *P, const E *Q, float Mt, float iZt, float Md, float iZd,
                             float c2, int V, const float *segsum, int nl, int lo, float base,
                             float t, int mode, TailShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(P) & 15u) == 0) &&
                      (!Q || (reinterpret_cast<uintptr_t>(Q) & 15u) == 0);
  const int K = (nl + kThreads - 1) / kThreads;
  const int tl = threadIdx.x * K, th = min(nl, tl + K);
  float local = 0.f;
  for (int j = tl; j < th; ++j) local = __fadd_rn(local, segsum[j]);
  float incl_w = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl_w, off);
    if (lane >= off) incl_w = __fadd_rn(incl_w, y);
  }
  if (lane == 31) sh.warp_tot[warp] = incl_w;
  __syncthreads();
  if (warp == 0) {   // warp offsets: base + inclusive scan of the warp totals
    float v = (lane < kWarps) ? sh.warp_tot[lane] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v = __fadd_rn(v, y);
    }
    if (lane < kWarps) sh.off[lane + 1] = __fadd_rn(base, v);
    if (lane == 0) {
      sh.off[0] = base;
      sh.seg = -1;
      sh.mode = mode;
      sh.base = base;
    }
  }
  __syncthreads();
  if (mode == 0) {
    const float up = __shfl_up_sync(0xffffffffu, incl_w, 1);
    const float excl = (lane == 0) ? sh.off[warp] : __fadd_rn(sh.off[warp], up);
    const float incl = __fadd_rn(sh.off[warp], incl_w);
    if (tl < th && excl <= t && t < incl) {
      float acc = excl;
      int found = -1, lastpos = -1;
      float lastbase = excl;
      for (int j = tl; j < th; ++j) {
        const float nxt = __fadd_rn(acc, segsum[j]);
        if (segsum[j] > 0.f) { lastpos = j; lastbase = acc; }
        if (nxt > t) { found = j; break; }
        acc = nxt;
      }
      if (found >= 0) { sh.seg = found; sh.base = acc; sh.mode = 0; }
      else { sh.seg = lastpos; sh.base = lastbase; sh.mode = 1; }
    }
  }
  __syncthreads();
  if (sh.seg < 0) {
    int last = -1;
    for (int j = tl; j < th; ++j)
      if (segsum[j] > 0.f) last = j;
    last = block_max_int(last, sh.red_i);
    if (threadIdx.x == 0) { sh.seg = last; sh.mode = 1; }
    __syncthreads();
  }
  if (warp == 0) {
    const int seg = lo + max(sh.seg, 0);   // never index before the slice
    float r[8];
    const float ls = lane_resid<E>(P, Q, seg, lane, V, vec_ok, Mt, iZt, Md, iZd, c2, r);
    int tok = segment_pick(r, ls, seg * kSeg + lane * 8, sh.base, t, sh.mode, lane);
    if (tok < 0) tok = V - 1;   // unreachable when the slice holds mass
    if (lane == 0) sh.token = tok;
  }
  __syncthreads();
  return sh.token;
}

// CTA-wide inverse-CDF draw over the whole row: the first k whose running sum strictly exceeds
// u * S. Returns -1 when Q is given and S == 0. segsum: shared memory, ceil(V/kSeg) floats.
template <typename E>
__device__ __noinline__ int draw_token_cta(const E *P, const E *Q, float Mt, float iZt, float Md, float iZd,
                              float c2, int V, float u, float *segsum, TailShared &sh) {
  const int nseg = (V + kSeg - 1) / kSeg;
  segment_sums<E>(P, Q, Mt, iZt, Md, iZd, c2, V, 0, nseg, segsum, 0);
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int j = 0; j < nseg; ++j) tot = __fadd_rn(tot, segsum[j]);
    sh.total = tot;
  }
  __syncthreads();
  const float S = sh.total;
  if (Q && S == 0.f) return -1;
  const float t = __fmul_rn(u, S);
  // t >= S after rounding leaves no crossing: pick_in_slice then takes the last r > 0
  return pick_in_slice<E>(P, Q, Mt, iZt, Md, iZd, c2, V, segsum, nseg, 0, 0.f, t,
                          t < S ? 0 : 1, sh);
}

// Warp-wide draw for rows of at most kWarpTailMaxV elements (<= 8 segments). The loads of
// several segments are issued together (four at a time for bf16, two for fp32); for rows of at
// most four segments the residual values stay in registers, so the crossing element is found
// without reading the rows again.
template <typename E>
__device__ int draw_token_warp(const E *P, const E *Q, float Mt, float iZt, float Md, float iZd,
                               float c2, int V, float u) {
  constexpr int kMaxSeg = kWarpTailMaxV / kSeg;
  constexpr int kRegSeg = 4;                          // segments kept in registers
  constexpr int kBatch = (sizeof(E) == 2) ? 4 : 2;    // segments whose loads fly together
  const int lane = threadIdx.x & 31;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(P) & 15u) == 0) &&
                      (!Q || (reinterpret_cast<uintptr_t>(Q) & 15u) == 0);
  const int nseg = (V + kSeg - 1) / kSeg;
  const bool keep = nseg <= kRegSeg;
  float ss[kMaxSeg], lsv[kRegSeg], rr[kRegSeg][8];
#pragma unroll
  for (int s0 = 0; s0 < kMaxSeg; s0 += kBatch) {
    if (s0 < nseg) {
      uint4 wp[kBatch][2], wq[kBatch][2];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int k0 = (s0 + q < nseg) ? (s0 + q) * kSeg + lane * 8 : V;
        load8_raw<E>(P, k0, V, vec_ok, wp[q]);
        if (Q) load8_raw<E>(Q, k0, V, vec_ok, wq[q]);
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int sg = s0 + q;
        float ls = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float r = resid(raw8_elem<E>(wp[q], e), Q ? raw8_elem<E>(wq[q], e) : -INFINITY,
                                Q != nullptr, Mt, iZt, Md, iZd, c2);
          ls = __fadd_rn(ls, r);
          if (sg < kRegSeg) rr[sg < kRegSeg ? sg : 0][e] = r;
        }
        if (sg < kRegSeg) lsv[sg < kRegSeg ? sg : 0] = ls;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ls = __fadd_rn(ls, __shfl_xor_sync(0xffffffffu, ls, off));
        ss[sg] = (sg < nseg) ? ls : 0.f;
      }
    } else {
#pragma unroll
      for (int q = 0; q < kBatch; ++q) ss[s0 + q] = 0.f;
    }
  }
  float S = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxSeg; ++s) S = __fadd_rn(S, ss[s]);
  if (Q && S == 0.f) return -1;
  const float t = __fmul_rn(u, S);
  int seg = -1, mode = 0, lastseg = -1;
  float base = 0.f, acc = 0.f, lastbase = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxSeg; ++s) {
    if (seg < 0 && s < nseg) {
      const float nxt = __fadd_rn(acc, ss[s]);
      if (ss[s] > 0.f) { lastseg = s; lastbase = acc; }
      if (nxt > t) { seg = s; base = acc; }
      acc = nxt;
    }
  }
  if (seg < 0) { seg = max(lastseg, 0); base = lastbase; mode = 1; }
  float r[8];
  float ls;
  if (keep) {
    ls = lsv[0];
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = rr[0][e];
#pragma unroll
    for (int q = 1; q < kRegSeg; ++q)
      if (q == seg) {
        ls = lsv[q];
#pragma unroll
        for (int e = 0; e < 8; ++e) r[e] = rr[q][e];
      }
  } else {
    ls = lane_resid<E>(P, Q, seg, lane, V, vec_ok, Mt, iZt, Md, iZd, c2, r);
  }
  const int tok = segment_pick(r, ls, seg * kSeg + lane * 8, base, t, mode, lane);
  return tok < 0 ? V - 1 : tok;
}

// ------------------------------------------------------------------ finishing helpers

__device__ __forceinline__ void fail_chain_row(const Params &p, int b, int tid, int nthreads) {
  const int g1 = p.gamma + 1;
  for (int j = tid; j < g1; j += nthreads) p.out_tokens[static_cast<long long>(b) * g1 + j] = -1;
  if (tid == 0 && p.accept_len) p.accept_len[b] = -1;   // no accept_len when only sampling
}

// the acceptance test u <= p_i(x_i)/q_i(x_i), with
// p_i(x_i)/q_i(x_i) = 2^(((lt - ld) + (Md - Mt)) * c2) * Zd / Zt
__device__ __forceinline__ bool rejects(float u, float lt, float ld, float Mt, float Zt, float Md,
                                        float Zd, float c2) {
  const float d = __fadd_rn(__fsub_rn(lt, ld), __fsub_rn(Md, Mt));
  const float ratio = __fmul_rn(ex2(__fmul_rn(d, c2)), __fdiv_rn(Zd, Zt));
  return !(u <= ratio);
}

__device__ __forceinline__ bool stats_ok(float m, float z) {
  return isfinite(m) && isfinite(z) && z > 0.f;
}

// argmax of a row is usable when it is finite (no NaN/+inf seen, some element above -inf)
__device__ __forceinline__ bool arg_ok(float v) { return v == v && v != -INFINITY; }

// Combines the unit partials of rows r = warp, warp + kWarps, ... of batch row b into per-row
// statistics. The loads for four rows per warp (two partials per lane each) are issued before
// any is combined, so this costs one round trip when C <= 64.
//
// keep (may be NULL): the unit partials of row keep_row are also copied there (C entries).
__device__ __forceinline__ void combine_rows_stats(const Params &p, int b, float *rowM,
                                                   float *rowZ, uint2 *keep = nullptr,
                                                   int keep_row = -1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint2 *base = p.ws_part + static_cast<long long>(b) * p.R * p.C;
  for (int r0 = warp; r0 < p.R; r0 += 4 * kWarps) {
    uint2 v[4][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = r0 + q * kWarps;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int c = lane + 32 * t;
        v[q][t] = (r < p.R && c < p.C) ? ldcg_u2(base + static_cast<long long>(r) * p.C + c)
                                       : make_uint2(0xff800000u, 0u);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = r0 + q * kWarps;
      if (r < p.R) {
        const bool kp = keep && r == keep_row;
        if (kp) {
          if (lane < p.C) keep[lane] = v[q][0];
          if (lane + 32 < p.C) keep[lane + 32] = v[q][1];
        }
        float m = -INFINITY, s = 0.f;
        stat_merge(m, s, __uint_as_float(v[q][0].x), __uint_as_float(v[q][0].y), p.c2);
        stat_merge(m, s, __uint_as_float(v[q][1].x), __uint_as_float(v[q][1].y), p.c2);
        // partials beyond the first 64: four loads in flight per lane, merged in index order
        const uint2 *pr = base + static_cast<long long>(r) * p.C;
        for (int c0 = lane + 64; c0 < p.C; c0 += 128) {
          uint2 w[4];
#pragma unroll
          for (int t = 0; t < 4; ++t)
            w[t] = (c0 + 32 * t < p.C) ? ldcg_u2(pr + c0 + 32 * t) : make_uint2(0xff800000u, 0u);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (kp && c0 + 32 * t < p.C) keep[c0 + 32 * t] = w[t];
            stat_merge(m, s, __uint_as_float(w[t].x), __uint_as_float(w[t].y), p.c2);
          }
        }
        warp_stat_merge(m, s, p.c2);
        if (lane == 0) { rowM[r] = m; rowZ[r] = s; }
      }
    }
  }
}

// Same for greedy argmax partials: g[r] = lowest index of the row maximum, ok[r] = the row is
// usable (finite maximum, no NaN / +inf seen).
__device__ __forceinline__ void combine_rows_arg(const Params &p, int b, int *g, int *ok) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint2 *base = p.ws_part + static_cast<long long>(b) * p.R * p.C;
  for (int r0 = warp; r0 < p.R; r0 += 4 * kWarps) {
    uint2 v[4][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = r0 + q * kWarps;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int c = lane + 32 * t;
        v[q][t] = (r < p.R && c < p.C) ? ldcg_u2(base + static_cast<long long>(r) * p.C + c)
                                       : make_uint2(0xff800000u, 0x7fffffffu);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = r0 + q * kWarps;
      if (r < p.R) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        arg_merge(bv, bi, __uint_as_float(v[q][0].x), static_cast<int>(v[q][0].y));
        arg_merge(bv, bi, __uint_as_float(v[q][1].x), static_cast<int>(v[q][1].y));
        const uint2 *pr = base + static_cast<long long>(r) * p.C;
        for (int c0 = lane + 64; c0 < p.C; c0 += 128) {
          uint2 w[4];
#pragma unroll
          for (int t = 0; t < 4; ++t)
            w[t] = (c0 + 32 * t < p.C) ? ldcg_u2(pr + c0 + 32 * t)
                                       : make_uint2(0xff800000u, 0x7fffffffu);
#pragma unroll
          for (int t = 0; t < 4; ++t)
            arg_merge(bv, bi, __uint_as_float(w[t].x), static_cast<int>(w[t].y));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, bv, off);
          const int i2 = __shfl_xor_sync(0xffffffffu, bi, off);
          arg_merge(bv, bi, v2, i2);
        }
        if (lane == 0) { g[r] = bi; ok[r] = arg_ok(bv) ? 1 : 0; }
      }
    }
  }
}

// Chain sampling, whole CTA: combines the statistics of every row of batch row b (rowM/rowZ in
// shared memory), copies the drafts to xs (shared memory) and runs the acceptance test of every
// draft with one warp ballot per 32 positions. Returns 0 with *n = the number of accepted
// drafts (on every thread), or a device error code (a non-finite row, a token outside [0, V)).
__device__ inline int chain_accept(const Params &p, int b, float *rowM, float *rowZ, int *xs,
                                   TailShared &sh, int *n_out, uint2 *keep_bonus = nullptr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = p.R, gamma = p.gamma;
  const float c2 = p.c2;
  const float *ub = p.uniforms + static_cast<long long>(b) * (gamma + 1);
  const int32_t *x = p.tokens + static_cast<long long>(b) * gamma;
  const float *xl = p.ws_xlogit + static_cast<long long>(b) * R;
  auto ldx = [&](int i) -> float { return ldcg_f(xl + i); };
  // one round trip: warp 0 fetches the first 32 positions' inputs, every thread a share of the
  // drafts, every warp the unit partials of its rows
  float ui = 0.f, lti = 0.f, ldi = 0.f;
  if (warp == 0 && lane < gamma) {
    ui = ub[lane];
    lti = ldx(lane);
    ldi = ldx(gamma + 1 + lane);
  }
  // gamma <= SPEC_MAX_GAMMA < kThreads: one draft per thread, kept in a register until the
  // partial loads below have been issued (a shared store would wait for it)
  const int xv = (static_cast<int>(threadIdx.x) < gamma) ? x[threadIdx.x] : 0;
  combine_rows_stats(p, b, rowM, rowZ, keep_bonus, gamma);
  if (static_cast<int>(threadIdx.x) < gamma) xs[threadIdx.x] = xv;
  __syncthreads();
  if (warp == 0) {
    int err = 0;
    for (int r = lane; r < R; r += 32)
      if (!stats_ok(rowM[r], rowZ[r])) err = SPEC_ERR_NONFINITE;
    for (int i = lane; i < gamma; i += 32)
      if (xs[i] < 0 || xs[i] >= p.V) err = err ? err : SPEC_ERR_TOKEN;
    const unsigned any_err = __ballot_sync(0xffffffffu, err != 0);
    int n = gamma;
    if (any_err) {
      err = __shfl_sync(0xffffffffu, err, __ffs(any_err) - 1);
    } else {
      for (int i0 = 0; i0 < gamma; i0 += 32) {
        const int i = i0 + lane;
        bool rej = false;
        if (i < gamma) {
          if (i0 > 0) { ui = ub[i]; lti = ldx(i); ldi = ldx(gamma + 1 + i); }
          const int rd = gamma + 1 + i;
          rej = rejects(ui, lti, ldi, rowM[i], rowZ[i], rowM[rd], rowZ[rd], c2);
        }
        const unsigned rb = __ballot_sync(0xffffffffu, rej);
        if (rb) { n = i0 + __ffs(rb) - 1; break; }
      }
    }
    if (lane == 0) { sh.n = n; sh.err = err; }
  }
  __syncthreads();
  *n_out = sh.n;
  return sh.err;
}

// out_tokens[b] = x_0..x_{n-1}, tok, then -1; accept_len[b] = n. x: the step's drafts.
__device__ __forceinline__ void emit_chain(const Params &p, int b, int n, int tok, const int *x,
                                           int tid, int nthreads) {
  const int g1 = p.gamma + 1;
  int32_t *o = p.out_tokens + static_cast<long long>(b) * g1;
  for (int j = tid; j < g1; j += nthreads) o[j] = (j < n) ? x[j] : (j == n ? tok : -1);
  if (tid == 0 && p.accept_len) p.accept_len[b] = n;
}

// Chain sampling, one warp, for steps whose rows are single units (gamma <= 31, V <=
// kWarpTailMaxV): lane i holds the statistics of rows i and i + 32 (m0/z0, m1/z1) and the
// logits at draft token x_i of target row i (lti) and draft row i (ldi).
template <typename E>
__device__ void tail_chain_sample_regs(const Params &p, int b, float m0, float z0, float m1,
                                       float z1, float lti, float ldi) {
  const int lane = threadIdx.x & 31;
  const int R = p.R, gamma = p.gamma;
  const float c2 = p.c2;
  const float *ub = p.uniforms + static_cast<long long>(b) * (gamma + 1);
  const int32_t *x = p.tokens + static_cast<long long>(b) * gamma;
  int xi = 0;
  float ui = 0.f;
  if (lane < gamma) {
    xi = x[lane];
    ui = ub[lane];
  }
  const float u = ub[gamma];
  int err = 0;
  if ((lane < R && !stats_ok(m0, z0)) || (lane + 32 < R && !stats_ok(m1, z1)))
    err = SPEC_ERR_NONFINITE;
  if (lane < gamma && (xi < 0 || xi >= p.V)) err = err ? err : SPEC_ERR_TOKEN;
  const unsigned any_err = __ballot_sync(0xffffffffu, err != 0);
  if (any_err) {
    err = __shfl_sync(0xffffffffu, err, __ffs(any_err) - 1);
    if (lane == 0) set_status(p.status, err);
    fail_chain_row(p, b, lane, 32);
    return;
  }
  // statistics of draft row gamma+1+lane (held by lane gamma+1+lane, or lane gamma+1+lane-32)
  const int rd = gamma + 1 + lane;
  const float dmA = __shfl_sync(0xffffffffu, m0, rd & 31);
  const float dzA = __shfl_sync(0xffffffffu, z0, rd & 31);
  const float dmB = __shfl_sync(0xffffffffu, m1, rd & 31);
  const float dzB = __shfl_sync(0xffffffffu, z1, rd & 31);
  const float Md_i = rd < 32 ? dmA : dmB, Zd_i = rd < 32 ? dzA : dzB;
  const bool rej = lane < gamma && rejects(ui, lti, ldi, m0, z0, Md_i, Zd_i, c2);
  const unsigned rb = __ballot_sync(0xffffffffu, rej);
  const int n = rb ? __ffs(rb) - 1 : gamma;
  const float Mt = __shfl_sync(0xffffffffu, m0, n);
  const float Zt = __shfl_sync(0xffffffffu, z0, n);
  const int rn = gamma + 1 + n;
  const float mA = __shfl_sync(0xffffffffu, m0, rn & 31), zA = __shfl_sync(0xffffffffu, z0, rn & 31);
  const float mB = __shfl_sync(0xffffffffu, m1, rn & 31), zB = __shfl_sync(0xffffffffu, z1, rn & 31);
  const float Md = rn < 32 ? mA : mB, Zd = rn < 32 ? zA : zB;
  const E *P = row_ptr<E>(p, b, n);
  const E *Q = (n < gamma) ? row_ptr<E>(p, b, rn) : nullptr;
  const float iZt = __frcp_rn(Zt), iZd = Q ? __frcp_rn(Zd) : 0.f;
  int tok = draw_token_warp<E>(P, Q, Mt, iZt, Q ? Md : 0.f, iZd, c2, p.V, u);
  if (tok < 0) tok = draw_token_warp<E>(P, nullptr, Mt, iZt, 0.f, 0.f, c2, p.V, u);
  emit_chain(p, b, n, tok, x, lane, 32);
}

// Greedy chain: smem holds g[R] (row argmaxes), gok[R] (row usable), xs[gamma], gathered here
// from the unit partials.
__device__ inline void tail_chain_greedy(const Params &p, int b, float *smem, TailShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = p.R, gamma = p.gamma;
  int *g = reinterpret_cast<int *>(smem);
  int *gok = g + R;
  int *xs = gok + R;
  const int32_t *x = p.tokens + static_cast<long long>(b) * gamma;
  const int xv = (static_cast<int>(threadIdx.x) < gamma) ? x[threadIdx.x] : 0;
  combine_rows_arg(p, b, g, gok);
  if (static_cast<int>(threadIdx.x) < gamma) xs[threadIdx.x] = xv;
  __syncthreads();
  if (warp == 0) {
    int err = 0;
    for (int r = lane; r < R; r += 32)
      if (!gok[r]) err = SPEC_ERR_NONFINITE;
    for (int i = lane; i < gamma; i += 32)
      if (xs[i] < 0 || xs[i] >= p.V) err = err ? err : SPEC_ERR_TOKEN;
    const unsigned any_err = __ballot_sync(0xffffffffu, err != 0);
    int n = gamma;
    if (any_err) {
      err = __shfl_sync(0xffffffffu, err, __ffs(any_err) - 1);
    } else {
      for (int i0 = 0; i0 < gamma; i0 += 32) {
        const int i = i0 + lane;
        const bool rej = (i < gamma) && (xs[i] != g[i]);
        const unsigned rb = __ballot_sync(0xffffffffu, rej);
        if (rb) { n = i0 + __ffs(rb) - 1; break; }
      }
    }
    if (lane == 0) { sh.n = n; sh.err = err; }
  }
  __syncthreads();
  if (sh.err) {
    if (threadIdx.x == 0) set_status(p.status, sh.err);
    fail_chain_row(p, b, threadIdx.x, kThreads);
    return;
  }
  emit_chain(p, b, sh.n, g[sh.n], xs, threadIdx.x, kThreads);
}

// Greedy tree (any N up to SPEC_MAX_NODES): smem holds g[N], then par, tok, anc, acc, dep
// (N ints each).
__device__ inline void tail_tree(const Params &p, int b, float *smem, TailShared &sh) {
  const int N = p.N;
  int *g = reinterpret_cast<int *>(smem);
  int *par = g + N;
  int *tok = par + N;
  int *anc = tok + N;
  int *acc = anc + N;
  int *dep = acc + N;
  const long long bN = static_cast<long long>(b) * N;
  if (threadIdx.x == 0) sh.err = 0;
  // one round trip: parents and tokens, and the argmax partials of every node
  for (int j = threadIdx.x; j < N; j += kThreads) {
    par[j] = p.parents[bN + j];
    tok[j] = (j == 0) ? 0 : p.tokens[bN + j];
  }
  combine_rows_arg(p, b, g, anc);   // anc[] holds the row-usable flags until reused below
  __syncthreads();
  for (int j = threadIdx.x; j < N; j += kThreads) {
    if (!anc[j]) atomicCAS(&sh.err, 0, SPEC_ERR_NONFINITE);
    const int pj = par[j], tj = tok[j];
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
  constexpr int kPer = (SPEC_MAX_NODES + kThreads - 1) / kThreads;
  for (int span = 1; span < N; span <<= 1) {
    int na[kPer], nc[kPer], nd[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int j = threadIdx.x + q * kThreads;
      if (j < N) {
        const int a = anc[j];
        na[q] = anc[a];
        nc[q] = acc[j] & acc[a];
        nd[q] = dep[j] + dep[a];
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int j = threadIdx.x + q * kThreads;
      if (j < N) { anc[j] = na[q]; acc[j] = nc[q]; dep[j] = nd[q]; }
    }
    __syncthreads();
  }
  // deepest accepted node, smallest index among equals
  int key = -1;
  for (int j = threadIdx.x; j < N; j += kThreads)
    if (acc[j]) key = max(key, (dep[j] << 11) | (2047 - j));
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

// Greedy tree verification for trees of at most 64 nodes: all warps combine the argmax
// partials into shared memory, then warp 0 holds nodes lane and lane + 32 in registers and does
// the rest with warp votes and shuffles (no block barriers): the accepted set level by level
// as a 64-bit mask, the deepest accepted node by a warp maximum, and the path by walking
// parents back from it.
// smem holds g[N] and the row-usable flags okf[N].
__device__ inline void tail_tree_small(const Params &p, int b, float *smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int N = p.N;
  int *g = reinterpret_cast<int *>(smem);
  int *okf = g + N;
  const long long bN = static_cast<long long>(b) * N;
  int par0 = -1, par1 = -1, tok0 = 0, tok1 = 0;
  if (warp == 0) {   // issued before the partial loads, used after them
    if (lane < N) {
      par0 = p.parents[bN + lane];
      tok0 = (lane == 0) ? 0 : p.tokens[bN + lane];
    }
    if (lane + 32 < N) {
      par1 = p.parents[bN + lane + 32];
      tok1 = p.tokens[bN + lane + 32];
    }
  }
  combine_rows_arg(p, b, g, okf);
  __syncthreads();
  if (warp != 0) return;   // no block barrier follows
  const int j0 = lane, j1 = lane + 32;
  const bool in0 = j0 < N, in1 = j1 < N;
  auto code = [&](int j, bool in, int par, int tok, int what) -> bool {
    if (!in) return false;
    if (what == 0) return okf[j] == 0;
    if (what == 1) return j == 0 ? (par != -1) : (par < 0 || par >= j);
    return j > 0 && (tok < 0 || tok >= p.V);
  };
  int err = 0;
  const int codes[3] = {SPEC_ERR_NONFINITE, SPEC_ERR_PARENT, SPEC_ERR_TOKEN};
#pragma unroll
  for (int w = 0; w < 3; ++w) {
    const bool bad = code(j0, in0, par0, tok0, w) || code(j1, in1, par1, tok1, w);
    if (!err && __any_sync(0xffffffffu, bad)) err = codes[w];
  }
  int32_t *pn = p.path_nodes + bN;
  int32_t *ot = p.out_tokens + bN;
  if (err) {
    if (in0) { pn[j0] = -1; ot[j0] = -1; }
    if (in1) { pn[j1] = -1; ot[j1] = -1; }
    if (lane == 0) { set_status(p.status, err); p.accept_len[b] = -1; }
    return;
  }
  // level by level: a node is accepted at step d when its parent was accepted (at step d - 1)
  // and its token is the parent's argmax, so the step at which it is accepted is its depth
  // (parents precede children, so a node's parent is always settled first). The accepted set
  // is one 64-bit mask, extended by two ballots per level.
  const bool m0 = in0 && j0 > 0 && tok0 == g[par0];
  const bool m1 = in1 && tok1 == g[par1];
  unsigned long long accm = 1ull;   // the root
  int dep0 = (in0 && j0 == 0) ? 0 : -1, dep1 = -1;
  for (int level = 1; level < N; ++level) {
    const bool a0 = m0 && dep0 < 0 && ((accm >> par0) & 1ull);
    const bool a1 = m1 && dep1 < 0 && ((accm >> par1) & 1ull);
    const unsigned lo = __ballot_sync(0xffffffffu, a0), hi = __ballot_sync(0xffffffffu, a1);
    if ((lo | hi) == 0u) break;
    if (a0) dep0 = level;
    if (a1) dep1 = level;
    accm |= static_cast<unsigned long long>(lo) | (static_cast<unsigned long long>(hi) << 32);
  }
  int key = -1;
  if (dep0 >= 0) key = (dep0 << 11) | (2047 - j0);
  if (dep1 >= 0) key = max(key, (dep1 << 11) | (2047 - j1));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, off));
  const int best = 2047 - (key & 2047);
  const int D = key >> 11;
  if (in0 && j0 > D) { pn[j0] = -1; ot[j0] = -1; }
  if (in1 && j1 > D) { pn[j1] = -1; ot[j1] = -1; }
  int v = best;
  for (int d = D; d >= 0; --d) {   // warp-uniform walk from the deepest node to the root
    const int src = v & 31;
    const int t0 = __shfl_sync(0xffffffffu, tok0, src), t1 = __shfl_sync(0xffffffffu, tok1, src);
    const int q0 = __shfl_sync(0xffffffffu, par0, src), q1 = __shfl_sync(0xffffffffu, par1, src);
    if (lane == 0) {
      pn[d] = v;
      if (d > 0) ot[d - 1] = (v >= 32) ? t1 : t0;
    }
    v = (v >= 32) ? q1 : q0;
  }
  if (lane == 0) {
    ot[D] = g[best];
    p.accept_len[b] = D;
  }
}

// The bonus draw (from p_gamma alone) of a row with no unaligned head or tail, from the stream
// kernel's unit partials: unit u holds p-mass w_u = s_u * 2^((m_u - M) * c2) / Z, so the unit
// where the running sum crosses t = u * sum(w) is found without reading the row; warp 0 then
// reads that one unit (4 KB) and finds the element with warp scans, in index order. Writes the
// outputs.
template <typename E>
__device__ void bonus_draw_units(const Params &p, int b, int n, float M, float Z,
                                 const uint2 *part, const int *xs) {
  constexpr int kEPV = Elem<E>::kPerVec;
  const int lane = threadIdx.x & 31;
  const int C = p.C;
  const float c2 = p.c2, iZ = __frcp_rn(Z);
  const float u = p.uniforms[static_cast<long long>(b) * (p.gamma + 1) + p.gamma];
  // lane l sums the masses of units [l*q, (l+1)*q) in order; a warp scan gives every prefix
  const int q = (C + 31) / 32;
  const int u0 = min(C, lane * q), u1 = min(C, u0 + q);
  auto mass = [&](int uc) -> float {
    const uint2 w = part[uc];
    return __fmul_rn(__fmul_rn(__uint_as_float(w.y), ex2_shift(__uint_as_float(w.x), M, c2)), iZ);
  };
  float ls = 0.f;
  for (int uc = u0; uc < u1; ++uc) ls = __fadd_rn(ls, mass(uc));
  float inc = ls;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc = __fadd_rn(inc, y);
  }
  const float S = __shfl_sync(0xffffffffu, inc, 31);
  const float t = __fmul_rn(u, S);
  const float exc = __shfl_up_sync(0xffffffffu, inc, 1);
  // the crossing unit: the owner lane scans its block; no crossing (rounding): last unit with mass
  const unsigned over = __ballot_sync(0xffffffffu, inc > t);
  int uc_sel = -1, mode = 0;
  float base = 0.f;
  if (over) {
    const int ol = __ffs(over) - 1;
    if (lane == ol) {
      float acc = (lane == 0) ? 0.f : exc;
      for (int uc = u0; uc < u1; ++uc) {
        const float nx = __fadd_rn(acc, mass(uc));
        if (nx > t) { uc_sel = uc; base = acc; break; }
        acc = nx;
      }
      if (uc_sel < 0) { uc_sel = u1 - 1; base = acc; }
    }
    uc_sel = __shfl_sync(0xffffffffu, uc_sel, ol);
    base = __shfl_sync(0xffffffffu, base, ol);
  } else {
    mode = 1;
    int last = -1;
    for (int uc = u0; uc < u1; ++uc)
      if (mass(uc) > 0.f) last = uc;
    const unsigned has = __ballot_sync(0xffffffffu, last >= 0);
    uc_sel = __shfl_sync(0xffffffffu, last, has ? 31 - __clz(has) : 0);
    uc_sel = max(uc_sel, 0);
  }
  // the element inside unit uc_sel: vectors j*32 + lane, elements in order
  const E *row = row_ptr<E>(p, b, n);
  const RowGeom g = row_geom<E>(row, p.V);
  uint4 buf[kVPL];
  float eh, et;
  load_span<E>(row, g, uc_sel * kUnitVecs, g.nv, false, lane, buf, eh, et);
  int tok = -1, lastpos = -1;
#pragma unroll
  for (int j = 0; j < kVPL; ++j) {
    float pe[kEPV];
    float vs = 0.f;
#pragma unroll
    for (int e = 0; e < kEPV; ++e) {
      pe[e] = __fmul_rn(ex2_shift(vec_elem<E>(buf[j], e), M, c2), iZ);
      vs = __fadd_rn(vs, pe[e]);
    }
    const int k0 = (uc_sel * kUnitVecs + j * 32 + lane) * kEPV;
#pragma unroll
    for (int e = 0; e < kEPV; ++e)
      if (pe[e] > 0.f) lastpos = k0 + e;
    float vi = vs;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, vi, off);
      if (lane >= off) vi = __fadd_rn(vi, y);
    }
    if (mode == 0 && tok < 0) {
      const float ve = __shfl_up_sync(0xffffffffu, vi, 1);
      const float lex = (lane == 0) ? base : __fadd_rn(base, ve);
      const unsigned cr = __ballot_sync(0xffffffffu, __fadd_rn(base, vi) > t);
      if (cr) {
        const int cl = __ffs(cr) - 1;
        int tk = -1;
        if (lane == cl) {
          float acc = lex;
          for (int e = 0; e < kEPV; ++e) {
            const float nx = __fadd_rn(acc, pe[e]);
            if (nx > t) { tk = k0 + e; break; }
            acc = nx;
          }
          if (tk < 0) tk = (lastpos >= k0) ? lastpos : k0 + kEPV - 1;
        }
        tok = __shfl_sync(0xffffffffu, tk, cl);
      }
      base = __fadd_rn(base, __shfl_sync(0xffffffffu, vi, 31));
    }
  }
  if (tok < 0) {   // rounding left no crossing inside the unit: its last element with mass
    const unsigned has = __ballot_sync(0xffffffffu, lastpos >= 0);
    tok = has ? __shfl_sync(0xffffffffu, lastpos, 31 - __clz(has)) : 0;
    tok = max(tok, 0);
  }
  emit_chain(p, b, n, tok, xs, lane, 32);
}

// The cluster draw when every CTA's slice has at most kWarps * kRegSegs segments: warp w of
// CTA `rank` loads segments rank*K + w*kRegSegs .. +kRegSegs - 1 (one round trip) and keeps
// them in registers. Warp totals -> CTA total -> cluster prefix through distributed shared
// memory; then the warp whose range holds u*S picks the token from its registers and writes
// the outputs, with no second pass over the rows and no block barrier after the cluster's.
template <typename E>
__device__ __forceinline__ void cluster_draw_regs(const Params &p, int b, int n, const E *P, const E *Q, float Mt,
                                  float iZt, float Md, float iZd, float u, const int *xs, int K,
                                  float *segsum, TailShared &sh, float &s_total) {
  namespace cg = cooperative_groups;
  constexpr int kSI = kRegSegs;
  cg::cluster_group cl = cg::this_cluster();
  const int S = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int V = p.V;
  const float c2 = p.c2;
  const int nseg = (V + kSeg - 1) / kSeg;
  const int lo = min(nseg, rank * K), hi = min(nseg, lo + K);
  const int s0 = lo + warp * kSI;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(P) & 15u) == 0) &&
                      (!Q || (reinterpret_cast<uintptr_t>(Q) & 15u) == 0);
  uint4 wp[kSI][2], wq[kSI][2];
#pragma unroll
  for (int t = 0; t < kSI; ++t) {
    const int k0 = (s0 + t < hi) ? (s0 + t) * kSeg + lane * 8 : V;
    load8_raw<E>(P, k0, V, vec_ok, wp[t]);
    if (Q) load8_raw<E>(Q, k0, V, vec_ok, wq[t]);
  }
  auto rval = [&](int t, int e) -> float {
    return resid(raw8_elem<E>(wp[t], e), Q ? raw8_elem<E>(wq[t], e) : -INFINITY, Q != nullptr,
                 Mt, iZt, Md, iZd, c2);
  };
  float lsum[kSI], ssum[kSI];
  float wtot = 0.f;
#pragma unroll
  for (int t = 0; t < kSI; ++t) {
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ls = __fadd_rn(ls, rval(t, e));
    lsum[t] = ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ls = __fadd_rn(ls, __shfl_xor_sync(0xffffffffu, ls, off));
    ssum[t] = ls;
    wtot = __fadd_rn(wtot, ls);
  }
  if (lane == 0) sh.warp_tot[warp] = wtot;
  __syncthreads();
  // every warp: the inclusive scan of the warp totals (lane w holds warps 0..w), so this warp's
  // offset inside the slice and the slice total come out identical in every warp
  const float wv = (lane < kWarps) ? sh.warp_tot[lane] : 0.f;
  float winc = wv;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, winc, off);
    if (lane >= off) winc = __fadd_rn(winc, y);
  }
  const float wexc = __shfl_up_sync(0xffffffffu, winc, 1);
  const float woff = (warp == 0) ? 0.f : __shfl_sync(0xffffffffu, wexc, warp);
  const float ctot = __shfl_sync(0xffffffffu, winc, kWarps - 1);
  if (threadIdx.x == 0) s_total = ctot;
  cluster_sync_publish();   // every slice total written
  // every warp: the cluster prefix (lane r holds rank r's inclusive prefix)
  float pre = (lane < S) ? *cl.map_shared_rank(&s_total, lane) : 0.f;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, pre, off);
    if (lane >= off) pre = __fadd_rn(pre, y);
  }
  cluster_sync_exec();   // every CTA has read its peers' totals
  const float Sall = __shfl_sync(0xffffffffu, pre, S - 1);
  if (Q && Sall == 0.f) {
    // the residual vanished: draw from p_n alone, on the first CTA of the cluster
    if (rank != 0) return;
    const int tok = draw_token_cta<E>(P, nullptr, Mt, iZt, 0.f, 0.f, c2, V, u, segsum, sh);
    emit_chain(p, b, n, tok, xs, threadIdx.x, kThreads);
    return;
  }
  const float t = __fmul_rn(u, Sall);
  // owner rank: the first whose inclusive prefix exceeds t, else the last holding mass
  const unsigned over = __ballot_sync(0xffffffffu, lane < S && pre > t);
  const float prev = __shfl_up_sync(0xffffffffu, pre, 1);
  const unsigned mass = __ballot_sync(0xffffffffu, lane < S && pre > (lane ? prev : 0.f));
  int owner, mode = 0;
  if (over) {
    owner = __ffs(over) - 1;
  } else {
    mode = 1;
    owner = mass ? 31 - __clz(mass) : 0;
  }
  if (rank != owner) return;
  const float base = (rank == 0) ? 0.f : __shfl_sync(0xffffffffu, pre, rank - 1);
  // owner warp inside the CTA: the first whose range ends above t (mode 0), else the last
  // warp with mass; decided from the scan every warp holds
  const unsigned wover = __ballot_sync(0xffffffffu, lane < kWarps && __fadd_rn(base, winc) > t);
  const unsigned wmass = __ballot_sync(0xffffffffu, lane < kWarps && wv > 0.f);
  int ow, wmode = mode;
  if (mode == 0 && wover) {
    ow = __ffs(wover) - 1;
  } else {
    wmode = 1;
    ow = wmass ? 31 - __clz(wmass) : 0;
  }
  if (warp != ow) return;
  // inside the owner warp: the segment, then the element
  float acc = __fadd_rn(base, woff);
  int seg = -1, lastseg = -1;
  float segbase = acc, lastbase = acc;
#pragma unroll
  for (int q = 0; q < kSI; ++q) {
    const float nx = __fadd_rn(acc, ssum[q]);
    if (s0 + q < hi) {
      if (ssum[q] > 0.f) { lastseg = q; lastbase = acc; }
      if (seg < 0 && wmode == 0 && nx > t) { seg = q; segbase = acc; }
    }
    acc = nx;
  }
  int smode = wmode;
  if (seg < 0) { seg = max(lastseg, 0); segbase = lastbase; smode = 1; }
  float r[8];
  float ls = 0.f;
#pragma unroll
  for (int q = 0; q < kSI; ++q)
    if (q == seg) {
#pragma unroll
      for (int e = 0; e < 8; ++e) r[e] = rval(q, e);
      ls = lsum[q];
    }
  int tok = segment_pick(r, ls, (s0 + seg) * kSeg + lane * 8, segbase, t, smode, lane);
  if (tok < 0) tok = V - 1;   // unreachable when the slice holds mass
  emit_chain(p, b, n, tok, xs, lane, 32);
}

// The correction / bonus draw of chain sampling over a thread-block cluster of S CTAs (S = 1:
// no cluster), after acceptance gave n: CTA `rank` sums r(k) = max(0, p_n(k) - q_n(k)) (or
// p_gamma(k)) over its slice of 256-element segments into segsum (shared memory); the slice
// totals are exchanged through distributed shared memory between two cluster barriers; the CTA
// whose slice holds u * S picks the token and writes the outputs. Every CTA of the cluster calls
// it; CTAs other than the writer return from it early.
template <typename E>
__device__ void cluster_draw(const Params &p, int b, int n, const float *rowM, const float *rowZ,
                             const int *xs, float *segsum, TailShared &sh, float &s_total,
                             float *s_pre) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int S = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int gamma = p.gamma;
  const E *P = row_ptr<E>(p, b, n);
  const E *Q = (n < gamma) ? row_ptr<E>(p, b, gamma + 1 + n) : nullptr;
  const float Mt = rowM[n], iZt = __frcp_rn(rowZ[n]);
  const float Md = Q ? rowM[gamma + 1 + n] : 0.f, iZd = Q ? __frcp_rn(rowZ[gamma + 1 + n]) : 0.f;
  const float u = p.uniforms[static_cast<long long>(b) * (gamma + 1) + gamma];
  const int nseg = (p.V + kSeg - 1) / kSeg;
  const int K = (nseg + S - 1) / S;
  if (K <= kWarps * kRegSegs) {   // the same on every CTA of the cluster
    cluster_draw_regs<E>(p, b, n, P, Q, Mt, iZt, Md, iZd, u, xs, K, segsum, sh, s_total);
    return;
  }
  const int lo = min(nseg, rank * K), hi = min(nseg, lo + K), nl = hi - lo;
  segment_sums<E>(P, Q, Mt, iZt, Md, iZd, p.c2, p.V, lo, hi, segsum, lo);
  __syncthreads();
  if (threadIdx.x < 32) {   // slice total: strided lane sums, then a fixed xor tree
    float tot = 0.f;
    for (int j = threadIdx.x; j < nl; j += 32) tot = __fadd_rn(tot, segsum[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot = __fadd_rn(tot, __shfl_xor_sync(0xffffffffu, tot, off));
    if (threadIdx.x == 0) s_total = tot;
  }
  cl.sync();   // every slice total written
  if (threadIdx.x < 32) {   // lane r reads rank r's total; inclusive scan in rank order
    const int r = threadIdx.x;
    float v = (r < S) ? *cl.map_shared_rank(&s_total, r) : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, v, off);
      if (r >= off) v = __fadd_rn(v, y);
    }
    if (r < S) s_pre[r + 1] = v;
    if (r == 0) s_pre[0] = 0.f;
  }
  cl.sync();   // every CTA has read its peers' totals; shared memory is private again
  const float Sall = s_pre[S];
  int tok = -1;
  if (Q && Sall == 0.f) {
    // the residual vanished: draw from p_n alone, on the first CTA of the cluster
    if (rank != 0) return;
    tok = draw_token_cta<E>(P, nullptr, Mt, iZt, 0.f, 0.f, p.c2, p.V, u, segsum, sh);
  } else {
    const float t = __fmul_rn(u, Sall);
    int owner = -1, mode = 0;
    for (int r = 0; r < S; ++r)
      if (owner < 0 && s_pre[r + 1] > t) owner = r;
    if (owner < 0) {   // t >= S after rounding: the last slice holding mass
      mode = 1;
      for (int r = 0; r < S; ++r)
        if (s_pre[r + 1] > s_pre[r]) owner = r;
      owner = max(owner, 0);
    }
    if (rank != owner) return;
    tok = pick_in_slice<E>(P, Q, Mt, iZt, Md, iZd, p.c2, p.V, segsum, nl, lo, s_pre[rank], t,
                           mode, sh);
  }
  emit_chain(p, b, n, tok, xs, threadIdx.x, kThreads);
}

// ------------------------------------------------------------------ the kernels
//
// Every call runs two kernels on its stream. The stream kernel reads every logit once and
// writes one partial per unit; the finishing kernel, launched as a programmatic dependent of
// the stream kernel (so its launch overlaps the stream kernel's last wave), waits for the
// stream kernel's results and turns them into outputs.

// One unit's result from its registers: the 8-byte partial (softmax statistics or argmax), and
// for chain sampling the logit at the row's draft token x when this unit holds it.
template <typename E, int MODE>
__device__ __forceinline__ void unit_work(const Params &p, int unit, const UnitId &u,
                                          const E *row, const RowGeom &g,
                                          const uint4 (&buf)[kVPL], float eh, float et, int x,
                                          int lane) {
  constexpr bool kStats = (MODE == kChainSample || MODE == kProbs);
  uint2 part;
  if constexpr (kStats) {
    float m, s;
    unit_stats<E>(buf, eh, et, p.c2, m, s);
    part = make_uint2(__float_as_uint(m), __float_as_uint(s));
  } else {
    float v;
    int i;
    unit_argmax<E>(buf, eh, et, g, u.chunk * kUnitVecs, lane, v, i);
    part = make_uint2(__float_as_uint(v), static_cast<uint32_t>(i));
  }
  if (lane == 0) p.ws_part[unit] = part;
  if constexpr (MODE == kChainSample) {
    if (x >= 0 && x < p.V) {
      const int vb = u.chunk * kUnitVecs;
      float val = 0.f;
      if (span_logit<E>(row, g, vb, vb + kUnitVecs, u.chunk == 0, x, lane, buf, &val) &&
          lane == 0)
        p.ws_xlogit[static_cast<long long>(u.b) * p.R + u.r] = val;
    }
  }
}

// The draft token of a chain-sampling row (-1 for the bonus row and other modes).
template <int MODE>
__device__ __forceinline__ int unit_token(const Params &p, const UnitId &u) {
  if constexpr (MODE == kChainSample) {
    if (u.r != p.gamma) {
      const int i = (u.r < p.Rt) ? u.r : u.r - p.Rt;
      return __ldg(p.tokens + static_cast<long long>(u.b) * p.gamma + i);
    }
  }
  return -1;
}

// The stream kernel: warp w of the grid reduces units w, w + W, w + 2W, ... (W warps in all),
// each to one 8-byte partial. For chain sampling it also records the logit at each row's draft
// token, taken from the registers of the lane that loaded it (or, for a head/tail element,
// loaded by chunk 0). No barriers, atomics or fences: the finishing kernel reads the partials
// only after this grid has completed.
template <typename E, int MODE>
__global__ void __launch_bounds__(kThreads, 2) stream_kernel(Params p) {
  // The finishing kernel may be scheduled as soon as every CTA of this grid is running; this
  // grid itself reads nothing before the kernel ahead of it on the stream has completed.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int W = gridDim.x * kWarps;
  for (int unit = blockIdx.x * kWarps + (threadIdx.x >> 5); unit < p.units; unit += W) {
    const UnitId u = unit_id(p, unit);
    // the draft token of this row, fetched before the unit's data so both loads overlap
    const int x = unit_token<MODE>(p, u);
    const E *row = row_ptr<E>(p, u.b, u.r);
    const RowGeom g = row_geom<E>(row, p.V);
    uint4 buf[kVPL];
    float eh, et;
    load_unit<E>(row, g, u.chunk, lane, buf, eh, et);
    unit_work<E, MODE>(p, unit, u, row, g, buf, eh, et, x, lane);
  }
}

// Lets the next kernel on the stream (the next call's stream kernel) be scheduled early, then
// waits until the stream kernel of this call has completed and its writes are visible.
__device__ __forceinline__ void wait_stream_kernel() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Finishing kernel for chain sampling: one thread-block cluster of S CTAs per batch row (S = the
// cluster size, blockIdx.x = b * S + rank). Every CTA of the cluster combines the row's
// partials and decides acceptance (cheap, redundant); CTA `rank` then sums the residual (or
// bonus) weights over its slice of the vocabulary into shared memory. The slice totals are
// exchanged through distributed shared memory after a cluster barrier; the CTA whose slice
// holds the crossing draws the token from its own segment sums and writes the outputs.
template <typename E>
__global__ void __launch_bounds__(kThreads, 2) finish_chain_sample(Params p) {
  namespace cg = cooperative_groups;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float *rowM = reinterpret_cast<float *>(smem_raw);
  float *rowZ = rowM + p.R;
  // [C] the bonus row's unit partials, at byte offset 8R: 8-byte aligned for every R
  uint2 *bonus_part = reinterpret_cast<uint2 *>(rowZ + p.R);
  float *segsum = reinterpret_cast<float *>(bonus_part + p.C);
  __shared__ TailShared sh;
  __shared__ int xs[SPEC_MAX_GAMMA];
  __shared__ float s_total;
  __shared__ float s_pre[kMaxCluster + 1];
  cg::cluster_group cl = cg::this_cluster();
  const int S = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / S;
  wait_stream_kernel();
  int n = 0;
  const int err = chain_accept(p, b, rowM, rowZ, xs, sh, &n, bonus_part);
  if (err) {   // the same on every CTA of the cluster: all of them leave here
    if (rank == 0) {
      if (threadIdx.x == 0) set_status(p.status, err);
      fail_chain_row(p, b, threadIdx.x, kThreads);
    }
    return;
  }
  if (n == p.gamma) {
    // the bonus draw, from the unit partials when the row has no unaligned head or tail (the
    // same decision on every CTA of the cluster; no CTA has touched a peer's shared memory)
    const RowGeom g = row_geom<E>(row_ptr<E>(p, b, n), p.V);
    if (g.h == 0 && g.tl == 0) {
      if (rank == 0 && threadIdx.x < 32)
        bonus_draw_units<E>(p, b, n, rowM[n], rowZ[n], bonus_part, xs);
      return;
    }
  }
  cluster_draw<E>(p, b, n, rowM, rowZ, xs, segsum, sh, s_total, s_pre);
}

// Finishing kernel for chain sampling when every row is a single unit (gamma <= 31, V <=
// kWarpTailMaxV): one warp per batch row; lane i holds rows i and i + 32 and the draft-token
// logits of position i. One CTA per SM at most is plenty (B / 16 CTAs), so each thread may use
// up to 128 registers and the draw keeps the residual of the rows in registers.
template <typename E>
__global__ void __launch_bounds__(kThreads, 1) finish_chain_sample_warp(Params p) {
  wait_stream_kernel();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (b >= p.B) return;
  const int R = p.R, gamma = p.gamma;
  const uint2 *part = p.ws_part + static_cast<long long>(b) * R;   // C == 1
  const float *xl = p.ws_xlogit + static_cast<long long>(b) * R;
  float m0 = 0.f, z0 = 1.f, m1 = 0.f, z1 = 1.f, lti = 0.f, ldi = 0.f;
  if (lane < R) {
    const uint2 v = ldcg_u2(part + lane);
    m0 = __uint_as_float(v.x);
    z0 = __uint_as_float(v.y);
  }
  if (lane + 32 < R) {
    const uint2 v = ldcg_u2(part + lane + 32);
    m1 = __uint_as_float(v.x);
    z1 = __uint_as_float(v.y);
  }
  if (lane < gamma) {
    lti = ldcg_f(xl + lane);
    ldi = ldcg_f(xl + gamma + 1 + lane);
  }
  tail_chain_sample_regs<E>(p, b, m0, z0, m1, z1, lti, ldi);
}

// Four consecutive elements of a row as fp32 (8 bytes of bf16 or 16 bytes of fp32; p must be
// aligned to that size).
template <typename E> __device__ __forceinline__ uint2 ld_quad_raw(const E *p);
template <> __device__ __forceinline__ uint2 ld_quad_raw<uint16_t>(const uint16_t *p) {
  return __ldcs(reinterpret_cast<const uint2 *>(p));
}
template <typename E> __device__ __forceinline__ float quad_elem(const uint2 &lo, const uint2 &hi,
                                                                 int e);
template <> __device__ __forceinline__ float quad_elem<uint16_t>(const uint2 &w, const uint2 &,
                                                                 int e) {
  const uint32_t x = (e < 2) ? w.x : w.y;
  return (e & 1) ? bf_hi(x) : bf_lo(x);
}
template <> __device__ __forceinline__ float quad_elem<float>(const uint2 &lo, const uint2 &hi,
                                                              int e) {
  const uint32_t x = e == 0 ? lo.x : e == 1 ? lo.y : e == 2 ? hi.x : hi.y;
  return __uint_as_float(x);
}

// Finishing kernel for probabilities: the same units as the stream kernel, grid-stride, so the
// write pass is spread evenly over every SM whatever the number of rows. A warp re-reads its
// unit (an L2 hit right after the stream pass) in groups of four elements, lane l taking groups
// l, l + 32, ..., so that each 16-byte store instruction of the warp covers 512 contiguous
// bytes of output; the row's C partials are combined while those loads are in flight. A row
// found invalid is written as NaN and reported once, by its chunk 0.
template <typename E, bool kGreedy>
__global__ void __launch_bounds__(kThreads, 2) finish_probs(Params p) {
  constexpr int kEPV = Elem<E>::kPerVec;
  constexpr int kQuads = kUnitVecs * kEPV / 4 / 32;   // groups of four per lane and unit
  wait_stream_kernel();
  const int lane = threadIdx.x & 31;
  const int W = gridDim.x * kWarps;
  const int V = p.V;
  const float c2 = p.c2;
  for (int unit = blockIdx.x * kWarps + (threadIdx.x >> 5); unit < p.units; unit += W) {
    const UnitId u = unit_id(p, unit);   // one logits row per batch row: u.b is the row
    const E *row = static_cast<const E *>(p.tgt) + static_cast<long long>(u.b) * V;
    const RowGeom g = row_geom<E>(row, V);
    const uint2 *part = p.ws_part + static_cast<long long>(u.b) * p.C;
    const uint2 w0 = (lane < p.C) ? ldcg_u2(part + lane)
                                  : make_uint2(0xff800000u, kGreedy ? 0x7fffffffu : 0u);
    // the unit's interior as groups of four: group q covers elements k0 + 4q .. k0 + 4q + 3
    const int k0 = g.h + u.chunk * kUnitVecs * kEPV;
    const int nq = min(kUnitVecs, g.nv - u.chunk * kUnitVecs) * kEPV / 4;
    const E *rq = row + k0;
    uint2 lo[kQuads], hi[kQuads];
#pragma unroll
    for (int i = 0; i < kQuads; ++i) {
      const int q = lane + 32 * i;
      if (q < nq) {
        if constexpr (sizeof(E) == 2) {
          lo[i] = ld_quad_raw<uint16_t>(rq + 4 * q);
        } else {
          const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(rq + 4 * q));
          lo[i] = make_uint2(v.x, v.y);
          hi[i] = make_uint2(v.z, v.w);
        }
      }
    }
    float eh = -INFINITY, et = -INFINITY;
    if (u.chunk == 0) {
      if (lane < g.h) eh = ld_elem<E>(row + lane);
      if (lane < g.tl) et = ld_elem<E>(row + g.h + g.nv * kEPV + lane);
    }
    float M = 0.f, iZ = 0.f;
    int gi = 0;
    bool ok;
    if constexpr (kGreedy) {
      float bv = __uint_as_float(w0.x);
      int bi = static_cast<int>(w0.y);
      for (int c = lane + 32; c < p.C; c += 32) {
        const uint2 w = ldcg_u2(part + c);
        arg_merge(bv, bi, __uint_as_float(w.x), static_cast<int>(w.y));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, off);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, off);
        arg_merge(bv, bi, v2, i2);
      }
      ok = arg_ok(bv);
      gi = bi;
    } else {
      float m = __uint_as_float(w0.x), s = __uint_as_float(w0.y);
      for (int c = lane + 32; c < p.C; c += 32) {
        const uint2 w = ldcg_u2(part + c);
        stat_merge(m, s, __uint_as_float(w.x), __uint_as_float(w.y), c2);
      }
      warp_stat_merge(m, s, c2);
      ok = stats_ok(m, s);
      M = m;
      iZ = __frcp_rn(s);
    }
    if (!ok && u.chunk == 0 && lane == 0) set_status(p.status, SPEC_ERR_NONFINITE);
    auto val = [&](float l, int k) -> float {
      if (!ok) return __int_as_float(0x7fc00000);
      if constexpr (kGreedy) return (k == gi) ? 1.f : 0.f;
      else return __fmul_rn(ex2_shift(l, M, c2), iZ);
    };
    float *out = p.out_probs + static_cast<long long>(u.b) * V;
    float *oq = out + k0;
    const bool vec_out = ((reinterpret_cast<uintptr_t>(oq) & 15u) == 0);
#pragma unroll
    for (int i = 0; i < kQuads; ++i) {
      const int q = lane + 32 * i;
      if (q < nq) {
        const int k = k0 + 4 * q;
        const float4 y = make_float4(val(quad_elem<E>(lo[i], hi[i], 0), k),
                                     val(quad_elem<E>(lo[i], hi[i], 1), k + 1),
                                     val(quad_elem<E>(lo[i], hi[i], 2), k + 2),
                                     val(quad_elem<E>(lo[i], hi[i], 3), k + 3));
        if (vec_out) {
          __stcs(reinterpret_cast<float4 *>(oq + 4 * q), y);
        } else {
          __stcs(oq + 4 * q, y.x);
          __stcs(oq + 4 * q + 1, y.y);
          __stcs(oq + 4 * q + 2, y.z);
          __stcs(oq + 4 * q + 3, y.w);
        }
      }
    }
    if (u.chunk == 0) {
      if (lane < g.h) __stcs(out + lane, val(eh, lane));
      const int kt = g.h + g.nv * kEPV + lane;
      if (lane < g.tl) __stcs(out + kt, val(et, kt));
    }
  }
}

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
// (out_v[r], out_i[r]) on lane 0. Lists are consumed.
template <int kK>
__device__ __forceinline__ void warp_take_topk(float (&lv)[kK], int (&li)[kK], int k, int lane,
                                               uint2 *out) {
  for (int r = 0; r < k; ++r) {
    float v = lv[0];
    int i = li[0];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
      const int i2 = __shfl_xor_sync(0xffffffffu, i, off);
      if (ranks_before(v2, i2, v, i)) { v = v2; i = i2; }
    }
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
  for (int unit = blockIdx.x * kWarps + warp; unit < p.units; unit += W) {
    const UnitId u = unit_id(p, unit);
    const E *row = static_cast<const E *>(p.tgt) + static_cast<long long>(u.b) * p.V;
    const RowGeom g = row_geom<E>(row, p.V);
    uint4 buf[kVPL];
    float eh, et;
    load_unit<E>(row, g, u.chunk, lane, buf, eh, et);
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
    // T: the k-th largest lane maximum (k rounds of a warp maximum; -inf if fewer lanes)
    float T = -INFINITY;
    {
      bool taken = !any_elem;
      for (int r = 0; r < k; ++r) {
        float v = taken ? -INFINITY : lm;
        int who = taken ? 32 : lane;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
          const int w2 = __shfl_xor_sync(0xffffffffu, who, off);
          if (ranks_before(v2, w2, v, who)) { v = v2; who = w2; }
        }
        if (who == lane) taken = true;
        T = v;
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

// One warp per row: the row's C*k unit candidates, merged.
template <int kK>
__global__ void __launch_bounds__(kThreads, 1) topk_finish(Params p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int row_i = blockIdx.x * kWarps + (threadIdx.x >> 5);
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
  for (int r = lane; r < k; r += 32) out[r] = invalid ? -1 : static_cast<int>(mine[r].y);
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
    for (int j = i; j >= 0; j = par[j]) mine[j >> 5] |= 1u << (j & 31);   // par[0] = -1 ends it
    for (int w = 0; w < W; ++w) out[static_cast<long long>(i) * W + w] = mine[w];
  }
}

// ------------------------------------------------------------------ row-resident probabilities
//
// When a row fits in the registers of a cluster of at most kMaxCluster CTAs, the probability
// helper is one kernel: the CTAs of cluster `row` load their share of the row once (groups of
// four elements, thread t taking groups t, t + 512, ..., so that loads and the 16-byte stores
// of the results are both contiguous across a warp), reduce it to softmax statistics (or an
// argmax) through warp shuffles, shared memory and, between CTAs, distributed shared memory,
// and write the probabilities straight from registers: one read and one write of the row, no
// partials in global memory, no second pass.
template <typename E>
constexpr int kResQuads = (sizeof(E) == 2) ? 16 : 8;   // groups of four per thread (64 KB/CTA)

template <typename E, bool kGreedy>
__global__ void __launch_bounds__(kThreads, 2) probs_resident(Params p) {
  namespace cg = cooperative_groups;
  constexpr int kEPV = Elem<E>::kPerVec;
  constexpr int kQ = kResQuads<E>;
  __shared__ float red_a[kWarps];
  __shared__ int red_i[kWarps];
  __shared__ float part_a, part_b;
  __shared__ int part_i;
  cg::cluster_group cl = cg::this_cluster();
  const int S = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int row_i = blockIdx.x / S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int V = p.V;
  const float c2 = p.c2;
  const E *row = static_cast<const E *>(p.tgt) + static_cast<long long>(row_i) * V;
  const RowGeom g = row_geom<E>(row, V);
  const int nq = g.nv * kEPV / 4;                       // interior groups of four
  const int per = (nq + S - 1) / S;
  const int qb = rank * per, qe = min(nq, qb + per);
  const E *rq = row + g.h;
  uint2 lo[kQ];
  uint2 hi[sizeof(E) == 4 ? kQ : 1];   // fp32 only: the upper two elements of each group
#pragma unroll
  for (int i = 0; i < kQ; ++i) {
    const int q = qb + tid + kThreads * i;
    if (q < qe) {
      if constexpr (sizeof(E) == 2) {
        lo[i] = ld_quad_raw<uint16_t>(rq + 4 * q);
      } else {
        const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(rq + 4 * q));
        lo[i] = make_uint2(v.x, v.y);
        hi[sizeof(E) == 4 ? i : 0] = make_uint2(v.z, v.w);
      }
    } else {
      lo[i] = make_uint2(Elem<E>::kNegInfWord, Elem<E>::kNegInfWord);
      if constexpr (sizeof(E) == 4) hi[i] = lo[i];
    }
  }
  // element e of group i, as fp32
  auto el = [&](int i, int e) -> float {
    if constexpr (sizeof(E) == 2) {
      const uint32_t x = (e < 2) ? lo[i].x : lo[i].y;
      return (e & 1) ? bf_hi_v(x) : bf_lo_v(x);
    } else {
      const uint32_t x = e == 0 ? lo[i].x : e == 1 ? lo[i].y : e == 2 ? hi[i].x : hi[i].y;
      return __uint_as_float(x);
    }
  };
  float eh = -INFINITY, et = -INFINITY;
  if (rank == 0) {
    if (tid < g.h) eh = ld_elem<E>(row + tid);
    if (tid < g.tl) et = ld_elem<E>(row + g.h + g.nv * kEPV + tid);
  }
  // this thread's elements, then the warp, the CTA and the cluster (all in fixed orders)
  float a = -INFINITY, bsum = 0.f;
  int ai = 0x7fffffff;
  if constexpr (kGreedy) {
    // the thread's maximum (NaN-propagating), then the lowest index holding it: head elements
    // precede the interior groups, which precede the tail
    a = fmax_nan(eh, et);
    if constexpr (sizeof(E) == 2) {
      uint32_t w = bmax2_nan(lo[0].x, lo[0].y);
#pragma unroll
      for (int i = 1; i < kQ; ++i) w = bmax2_nan(w, bmax2_nan(lo[i].x, lo[i].y));
      a = fmax_nan(a, fmax_nan(bf_lo(w), bf_hi(w)));
    } else {
#pragma unroll
      for (int i = 0; i < kQ; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) a = fmax_nan(a, el(i, e));
    }
    if (a == INFINITY) a = __int_as_float(0x7fc00000);
    if (a == a && a != -INFINITY) {
      if (eh == a) {
        ai = tid;
      } else {
#pragma unroll
        for (int i = kQ - 1; i >= 0; --i)
#pragma unroll
          for (int e = 3; e >= 0; --e)
            if (el(i, e) == a) ai = g.h + 4 * (qb + tid + kThreads * i) + e;
        if (ai == 0x7fffffff) ai = g.h + g.nv * kEPV + tid;   // the tail element
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, a, off);
      const int i2 = __shfl_xor_sync(0xffffffffu, ai, off);
      arg_merge(a, ai, v2, i2);
    }
  } else {
    a = fmax_nan(eh, et);
    if constexpr (sizeof(E) == 2) {
      uint32_t w = bmax2_nan(lo[0].x, lo[0].y);
#pragma unroll
      for (int i = 1; i < kQ; ++i) w = bmax2_nan(w, bmax2_nan(lo[i].x, lo[i].y));
      a = fmax_nan(a, fmax_nan(bf_lo(w), bf_hi(w)));
    } else {
#pragma unroll
      for (int i = 0; i < kQ; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) a = fmax_nan(a, el(i, e));
    }
    if (a != -INFINITY) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kQ; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          acc[e] = __fadd_rn(acc[e], ex2_shift(el(i, e), a, c2));
      bsum = __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3]));
      bsum = __fadd_rn(bsum, __fadd_rn(ex2_shift(eh, a, c2), ex2_shift(et, a, c2)));
    }
    warp_stat_merge(a, bsum, c2);
  }
  if (lane == 0) {
    red_a[warp] = a;
    if constexpr (kGreedy) red_i[warp] = ai;
    else red_i[warp] = __float_as_int(bsum);
  }
  __syncthreads();
  if (warp == 0) {
    float v = (lane < kWarps) ? red_a[lane] : -INFINITY;
    int w = (lane < kWarps) ? red_i[lane] : (kGreedy ? 0x7fffffff : 0);
    if constexpr (kGreedy) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
        const int i2 = __shfl_xor_sync(0xffffffffu, w, off);
        arg_merge(v, w, v2, i2);
      }
      if (lane == 0) { part_a = v; part_i = w; }
    } else {
      float z = __int_as_float(w);
      warp_stat_merge(v, z, c2);
      if (lane == 0) { part_a = v; part_b = z; }
    }
  }
  if (S > 1) {
    cl.sync();   // every CTA's partial written
    if (warp == 0) {
      float v = -INFINITY, z = 0.f;
      int w = 0x7fffffff;
      if (lane < S) {
        v = *cl.map_shared_rank(&part_a, lane);
        if constexpr (kGreedy) w = *cl.map_shared_rank(&part_i, lane);
        else z = *cl.map_shared_rank(&part_b, lane);
      }
      if constexpr (kGreedy) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
          const int i2 = __shfl_xor_sync(0xffffffffu, w, off);
          arg_merge(v, w, v2, i2);
        }
      } else {
        warp_stat_merge(v, z, c2);
      }
      __syncwarp();
      if (lane == 0) { red_a[0] = v; red_i[0] = kGreedy ? w : __float_as_int(z); }
    }
    cl.sync();   // every CTA has read its peers' partials
  } else {
    __syncthreads();
    if (tid == 0) { red_a[0] = part_a; red_i[0] = kGreedy ? part_i : __float_as_int(part_b); }
  }
  __syncthreads();
  const float M = red_a[0];
  const int gi = red_i[0];
  const float Z = __int_as_float(red_i[0]);
  const bool ok = kGreedy ? (arg_ok(M) && M != INFINITY) : stats_ok(M, Z);
  const float iZ = kGreedy ? 0.f : __frcp_rn(Z);
  if (!ok && rank == 0 && tid == 0) set_status(p.status, SPEC_ERR_NONFINITE);
  auto val = [&](float l, int k) -> float {
    if (!ok) return __int_as_float(0x7fc00000);
    if constexpr (kGreedy) return (k == gi) ? 1.f : 0.f;
    else return __fmul_rn(ex2_shift(l, M, c2), iZ);
  };
  float *out = p.out_probs + static_cast<long long>(row_i) * V;
  float *oq = out + g.h;
  const bool vec_out = ((reinterpret_cast<uintptr_t>(oq) & 15u) == 0);
#pragma unroll
  for (int i = 0; i < kQ; ++i) {
    const int q = qb + tid + kThreads * i;
    if (q < qe) {
      const int k = g.h + 4 * q;
      const float4 y = make_float4(val(el(i, 0), k),
                                   val(el(i, 1), k + 1),
                                   val(el(i, 2), k + 2),
                                   val(el(i, 3), k + 3));
      if (vec_out) {
        __stcs(reinterpret_cast<float4 *>(oq + 4 * q), y);
      } else {
        __stcs(oq + 4 * q, y.x);
        __stcs(oq + 4 * q + 1, y.y);
        __stcs(oq + 4 * q + 2, y.z);
        __stcs(oq + 4 * q + 3, y.w);
      }
    }
  }
  if (rank == 0) {
    if (tid < g.h) __stcs(out + tid, val(eh, tid));
    const int kt = g.h + g.nv * kEPV + tid;
    if (tid < g.tl) __stcs(out + kt, val(et, kt));
  }
}

// Finishing kernel for greedy chains and trees: one CTA per batch row.
template <typename E, int MODE>
__global__ void __launch_bounds__(kThreads, 2) finish_cta(Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float *scratch = reinterpret_cast<float *>(smem_raw);
  __shared__ TailShared sh;
  wait_stream_kernel();
  const int b = blockIdx.x;
  if constexpr (MODE == kChainGreedy) tail_chain_greedy(p, b, scratch, sh);
  else if (p.N <= 64) tail_tree_small(p, b, scratch);
  else tail_tree(p, b, scratch, sh);
}

}  // namespace specv

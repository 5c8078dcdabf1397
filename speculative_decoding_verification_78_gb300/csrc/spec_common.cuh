// spec_common.cuh -- constants, kernel parameters, element access, row geometry, and the per-unit
// reductions (softmax statistics, argmax) shared by every kernel.
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
  int tile_units;            // chain: units are 256-column tiles of the fused LM-head producer
                             // (not 4 KB stream units), so the bonus draw takes the full pass
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
// Order-preserving map of fp32 values to unsigned integers (negative bit patterns reversed, the
// sign bit set on the others): a < b as floats iff key(a) < key(b), -0 just below +0, and every
// NaN, whatever its sign bit, the largest key (above +inf). key_float undoes it (NaN comes back
// as 0x7fffffff).
__device__ __forceinline__ unsigned float_key(float f) {
  const unsigned b = __float_as_uint(f);
  const unsigned k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (f != f) ? 0xffffffffu : k;
}
__device__ __forceinline__ float key_float(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
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

// ------------------------------------------------------------------ paired fp32 arithmetic
//
// Blackwell's f32x2 instructions apply one operation to two fp32 values held in a register
// pair. Each half is rounded to nearest exactly like the scalar instruction, so paired code
// gives the same bits as the scalar code it replaces, with half the arithmetic instructions.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void up2(f32x2 v, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// ex2_shift of two values: 2^((x - m) * c2) for both halves of x (m2, c22: m and c2 twice)
__device__ __forceinline__ f32x2 ex2_shift2(f32x2 x, f32x2 m2, f32x2 c22) {
  float t0, t1;
  up2(mul2(sub2(x, m2), c22), t0, t1);
  return pk2(ex2(t0), ex2(t1));
}

__device__ __forceinline__ uint2 ldcg_u2(const uint2 *p) { return __ldcg(p); }
__device__ __forceinline__ float ldcg_f(const float *p) { return __ldcg(p); }

// Cluster barrier whose arrival publishes this CTA's earlier writes, including its stores into
// peers' shared memory, to every CTA of the cluster (release / acquire). The exchanges push:
// each CTA stores its value into a slot of every peer before the barrier, so after it every
// value is local and no CTA reads a peer's shared memory (a peer may then leave at once).
__device__ __forceinline__ void cluster_sync_publish() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// A CTA may touch a peer's shared memory only once that peer is known to be running. Every
// thread of a clustered kernel arrives here at entry (relaxed: nothing is published), and
// waits (cluster_started_wait) before its first store into a peer; by then the other CTAs have
// long arrived, so the wait costs almost nothing. The arrival and the wait are one barrier
// phase: the publish barrier that follows is the next one. A CTA that leaves without storing
// into peers (every CTA of its cluster takes the same path) never waits.
__device__ __forceinline__ void cluster_started_arrive() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_started_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void set_status(int32_t *status, int code) {
  atomicCAS(reinterpret_cast<int *>(status), 0, code);
}

// ------------------------------------------------------------------ the checked build
//
// SPEC_CHECK(p, cond) guards a memory access by an index the kernel computed. In the checked
// build (compiled with SPEC_CHECKED, libspec_verify_checked.so) a false condition records
// SPEC_ERR_CHECK in *status and the guarded access is skipped; in the normal build it is the
// constant true and costs nothing.
#ifdef SPEC_CHECKED
static __device__ __noinline__ void spec_check_failed(int32_t *status) {
  atomicCAS(reinterpret_cast<int *>(status), 0, SPEC_ERR_CHECK);
}
#define SPEC_CHECK(p, cond) ((cond) ? true : (spec_check_failed((p).status), false))
#else
#define SPEC_CHECK(p, cond) true
#endif

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
  if (!SPEC_CHECK(p, b >= 0 && b < p.B && r >= 0 && r < p.R)) b = r = 0;
  if (r < p.Rt)
    return static_cast<const E *>(p.tgt) + (static_cast<long long>(b) * p.Rt + r) * p.V;
  return static_cast<const E *>(p.drf) + (static_cast<long long>(b) * p.Rd + (r - p.Rt)) * p.V;
}

struct UnitId {
  int b, r, chunk;
};

// unit -> (batch row, row, chunk), 32-bit unsigned division only
__device__ __forceinline__ UnitId unit_id(const Params &p, int unit) {
  if (!SPEC_CHECK(p, unit >= 0 && unit < p.units)) unit = 0;
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

// The warp's combined pair on every lane: the maximum M in one redux.sync (NaN, then +inf,
// rank highest, so they still poison), then each lane's sum rescaled to M once and the scaled
// sums added by a butterfly (identical on every lane: each step adds the same two values).
__device__ __forceinline__ void warp_stat_merge(float &m, float &s, float c2) {
  const float M = key_float(__reduce_max_sync(0xffffffffu, float_key(m)));
  float t = (M == -INFINITY) ? 0.f : __fmul_rn(s, ex2_shift(m, M, c2));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, off));
  m = M;
  s = t;
}

template <typename E>
__device__ __forceinline__ void unit_stats(const uint4 (&buf)[kVPL], float eh, float et,
                                           float c2, float &m_out, float &s_out) {
  constexpr int kEPV = Elem<E>::kPerVec;
  const float m = unit_lane_max<E>(buf, eh, et);
  float s = 0.f;
  if (m != -INFINITY) {
    // four running sums (element e goes to sum e mod 4), two per paired instruction
    f32x2 a01 = pk2(0.f, 0.f), a23 = pk2(0.f, 0.f);
    const f32x2 m2 = pk2(m, m), c22 = pk2(c2, c2);
#pragma unroll
    for (int j = 0; j < kVPL; ++j)
#pragma unroll
      for (int e = 0; e < kEPV; e += 4) {
        a01 = add2(a01, ex2_shift2(pk2(vec_elem<E>(buf[j], e), vec_elem<E>(buf[j], e + 1)), m2, c22));
        a23 = add2(a23, ex2_shift2(pk2(vec_elem<E>(buf[j], e + 2), vec_elem<E>(buf[j], e + 3)), m2, c22));
      }
    float acc[4];
    up2(a01, acc[0], acc[1]);
    up2(a23, acc[2], acc[3]);
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
// Selects instead of branches: it sits in shuffle-reduction chains on the critical path.
__device__ __forceinline__ void arg_merge(float &v, int &i, float v2, int i2) {
  const bool nan = (v2 != v2) | (v != v);
  const bool take = (v2 > v) | ((v2 == v) & (i2 < i));
  i = take ? i2 : i;
  v = nan ? __int_as_float(0x7fc00000) : (take ? v2 : v);
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
  // the warp maximum as one redux.sync over an order-preserving integer image of the floats, in
  // which NaN ranks above +inf, so that it still poisons the unit
  float wm = key_float(__reduce_max_sync(0xffffffffu, float_key(lm)));
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
    idx = __reduce_min_sync(0xffffffffu, idx);
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

}  // namespace specv

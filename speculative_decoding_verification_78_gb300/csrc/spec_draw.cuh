// spec_draw.cuh -- the inverse-CDF draw of the correction / bonus token over the residual
// max(0, p - q) (or p alone): segment sums, block and warp scans, the pick.
#pragma once

#include "spec_common.cuh"

namespace specv {

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

// The row constants of a draw, each twice, for the paired form of resid.
struct ResidK {
  f32x2 Mt, iZt, Md, iZd, c2;
};
__device__ __forceinline__ ResidK resid_k(float Mt, float iZt, float Md, float iZd, float c2) {
  return ResidK{pk2(Mt, Mt), pk2(iZt, iZt), pk2(Md, Md), pk2(iZd, iZd), pk2(c2, c2)};
}

// resid of the 8 elements of one lane's slot (wq unused without Q), two elements per paired
// instruction: the same operations and roundings as resid, hence the same values.
template <typename E>
__device__ __forceinline__ void resid8(const uint4 (&wp)[2], const uint4 (&wq)[2], bool hasq,
                                       const ResidK &k, float (&r)[8]) {
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const f32x2 p =
        mul2(ex2_shift2(pk2(raw8_elem<E>(wp, e), raw8_elem<E>(wp, e + 1)), k.Mt, k.c2), k.iZt);
    if (!hasq) {
      up2(p, r[e], r[e + 1]);
      continue;
    }
    const f32x2 q =
        mul2(ex2_shift2(pk2(raw8_elem<E>(wq, e), raw8_elem<E>(wq, e + 1)), k.Md, k.c2), k.iZd);
    float d0, d1;
    up2(sub2(p, q), d0, d1);
    r[e] = fmaxf(d0, 0.f);
    r[e + 1] = fmaxf(d1, 0.f);
  }
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
  resid8<E>(wp, wq, Q != nullptr, resid_k(Mt, iZt, Md, iZd, c2), r);
  float ls = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) ls = __fadd_rn(ls, r[e]);
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
    const ResidK rk = resid_k(Mt, iZt, Md, iZd, c2);
#pragma unroll
    for (int t = 0; t < kSegIter; ++t) {
      float r[8];
      resid8<E>(wp[t], wq[t], Q != nullptr, rk, r);
      float ls = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ls = __fadd_rn(ls, r[e]);
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
// several segments are issued together (four at a time); for rows of at
// most four segments the residual values stay in registers, so the crossing element is found
// without reading the rows again.
template <typename E>
__device__ int draw_token_warp(const E *P, const E *Q, float Mt, float iZt, float Md, float iZd,
                               float c2, int V, float u) {
  constexpr int kMaxSeg = kWarpTailMaxV / kSeg;
  constexpr int kRegSeg = 4;                          // segments kept in registers
  constexpr int kBatch = 4;                           // segments whose loads fly together
  const int lane = threadIdx.x & 31;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(P) & 15u) == 0) &&
                      (!Q || (reinterpret_cast<uintptr_t>(Q) & 15u) == 0);
  const int nseg = (V + kSeg - 1) / kSeg;
  const bool keep = nseg <= kRegSeg;
  const ResidK rk = resid_k(Mt, iZt, Md, iZd, c2);
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
        float r8[8];
        resid8<E>(wp[q], wq[q], Q != nullptr, rk, r8);
        float ls = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          ls = __fadd_rn(ls, r8[e]);
          if (sg < kRegSeg) rr[sg < kRegSeg ? sg : 0][e] = r8[e];
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

}  // namespace specv

// spec_kernels.cuh -- the verification kernels: the stream kernel, the finishing kernels, and the
// probability helper (row-resident, or the stream kernel plus a write pass).
#pragma once

#include "spec_finish.cuh"

namespace specv {

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
  if (lane == 0 && SPEC_CHECK(p, unit >= 0 && unit < p.units)) p.ws_part[unit] = part;
  if constexpr (MODE == kChainSample) {
    if (x >= 0 && x < p.V) {
      const int vb = u.chunk * kUnitVecs;
      float val = 0.f;
      if (span_logit<E>(row, g, vb, vb + kUnitVecs, u.chunk == 0, x, lane, buf, &val) &&
          lane == 0 && SPEC_CHECK(p, u.b < p.B && u.r < p.R))
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
      if (!SPEC_CHECK(p, u.b >= 0 && u.b < p.B && i >= 0 && i < p.gamma)) return -1;
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
    if (!SPEC_CHECK(p, u.b < p.B && u.r < p.R && u.chunk < p.C)) continue;
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
// pushed into every CTA's shared memory before one cluster barrier; the CTA whose slice holds
// the crossing draws the token from its own segment sums and writes the outputs.
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
  __shared__ float s_tot[kMaxCluster];   // slice totals pushed by every CTA of the cluster
  __shared__ float s_pre[kMaxCluster + 1];
  cg::cluster_group cl = cg::this_cluster();
  const int S = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / S;
  cluster_started_arrive();   // the draw's exchange waits for it before touching peers
  wait_stream_kernel();
  if (!SPEC_CHECK(p, b < p.B)) return;   // the same on every CTA of the cluster
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
    if (g.h == 0 && g.tl == 0 && !p.tile_units) {
      if (rank == 0 && threadIdx.x < 32)
        bonus_draw_units<E>(p, b, n, rowM[n], rowZ[n], bonus_part, xs);
      return;
    }
  }
  cluster_draw<E>(p, b, n, rowM, rowZ, xs, segsum, sh, s_tot, s_pre);
}

// Finishing kernel for sampling (gamma = 0, so every row's draw is the bonus draw from p_0) when
// every row starts and ends on a 16-byte boundary: one warp per row, in CTAs of any number of
// warps. The warp combines the row's C unit partials (staging them in shared memory), then
// bonus_draw_units finds the unit where the running mass crosses u * S from those partials and
// the element inside it from one 4 KB read of the row: no pass over the row.
template <typename E>
__global__ void __launch_bounds__(kThreads, 1) finish_sample_warp(Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  wait_stream_kernel();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int b = blockIdx.x * static_cast<int>(blockDim.x >> 5) + w;
  if (b >= p.B) return;
  const int C = p.C;
  uint2 *part = reinterpret_cast<uint2 *>(smem_raw) + static_cast<long long>(w) * C;
  const uint2 *src = p.ws_part + static_cast<long long>(b) * C;   // one row per batch row
  const uint2 none = make_uint2(0xff800000u, 0u);
  float m = -INFINITY, s = 0.f;
  for (int c0 = 0; c0 < C; c0 += 128) {   // four loads in flight per lane, merged in order
    uint2 v[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int c = c0 + lane + 32 * t;
      v[t] = (c < C) ? ldcg_u2(src + c) : none;
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int c = c0 + lane + 32 * t;
      if (c < C) part[c] = v[t];
      stat_merge(m, s, __uint_as_float(v[t].x), __uint_as_float(v[t].y), p.c2);
    }
  }
  warp_stat_merge(m, s, p.c2);
  if (!stats_ok(m, s)) {
    if (lane == 0) set_status(p.status, SPEC_ERR_NONFINITE);
    fail_chain_row(p, b, lane, 32);
    return;
  }
  __syncwarp();   // the partials staged by every lane
  bonus_draw_units<E>(p, b, 0, m, s, part, nullptr);
}

// Finishing kernel for chain sampling when every row is a single unit (gamma <= 31, V <=
// kWarpTailMaxV): one warp per batch row; lane i holds rows i and i + 32 and the draft-token
// logits of position i. Launched with small CTAs (any number of warps each) so that the batch
// rows spread over every SM; each thread may use up to 128 registers, and the draw keeps the
// residual of the rows in registers.
template <typename E>
__global__ void __launch_bounds__(kThreads, 1) finish_chain_sample_warp(Params p) {
  wait_stream_kernel();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * static_cast<int>(blockDim.x >> 5) + (threadIdx.x >> 5);
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
    if (!SPEC_CHECK(p, u.b < p.B && nq >= 0 && k0 + 4 * nq <= V)) continue;
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
  __shared__ float in_a[kMaxCluster];   // the CTA partials of the cluster, pushed by each CTA
  __shared__ int in_b[kMaxCluster];
  cg::cluster_group cl = cg::this_cluster();
  const int S = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int row_i = blockIdx.x / S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (S > 1) cluster_started_arrive();   // waited for before the first store into a peer
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int V = p.V;
  const float c2 = p.c2;
  const E *row = static_cast<const E *>(p.tgt) +
                 static_cast<long long>(SPEC_CHECK(p, row_i < p.B) ? row_i : 0) * V;
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
      // (scalar: the paired form of this pass measured slower here, unlike the write pass)
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
  if (S > 1) cluster_started_wait();   // every peer is running before warp 0 stores into it
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
      if (S == 1 && lane == 0) { red_a[0] = v; red_i[0] = w; }
      // push this CTA's partial (the same on every lane after the butterfly) into slot
      // `rank` of every CTA of the cluster
      if (S > 1 && lane < S) {
        *cl.map_shared_rank(&in_a[rank], lane) = v;
        *cl.map_shared_rank(&in_b[rank], lane) = w;
      }
    } else {
      float z = __int_as_float(w);
      warp_stat_merge(v, z, c2);
      if (S == 1 && lane == 0) { red_a[0] = v; red_i[0] = __float_as_int(z); }
      if (S > 1 && lane < S) {
        *cl.map_shared_rank(&in_a[rank], lane) = v;
        *cl.map_shared_rank(&in_b[rank], lane) = __float_as_int(z);
      }
    }
  }
  if (S > 1) {
    // one barrier: afterwards every partial is local and no CTA touches a peer's memory again
    cluster_sync_publish();
    if (warp == 0) {
      float v = (lane < S) ? in_a[lane] : -INFINITY;
      int w = (lane < S) ? in_b[lane] : (kGreedy ? 0x7fffffff : 0);
      if constexpr (kGreedy) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
          const int i2 = __shfl_xor_sync(0xffffffffu, w, off);
          arg_merge(v, w, v2, i2);
        }
        if (lane == 0) { red_a[0] = v; red_i[0] = w; }
      } else {
        float z = __int_as_float(w);
        warp_stat_merge(v, z, c2);
        if (lane == 0) { red_a[0] = v; red_i[0] = __float_as_int(z); }
      }
    }
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
  const f32x2 M2 = pk2(M, M), c22 = pk2(c2, c2), iZ2 = pk2(iZ, iZ);
  // the four probabilities of group i: val() of each element, two per paired instruction
  auto val4 = [&](int i, int k) -> float4 {
    if (kGreedy || !ok)
      return make_float4(val(el(i, 0), k), val(el(i, 1), k + 1), val(el(i, 2), k + 2),
                         val(el(i, 3), k + 3));
    float4 y;
    up2(mul2(ex2_shift2(pk2(el(i, 0), el(i, 1)), M2, c22), iZ2), y.x, y.y);
    up2(mul2(ex2_shift2(pk2(el(i, 2), el(i, 3)), M2, c22), iZ2), y.z, y.w);
    return y;
  };
#pragma unroll
  for (int i = 0; i < kQ; ++i) {
    const int q = qb + tid + kThreads * i;
    if (q < qe) {
      const int k = g.h + 4 * q;
      const float4 y = val4(i, k);
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
  if (!SPEC_CHECK(p, b < p.B)) return;
  if constexpr (MODE == kChainGreedy) tail_chain_greedy(p, b, scratch, sh);
  else if (p.N <= 64) tail_tree_small(p, b, scratch);
  else tail_tree(p, b, scratch, sh);
}

}  // namespace specv

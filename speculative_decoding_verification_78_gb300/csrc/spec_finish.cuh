// spec_finish.cuh -- what the finishing kernels do after the stream pass: combining unit
// partials into row results, the acceptance test, emitting a step, greedy chains and trees,
// and the cluster draws.
#pragma once

#include "spec_draw.cuh"

namespace specv {

// ------------------------------------------------------------------ finishing helpers

__device__ __forceinline__ void fail_chain_row(const Params &p, int b, int tid, int nthreads) {
  if (!SPEC_CHECK(p, b >= 0 && b < p.B)) return;
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

// Lanes that combine one row's unit partials: the smallest power of two L with 2L >= C (at most
// 32), so that each lane merges at most two partials (when C <= 64) before log2(L) shuffle
// rounds inside its group of L lanes; a warp combines 32 / L rows at once. Short dependent
// chains matter here: this runs after the stream pass, on the critical path of every call.
__device__ __forceinline__ int combine_lanes(int C) {
  int L = 1;
  while (L < 32 && 2 * L < C) L <<= 1;
  return L;
}

// Combines the unit partials of every row of batch row b into per-row statistics (rowM, rowZ
// in shared memory). Each warp takes 32 / L rows per pass and two passes per round trip: all
// of a round's loads are issued before any is merged. Partials beyond the first 2L of a row
// (C > 64) are merged four per lane per round trip, in a fixed order.
//
// keep (may be NULL): the unit partials of row keep_row are also copied there (C entries).
__device__ __forceinline__ void combine_rows_stats(const Params &p, int b, float *rowM,
                                                   float *rowZ, uint2 *keep = nullptr,
                                                   int keep_row = -1) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = p.R, C = p.C;
  const int L = combine_lanes(C);
  const int sub = lane & (L - 1), rpw = 32 / L, pass = kWarps * rpw;
  if (!SPEC_CHECK(p, b >= 0 && b < p.B)) b = 0;
  const uint2 *base = p.ws_part + static_cast<long long>(b) * R * C;
  const uint2 none = make_uint2(0xff800000u, 0u);
  for (int r0 = warp * rpw; r0 < R; r0 += 2 * pass) {
    uint2 v[2][2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int r = r0 + q * pass + lane / L;
      const uint2 *pr = base + static_cast<long long>(r) * C;
      v[q][0] = (r < R && sub < C) ? ldcg_u2(pr + sub) : none;
      v[q][1] = (r < R && sub + L < C) ? ldcg_u2(pr + sub + L) : none;
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (r0 + q * pass >= R) break;   // warp-uniform
      const int r = r0 + q * pass + lane / L;
      const bool kp = keep && r == keep_row;
      if (kp) {
        if (sub < C) keep[sub] = v[q][0];
        if (sub + L < C) keep[sub + L] = v[q][1];
      }
      float m = -INFINITY, s = 0.f;
      stat_merge(m, s, __uint_as_float(v[q][0].x), __uint_as_float(v[q][0].y), p.c2);
      stat_merge(m, s, __uint_as_float(v[q][1].x), __uint_as_float(v[q][1].y), p.c2);
      const uint2 *pr = base + static_cast<long long>(r) * C;
      for (int c0 = sub + 2 * L; c0 < C + sub; c0 += 4 * L) {   // C > 64 only (then L = 32)
        uint2 w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          w[t] = (r < R && c0 + t * L < C) ? ldcg_u2(pr + c0 + t * L) : none;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (kp && c0 + t * L < C) keep[c0 + t * L] = w[t];
          stat_merge(m, s, __uint_as_float(w[t].x), __uint_as_float(w[t].y), p.c2);
        }
      }
      // the group's pair: its maximum (NaN-propagating), then each lane's sum rescaled to it
      // once and the scaled sums added, both by butterflies inside the group of L lanes
      float M = m;
      for (int off = L >> 1; off > 0; off >>= 1) M = fmax_nan(M, __shfl_xor_sync(0xffffffffu, M, off));
      float t = (M == -INFINITY) ? 0.f : __fmul_rn(s, ex2_shift(m, M, p.c2));
      for (int off = L >> 1; off > 0; off >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, off));
      if (r < R && sub == 0) { rowM[r] = M; rowZ[r] = t; }
    }
  }
}

// Same for greedy argmax partials: g[r] = lowest index of the row maximum, ok[r] = the row is
// usable (finite maximum, no NaN / +inf seen).
__device__ __forceinline__ void combine_rows_arg(const Params &p, int b, int *g, int *ok) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = p.R, C = p.C;
  const int L = combine_lanes(C);
  const int sub = lane & (L - 1), rpw = 32 / L, pass = kWarps * rpw;
  if (!SPEC_CHECK(p, b >= 0 && b < p.B)) b = 0;
  const uint2 *base = p.ws_part + static_cast<long long>(b) * R * C;
  const uint2 none = make_uint2(0xff800000u, 0x7fffffffu);
  for (int r0 = warp * rpw; r0 < R; r0 += 2 * pass) {
    uint2 v[2][2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int r = r0 + q * pass + lane / L;
      const uint2 *pr = base + static_cast<long long>(r) * C;
      v[q][0] = (r < R && sub < C) ? ldcg_u2(pr + sub) : none;
      v[q][1] = (r < R && sub + L < C) ? ldcg_u2(pr + sub + L) : none;
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (r0 + q * pass >= R) break;   // warp-uniform
      const int r = r0 + q * pass + lane / L;
      float bv = -INFINITY;
      int bi = 0x7fffffff;
      arg_merge(bv, bi, __uint_as_float(v[q][0].x), static_cast<int>(v[q][0].y));
      arg_merge(bv, bi, __uint_as_float(v[q][1].x), static_cast<int>(v[q][1].y));
      const uint2 *pr = base + static_cast<long long>(r) * C;
      for (int c0 = sub + 2 * L; c0 < C + sub; c0 += 4 * L) {   // C > 64 only (then L = 32)
        uint2 w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
          w[t] = (r < R && c0 + t * L < C) ? ldcg_u2(pr + c0 + t * L) : none;
#pragma unroll
        for (int t = 0; t < 4; ++t)
          arg_merge(bv, bi, __uint_as_float(w[t].x), static_cast<int>(w[t].y));
      }
      for (int off = L >> 1; off > 0; off >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, off);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, off);
        arg_merge(bv, bi, v2, i2);
      }
      if (r < R && sub == 0) { g[r] = bi; ok[r] = arg_ok(bv) ? 1 : 0; }
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
  if (!SPEC_CHECK(p, b >= 0 && b < p.B && n >= 0 && n <= p.gamma)) return;
  (void)SPEC_CHECK(p, tok >= 0 && tok < p.V);
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
        int a = anc[j];
        if (!SPEC_CHECK(p, a >= 0 && a < N)) a = 0;
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
  if (threadIdx.x == 0 && SPEC_CHECK(p, best >= 0 && best < N && D >= 0 && D < N)) {
    int v = best;
    for (int d = D; d >= 0; --d) {
      if (!SPEC_CHECK(p, v >= 0 && v < N)) break;
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
// the rest without block barriers. Acceptance and depth come from pointer jumping: each node
// keeps (ancestor, edges to it, all of those edges matched) and composes it with its ancestor's
// triple, so a tree of depth D takes ceil(log2(D + 1)) rounds of shuffles. The deepest accepted
// node is one warp maximum; the path is walked back through parents staged in shared memory,
// one lane per depth.
// smem holds g[N], the row-usable flags okf[N], then parents and tokens [N] each.
__device__ inline void tail_tree_small(const Params &p, int b, float *smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int N = p.N;
  int *g = reinterpret_cast<int *>(smem);
  int *okf = g + N;
  int *par_s = okf + N;
  int *tok_s = par_s + N;
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
  // the first failing check of a node: 1 its row is not usable, 2 a bad parent, 3 a bad token;
  // the tree's error is the smallest over its nodes
  auto check = [&](int j, bool in, int par, int tok) -> int {
    if (!in) return 4;
    if (okf[j] == 0) return 1;
    if (j == 0 ? (par != -1) : (par < 0 || par >= j)) return 2;
    if (j > 0 && (tok < 0 || tok >= p.V)) return 3;
    return 4;
  };
  const int first = __reduce_min_sync(0xffffffffu, min(check(j0, in0, par0, tok0),
                                                       check(j1, in1, par1, tok1)));
  int32_t *pn = p.path_nodes + bN;
  int32_t *ot = p.out_tokens + bN;
  if (first < 4) {
    if (in0) { pn[j0] = -1; ot[j0] = -1; }
    if (in1) { pn[j1] = -1; ot[j1] = -1; }
    if (lane == 0) {
      set_status(p.status, first == 1 ? SPEC_ERR_NONFINITE
                                      : (first == 2 ? SPEC_ERR_PARENT : SPEC_ERR_TOKEN));
      p.accept_len[b] = -1;
    }
    return;
  }
  if (in0) { par_s[j0] = par0; tok_s[j0] = tok0; }
  if (in1) { par_s[j1] = par1; tok_s[j1] = tok1; }
  // node state: bits 0..6 ancestor + 1 (0: past the root), 7..13 edges to it, 14 all matched
  auto pack = [](int anc, int dep, bool ok) -> int {
    return (anc + 1) | (dep << 7) | (ok ? (1 << 14) : 0);
  };
  int s0 = pack(-1, 0, in0);   // the root (j0 == 0) is accepted at depth 0
  if (in0 && j0 > 0) s0 = pack(par0, 1, tok0 == g[par0]);
  int s1 = in1 ? pack(par1, 1, tok1 == g[par1]) : pack(-1, 0, false);
  for (;;) {
    const int a0 = (s0 & 127) - 1, a1 = (s1 & 127) - 1;
    if (!__any_sync(0xffffffffu, a0 >= 0 || a1 >= 0)) break;
    // every lane reads the old states of both ancestors before any state changes
    const int x0 = __shfl_sync(0xffffffffu, s0, a0 & 31), y0 = __shfl_sync(0xffffffffu, s1, a0 & 31);
    const int x1 = __shfl_sync(0xffffffffu, s0, a1 & 31), y1 = __shfl_sync(0xffffffffu, s1, a1 & 31);
    const int t0 = (a0 >= 32) ? y0 : x0, t1 = (a1 >= 32) ? y1 : x1;
    // compose: the ancestor's ancestor, the summed edge counts, both chains matched
    // (depths add without carry: a tree of at most 64 nodes is at most 63 deep)
    constexpr int kDep = 127 << 7;
    if (a0 >= 0) s0 = (t0 & 127) | ((s0 & kDep) + (t0 & kDep)) | (s0 & t0 & (1 << 14));
    if (a1 >= 0) s1 = (t1 & 127) | ((s1 & kDep) + (t1 & kDep)) | (s1 & t1 & (1 << 14));
  }
  // deepest accepted node, smallest index on equal depth (the root is always accepted)
  auto key = [](int s, int j) -> unsigned {
    return (s & (1 << 14)) ? ((static_cast<unsigned>((s >> 7) & 127) << 11) | (2047u - j)) + 1u
                           : 0u;
  };
  const unsigned kmax = __reduce_max_sync(0xffffffffu, max(key(s0, j0), in1 ? key(s1, j1) : 0u));
  const int best = 2047 - static_cast<int>((kmax - 1u) & 2047u);
  const int D = static_cast<int>((kmax - 1u) >> 11);
  if (in0 && j0 > D) { pn[j0] = -1; ot[j0] = -1; }
  if (in1 && j1 > D) { pn[j1] = -1; ot[j1] = -1; }
  __syncwarp();   // parents and tokens staged
  // lane d writes the path node at depth d (and d + 32): D - d steps up from the deepest node
  for (int d = lane; d <= D; d += 32) {
    int v = best;
    for (int k = d; k < D; ++k) v = SPEC_CHECK(p, v >= 0 && v < N) ? par_s[v] : 0;
    if (!SPEC_CHECK(p, v >= 0 && v < N && d < N)) break;
    pn[d] = v;
    if (d > 0) ot[d - 1] = tok_s[v];
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
  if (!SPEC_CHECK(p, uc_sel >= 0 && uc_sel < C)) uc_sel = 0;
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
// them in registers. Warp totals -> CTA total, pushed into every peer's shared memory before
// one cluster barrier -> cluster prefix; then the warp whose range holds u*S picks the token
// from its registers and writes the outputs, with no second pass over the rows and no block
// barrier after the cluster's.
template <typename E>
__device__ __forceinline__ void cluster_draw_regs(const Params &p, int b, int n, const E *P, const E *Q, float Mt,
                                  float iZt, float Md, float iZd, float u, const int *xs, int K,
                                  float *segsum, TailShared &sh, float *s_tot) {
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
  const ResidK rk = resid_k(Mt, iZt, Md, iZd, c2);
  float lsum[kSI], ssum[kSI];
  float wtot = 0.f;
#pragma unroll
  for (int t = 0; t < kSI; ++t) {
    float r8[8];
    resid8<E>(wp[t], wq[t], Q != nullptr, rk, r8);
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ls = __fadd_rn(ls, r8[e]);
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
  // push this CTA's slice total into slot `rank` of every CTA of the cluster (every peer has
  // started: the entry arrival's phase completes here), then one barrier: afterwards every
  // total is local, and no CTA touches a peer's shared memory again
  cluster_started_wait();
  if (warp == 0 && lane < S) *cl.map_shared_rank(&s_tot[rank], lane) = ctot;
  cluster_sync_publish();
  // every warp: the cluster prefix (lane r holds rank r's inclusive prefix)
  float pre = (lane < S) ? s_tot[lane] : 0.f;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, pre, off);
    if (lane >= off) pre = __fadd_rn(pre, y);
  }
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
      resid8<E>(wp[q], wq[q], Q != nullptr, rk, r);
      ls = lsum[q];
    }
  int tok = segment_pick(r, ls, (s0 + seg) * kSeg + lane * 8, segbase, t, smode, lane);
  if (tok < 0) tok = V - 1;   // unreachable when the slice holds mass
  emit_chain(p, b, n, tok, xs, lane, 32);
}

// The correction / bonus draw of chain sampling over a thread-block cluster of S CTAs (S = 1:
// no cluster), after acceptance gave n: CTA `rank` sums r(k) = max(0, p_n(k) - q_n(k)) (or
// p_gamma(k)) over its slice of 256-element segments into segsum (shared memory); each CTA
// pushes its slice total into every peer's shared memory before one cluster barrier; the CTA
// whose slice holds u * S picks the token and writes the outputs. Every CTA of the cluster calls
// it; CTAs other than the writer return from it early.
template <typename E>
__device__ void cluster_draw(const Params &p, int b, int n, const float *rowM, const float *rowZ,
                             const int *xs, float *segsum, TailShared &sh, float *s_tot,
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
    cluster_draw_regs<E>(p, b, n, P, Q, Mt, iZt, Md, iZd, u, xs, K, segsum, sh, s_tot);
    return;
  }
  const int lo = min(nseg, rank * K), hi = min(nseg, lo + K), nl = hi - lo;
  segment_sums<E>(P, Q, Mt, iZt, Md, iZd, p.c2, p.V, lo, hi, segsum, lo);
  __syncthreads();
  cluster_started_wait();   // every peer is running before any store into its shared memory
  if (threadIdx.x < 32) {   // slice total: strided lane sums, then a fixed xor tree
    float tot = 0.f;
    for (int j = threadIdx.x; j < nl; j += 32) tot = __fadd_rn(tot, segsum[j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot = __fadd_rn(tot, __shfl_xor_sync(0xffffffffu, tot, off));
    if (threadIdx.x < S) *cl.map_shared_rank(&s_tot[rank], threadIdx.x) = tot;
  }
  cluster_sync_publish();   // every slice total pushed to every CTA
  if (threadIdx.x < 32) {   // lane r holds rank r's total; inclusive scan in rank order
    const int r = threadIdx.x;
    float v = (r < S) ? s_tot[r] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, v, off);
      if (r >= off) v = __fadd_rn(v, y);
    }
    if (r < S) s_pre[r + 1] = v;
    if (r == 0) s_pre[0] = 0.f;
  }
  __syncthreads();   // local only: no CTA reads a peer's shared memory after the barrier
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

}  // namespace specv

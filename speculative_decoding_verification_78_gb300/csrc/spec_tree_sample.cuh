// spec_tree_sample.cuh -- stochastic (T > 0) tree verification: the walk of the candidate tree by
// sequential per-sibling rejection sampling.
//
// At the current node the children are tested in index order against a distribution r that
// starts as the target's p at the node: child c with token x is accepted when u_c <= r(x)/q(x)
// (q: the drafter's distribution at the node); a rejection replaces r by
// norm(max(0, r - q)). An accepted child becomes the current node; when every child is rejected
// (or the node has none) the last token is drawn from r by inverse CDF. r is never stored: after
// j rejections r(k) = max(0, ... max(0, p(k) - q(k)) / S_1 ... - q(k)) / S_j, recomputed from
// the two logits at k and the normalisers S_1 .. S_j, each of which took one pass over the
// node's two rows.
//
// The stream kernel has already reduced every target and draft row of every node to softmax
// statistics (rows 0 .. N-1 target, N .. 2N-1 draft); one CTA per tree combines them and walks.
#pragma once

#include <cooperative_groups.h>

#include "spec_finish.cuh"

namespace specv {

constexpr int kTsMaxUpdates = SPEC_MAX_NODES;   // residual updates of one node: one per child

// r at one element: p, then the node's residual updates so far
__device__ __forceinline__ float ts_weight(float p, float q, const float *invS, int nS) {
  float r = p;
  for (int i = 0; i < nS; ++i) r = __fmul_rn(fmaxf(__fsub_rn(r, q), 0.f), invS[i]);
  return r;
}

// p and q of the 8 elements [k0, k0 + 8) of the node's two rows (-inf beyond V: p = q = 0)
template <typename E>
__device__ __forceinline__ void ts_load8(const E *P, const E *Q, int k0, int V, bool vec_ok,
                                         float Mt, float iZt, float Md, float iZd, float c2,
                                         float (&pp)[8], float (&qq)[8]) {
  uint4 wp[2], wq[2];
  load8_raw<E>(P, k0, V, vec_ok, wp);
  load8_raw<E>(Q, k0, V, vec_ok, wq);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    pp[e] = __fmul_rn(ex2_shift(raw8_elem<E>(wp, e), Mt, c2), iZt);
    qq[e] = __fmul_rn(ex2_shift(raw8_elem<E>(wq, e), Md, c2), iZd);
  }
}

struct TsShared {
  int cur, depth, nchild, next, nS, err, token;
  float u0;
  float Mt, iZt, Md, iZd;
  float red[kWarps];
  float invS[kTsMaxUpdates];
  float lt[SPEC_MAX_NODES], ld[SPEC_MAX_NODES];   // logits at the children's tokens
  float off[kWarps + 1];
  int seg, mode;
  float base;
};

// Sum over the node's rows of the weight `next` (an update: max(0, r - q); else r itself) in a
// fixed order: lanes sum their 8 elements, warps their segments (segment s = 256 elements,
// warp s % kWarps), then the warps in order. With `segsum`, each segment's sum is also stored.
template <typename E>
__device__ float ts_pass(const E *P, const E *Q, int V, bool vec_ok, const TsShared &sh,
                         float c2, bool update, float *segsum, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nseg = (V + kSeg - 1) / kSeg;
  float wsum = 0.f;
  for (int s = warp; s < nseg; s += kWarps) {
    float pp[8], qq[8];
    ts_load8<E>(P, Q, s * kSeg + lane * 8, V, vec_ok, sh.Mt, sh.iZt, sh.Md, sh.iZd, c2, pp, qq);
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float r = ts_weight(pp[e], qq[e], sh.invS, sh.nS);
      ls = __fadd_rn(ls, update ? fmaxf(__fsub_rn(r, qq[e]), 0.f) : r);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ls = __fadd_rn(ls, __shfl_xor_sync(0xffffffffu, ls, off));
    if (segsum && lane == 0) segsum[s] = ls;
    wsum = __fadd_rn(wsum, ls);
  }
  if (lane == 0) red[warp] = wsum;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < kWarps; ++w) tot = __fadd_rn(tot, red[w]);
  __syncthreads();   // red is reused by the next pass
  return tot;
}

// The inverse-CDF draw from r over the node's rows with u: the first k whose running sum
// strictly exceeds u * S (S: the sum of the segment sums in order), or, when rounding leaves
// none, the last k with r(k) > 0. segsum: shared memory, ceil(V / kSeg) floats.
template <typename E>
__device__ int ts_draw(const E *P, const E *Q, int V, bool vec_ok, TsShared &sh, float c2,
                       float u, float *segsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nseg = (V + kSeg - 1) / kSeg;
  ts_pass<E>(P, Q, V, vec_ok, sh, c2, false, segsum, sh.red);
  // the segments' inclusive prefix sums in index order: thread t takes segments
  // [t*K, (t+1)*K) sequentially, a warp scan, then the warps' offsets
  const int K = (nseg + kThreads - 1) / kThreads;
  const int tl = threadIdx.x * K, th = min(nseg, tl + K);
  float local = 0.f;
  for (int j = tl; j < th; ++j) local = __fadd_rn(local, segsum[j]);
  float incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl = __fadd_rn(incl, y);
  }
  if (lane == 31) sh.red[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    float v = lane < kWarps ? sh.red[lane] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v = __fadd_rn(v, y);
    }
    if (lane < kWarps) sh.off[lane + 1] = v;
    if (lane == 0) { sh.off[0] = 0.f; sh.seg = -1; }
  }
  __syncthreads();
  const float S = sh.off[kWarps];
  const float t = __fmul_rn(u, S);
  int mode = t < S ? 0 : 1;
  if (mode == 0) {
    const float up = __shfl_up_sync(0xffffffffu, incl, 1);
    const float ex = lane == 0 ? sh.off[warp] : __fadd_rn(sh.off[warp], up);
    const float in = __fadd_rn(sh.off[warp], incl);
    if (tl < th && ex <= t && t < in) {
      float acc = ex;
      int found = -1;
      for (int j = tl; j < th; ++j) {
        const float nx = __fadd_rn(acc, segsum[j]);
        if (nx > t) { found = j; break; }
        acc = nx;
      }
      if (found >= 0) { sh.seg = found; sh.base = acc; }
    }
  }
  __syncthreads();
  if (sh.seg < 0) {   // no crossing (rounding): the last segment holding mass
    int last = -1;
    for (int j = tl; j < th; ++j)
      if (segsum[j] > 0.f) last = j;
    last = block_max_int(last, reinterpret_cast<int *>(sh.red));
    if (threadIdx.x == 0) { sh.seg = max(last, 0); sh.base = 0.f; }
    mode = 1;
    __syncthreads();
  }
  if (warp == 0) {
    const int seg = sh.seg;
    float pp[8], qq[8], r[8];
    ts_load8<E>(P, Q, seg * kSeg + lane * 8, V, vec_ok, sh.Mt, sh.iZt, sh.Md, sh.iZd, c2, pp, qq);
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      r[e] = ts_weight(pp[e], qq[e], sh.invS, sh.nS);
      ls = __fadd_rn(ls, r[e]);
    }
    int tok = segment_pick(r, ls, seg * kSeg + lane * 8, sh.base, t, mode, lane);
    if (tok < 0) tok = V - 1;   // unreachable: the segment holds mass
    if (lane == 0) sh.token = tok;
  }
  __syncthreads();
  return sh.token;
}

// Finishing kernel of stochastic tree verification: one CTA per tree (blockIdx.x = b). Dynamic
// shared memory: rowM, rowZ [2N], parents, tokens [N], the current node's children [N], segment
// sums [ceil(V / kSeg)].
template <typename E>
__global__ void __launch_bounds__(kThreads, 1) finish_tree_sample(Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int N = p.N, V = p.V, R = p.R;
  float *rowM = reinterpret_cast<float *>(smem_raw);
  float *rowZ = rowM + R;
  int *par = reinterpret_cast<int *>(rowZ + R);
  int *tok = par + N;
  int *ch = tok + N;
  float *segsum = reinterpret_cast<float *>(ch + N);
  __shared__ TsShared sh;
  wait_stream_kernel();
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long bN = static_cast<long long>(b) * N;
  const float c2 = p.c2;
  if (tid == 0) {
    sh.err = 0;
    sh.u0 = p.uniforms[bN];
  }
  for (int j = tid; j < N; j += kThreads) {
    par[j] = p.parents[bN + j];
    tok[j] = j == 0 ? 0 : p.tokens[bN + j];
  }
  combine_rows_stats(p, b, rowM, rowZ);
  __syncthreads();
  // the oracle's order of checks: parents, then tokens, then rows
  int e1 = 0, e2 = 0, e3 = 0;
  for (int j = tid; j < N; j += kThreads) {
    if (j == 0 ? par[j] != -1 : (par[j] < 0 || par[j] >= j)) e1 = 1;
    if (j > 0 && (tok[j] < 0 || tok[j] >= V)) e2 = 1;
  }
  for (int r = tid; r < R; r += kThreads)
    if (!stats_ok(rowM[r], rowZ[r])) e3 = 1;
  e1 = __syncthreads_or(e1);
  e2 = __syncthreads_or(e2);
  e3 = __syncthreads_or(e3);
  int32_t *pn = p.path_nodes + bN;
  int32_t *ot = p.out_tokens + bN;
  const int err = e1 ? SPEC_ERR_PARENT : e2 ? SPEC_ERR_TOKEN : e3 ? SPEC_ERR_NONFINITE : 0;
  for (int j = tid; j < N; j += kThreads) { pn[j] = -1; ot[j] = -1; }
  if (err) {
    if (tid == 0) { set_status(p.status, err); p.accept_len[b] = -1; }
    return;
  }
  if (tid == 0) { sh.cur = 0; sh.depth = 0; }
  __syncthreads();
  for (;;) {
    const int cur = sh.cur;
    const E *P = row_ptr<E>(p, b, cur);
    const E *Q = row_ptr<E>(p, b, N + cur);
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(P) & 15u) == 0) &&
                        ((reinterpret_cast<uintptr_t>(Q) & 15u) == 0);
    // the children of cur in index order (a block-wide compaction), their tokens' logits in
    // the node's two rows (one round trip for all of them)
    int is_child = 0, rank_in = 0;
    {
      int base = 0;
      for (int j0 = 0; j0 < N; j0 += kThreads) {
        const int j = j0 + tid;
        is_child = (j < N && j > cur && par[j] == cur) ? 1 : 0;
        const unsigned bal = __ballot_sync(0xffffffffu, is_child);
        if (lane == 0) sh.red[warp] = __int_as_float(__popc(bal));
        __syncthreads();
        int before = base;
        for (int w = 0; w < warp; ++w) before += __float_as_int(sh.red[w]);
        rank_in = before + __popc(bal & ((1u << lane) - 1u));
        if (is_child) ch[rank_in] = j;
        int total = 0;
        for (int w = 0; w < kWarps; ++w) total += __float_as_int(sh.red[w]);
        base += total;
        __syncthreads();
      }
      if (tid == 0) {
        sh.nchild = base;
        sh.next = -1;
        sh.nS = 0;
        sh.Mt = rowM[cur];
        sh.iZt = __frcp_rn(rowZ[cur]);
        sh.Md = rowM[N + cur];
        sh.iZd = __frcp_rn(rowZ[N + cur]);
      }
    }
    __syncthreads();
    const int nc = sh.nchild;
    for (int i = tid; i < nc; i += kThreads) {
      const int c = ch[i];
      const int x = SPEC_CHECK(p, c > cur && c < N) ? tok[c] : 0;
      if (!SPEC_CHECK(p, x >= 0 && x < V && i < SPEC_MAX_NODES)) continue;
      sh.lt[i] = ld_elem<E>(P + x);
      sh.ld[i] = ld_elem<E>(Q + x);
    }
    __syncthreads();
    for (int i = 0; i < nc; ++i) {
      // the test of child i (the same on every thread)
      const int c = ch[i];
      const float px = __fmul_rn(ex2_shift(sh.lt[i], sh.Mt, c2), sh.iZt);
      const float qx = __fmul_rn(ex2_shift(sh.ld[i], sh.Md, c2), sh.iZd);
      const float rx = ts_weight(px, qx, sh.invS, sh.nS);
      const float ratio = qx > 0.f ? __fdiv_rn(rx, qx) : (rx > 0.f ? INFINITY : 0.f);
      const float uc = p.uniforms[bN + c];
      if (uc <= ratio) {
        if (tid == 0) sh.next = c;
        break;
      }
      // rejected: one pass for the mass of max(0, r - q); the next sibling's test uses it
      const float S = ts_pass<E>(P, Q, V, vec_ok, sh, c2, true, nullptr, sh.red);
      if (S > 0.f && tid == 0 && sh.nS < kTsMaxUpdates) {
        sh.invS[sh.nS] = __frcp_rn(S);
        sh.nS = sh.nS + 1;
      }
      __syncthreads();
    }
    __syncthreads();
    const int next = sh.next;
    if (next >= 0) {
      if (tid == 0 && SPEC_CHECK(p, next < N && sh.depth + 1 < N)) {
        const int d = sh.depth + 1;
        pn[d] = next;
        ot[d - 1] = tok[next];
        sh.depth = d;
        sh.cur = next;
      }
      __syncthreads();
      continue;
    }
    const int t = ts_draw<E>(P, Q, V, vec_ok, sh, c2, sh.u0, segsum);
    if (tid == 0 && SPEC_CHECK(p, t >= 0 && t < V && sh.depth < N)) {
      pn[0] = 0;
      ot[sh.depth] = t;
      p.accept_len[b] = sh.depth;
    }
    return;
  }
}

// ------------------------------------------------------------------ the walk over a cluster

// The walk with one thread-block cluster of S CTAs per tree (blockIdx.x = b * S + rank): every
// CTA runs the walk's control (the same decisions: they combine the same statistics, load the
// same children's logits and reduce the same totals in the same order), and CTA `rank` owns
// the vocabulary slice of segments [rank * nsl, (rank + 1) * nsl). At each visited node a CTA
// computes p and q of its slice once into shared memory (fp32); every pass after that (each
// rejection's residual mass, the final draw's segment sums) reads them there. A pass's slice
// totals are pushed into every CTA of the cluster (two alternating slot arrays, so one cluster
// barrier per pass) and summed in rank order. The final draw's crossing is found from the
// slice totals; the CTA holding it picks the token. Rank 0 writes the path and the outputs.
// Dynamic shared memory: rowM, rowZ [2N]; parents, tokens, children [N]; the slice's segment
// sums [nsl]; then (16-byte aligned) p and q of the slice, nsl * kSeg floats each.
struct TsClusterShared {
  float tot[2][kMaxCluster];   // slice totals of the last two passes, by rank
};

// p and q of this CTA's slice [k_lo, k_lo + 8 * ngroups) into shared memory (0 past V): groups of
// 8 elements, four groups per thread in flight.
template <typename E>
__device__ __forceinline__ void tsc_stage(const E *P, const E *Q, int V, int k_lo, int ngroups,
                                          float Mt, float iZt, float Md, float iZd, float c2,
                                          float *ps, float *qs) {
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(P) | reinterpret_cast<uintptr_t>(Q)) & 15u) == 0;
  for (int g0 = threadIdx.x; g0 < ngroups; g0 += 4 * kThreads) {
    uint4 wp[4][2], wq[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * kThreads;
      const int k0 = g < ngroups ? k_lo + 8 * g : V;   // past V: -inf, p = q = 0
      load8_raw<E>(P, k0, V, vec_ok, wp[u]);
      load8_raw<E>(Q, k0, V, vec_ok, wq[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * kThreads;
      if (g >= ngroups) continue;
      float pv[8], qv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        pv[e] = __fmul_rn(ex2_shift(raw8_elem<E>(wp[u], e), Mt, c2), iZt);
        qv[e] = __fmul_rn(ex2_shift(raw8_elem<E>(wq[u], e), Md, c2), iZd);
      }
      float4 *pd = reinterpret_cast<float4 *>(ps + 8 * g);
      float4 *qd = reinterpret_cast<float4 *>(qs + 8 * g);
      pd[0] = make_float4(pv[0], pv[1], pv[2], pv[3]);
      pd[1] = make_float4(pv[4], pv[5], pv[6], pv[7]);
      qd[0] = make_float4(qv[0], qv[1], qv[2], qv[3]);
      qd[1] = make_float4(qv[4], qv[5], qv[6], qv[7]);
    }
  }
}

// Asks L2 for this CTA's slice [k_lo, k_lo + n) of one row, one 128-byte line per thread and
// step (a hint: nothing waits for it), so that a later tsc_stage of the row finds it there.
template <typename E>
__device__ __forceinline__ void tsc_prefetch(const E *row, int V, int k_lo, int n) {
  constexpr int kLine = 128 / static_cast<int>(sizeof(E));
  const int hi = min(V, k_lo + n);
  for (int k = k_lo + static_cast<int>(threadIdx.x) * kLine; k < hi; k += kThreads * kLine)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + k));
}

// This CTA's slice total of the pass's weight (the update max(0, r - q), or r itself), in a fixed
// order: a lane's 8 elements, the warp's segments (segment j of the slice: warp j % kWarps),
// then the warps in order. With `segsum`, each segment's sum is stored too.
__device__ __forceinline__ float tsc_slice_pass(const float *ps, const float *qs, int nsl,
                                                const TsShared &sh, bool update, float *segsum,
                                                float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float wsum = 0.f;
  for (int j = warp; j < nsl; j += kWarps) {
    const float4 *pa = reinterpret_cast<const float4 *>(ps + j * kSeg + lane * 8);
    const float4 *qa = reinterpret_cast<const float4 *>(qs + j * kSeg + lane * 8);
    const float4 p0 = pa[0], p1 = pa[1], q0 = qa[0], q1 = qa[1];
    const float pp[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    const float qq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float ls = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float r = ts_weight(pp[e], qq[e], sh.invS, sh.nS);
      ls = __fadd_rn(ls, update ? fmaxf(__fsub_rn(r, qq[e]), 0.f) : r);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ls = __fadd_rn(ls, __shfl_xor_sync(0xffffffffu, ls, off));
    if (segsum && lane == 0) segsum[j] = ls;
    wsum = __fadd_rn(wsum, ls);
  }
  if (lane == 0) red[warp] = wsum;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < kWarps; ++w) tot = __fadd_rn(tot, red[w]);
  __syncthreads();   // red is reused by the next pass
  return tot;
}

// Pushes this CTA's slice total into slot array `buf` of every CTA of the cluster, then one
// cluster barrier; returns the S totals' sum in rank order, and (in `before`) the sum of the
// totals of the ranks below this one.
__device__ __forceinline__ float tsc_allreduce(float mine, int buf, TsClusterShared &cs, int S,
                                               int rank) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  if (threadIdx.x < static_cast<unsigned>(S)) {
    float *dst = cl.map_shared_rank(&cs.tot[buf][rank], static_cast<int>(threadIdx.x));
    *dst = mine;
  }
  cl.sync();
  float t = 0.f;
  for (int r = 0; r < S; ++r) t = __fadd_rn(t, cs.tot[buf][r]);
  return t;
}

template <typename E>
__global__ void __launch_bounds__(kThreads, 1) finish_tree_sample_cluster(Params p) {
  namespace cg = cooperative_groups;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  cg::cluster_group cl = cg::this_cluster();
  const int S = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int N = p.N, V = p.V, R = p.R;
  const int nseg = (V + kSeg - 1) / kSeg;
  const int nsl = (nseg + S - 1) / S;
  if (!SPEC_CHECK(p, S >= 1 && S <= kMaxCluster)) return;   // the same on every CTA
  const int k_lo = rank * nsl * kSeg;
  float *rowM = reinterpret_cast<float *>(smem_raw);
  float *rowZ = rowM + R;
  int *par = reinterpret_cast<int *>(rowZ + R);
  int *tok = par + N;
  int *ch = tok + N;
  float *segsum = reinterpret_cast<float *>(ch + N);
  float *ps = reinterpret_cast<float *>(
      (reinterpret_cast<uintptr_t>(segsum + nsl) + 15) & ~static_cast<uintptr_t>(15));
  float *qs = ps + nsl * kSeg;
  __shared__ TsShared sh;
  __shared__ TsClusterShared cs;
  cluster_started_arrive();   // the first push waits for it before touching peers
  const int b = blockIdx.x / S;
  // the root's rows are inputs (the stream kernel only reads them): ask L2 for this CTA's slices
  // while the stream kernel drains
  if (b < p.B) {
    tsc_prefetch<E>(row_ptr<E>(p, b, 0), V, k_lo, nsl * kSeg);
    tsc_prefetch<E>(row_ptr<E>(p, b, N), V, k_lo, nsl * kSeg);
  }
  wait_stream_kernel();
  if (!SPEC_CHECK(p, b < p.B)) return;   // the same on every CTA of the cluster
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long bN = static_cast<long long>(b) * N;
  const float c2 = p.c2;
  if (tid == 0) sh.u0 = p.uniforms[bN];
  for (int j = tid; j < N; j += kThreads) {
    par[j] = p.parents[bN + j];
    tok[j] = j == 0 ? 0 : p.tokens[bN + j];
  }
  combine_rows_stats(p, b, rowM, rowZ);
  __syncthreads();
  // the oracle's order of checks: parents, then tokens, then rows
  int e1 = 0, e2 = 0, e3 = 0;
  for (int j = tid; j < N; j += kThreads) {
    if (j == 0 ? par[j] != -1 : (par[j] < 0 || par[j] >= j)) e1 = 1;
    if (j > 0 && (tok[j] < 0 || tok[j] >= V)) e2 = 1;
  }
  for (int r = tid; r < R; r += kThreads)
    if (!stats_ok(rowM[r], rowZ[r])) e3 = 1;
  e1 = __syncthreads_or(e1);
  e2 = __syncthreads_or(e2);
  e3 = __syncthreads_or(e3);
  int32_t *pn = p.path_nodes + bN;
  int32_t *ot = p.out_tokens + bN;
  const int err = e1 ? SPEC_ERR_PARENT : e2 ? SPEC_ERR_TOKEN : e3 ? SPEC_ERR_NONFINITE : 0;
  if (rank == 0)
    for (int j = tid; j < N; j += kThreads) { pn[j] = -1; ot[j] = -1; }
  if (err) {   // the same on every CTA of the cluster: all of them leave here
    if (rank == 0 && tid == 0) { set_status(p.status, err); p.accept_len[b] = -1; }
    return;
  }
  cluster_started_wait();
  if (tid == 0) { sh.cur = 0; sh.depth = 0; }
  __syncthreads();
  int pass = 0;   // cluster passes so far: selects the slot array
  for (;;) {
    const int cur = sh.cur;
    const E *P = row_ptr<E>(p, b, cur);
    const E *Q = row_ptr<E>(p, b, N + cur);
    // the children of cur in index order (a block-wide compaction)
    {
      int base = 0;
      for (int j0 = 0; j0 < N; j0 += kThreads) {
        const int j = j0 + tid;
        const int is_child = (j < N && j > cur && par[j] == cur) ? 1 : 0;
        const unsigned bal = __ballot_sync(0xffffffffu, is_child);
        if (lane == 0) sh.red[warp] = __int_as_float(__popc(bal));
        __syncthreads();
        int before = base;
        for (int w = 0; w < warp; ++w) before += __float_as_int(sh.red[w]);
        const int rank_in = before + __popc(bal & ((1u << lane) - 1u));
        if (is_child && SPEC_CHECK(p, rank_in < N)) ch[rank_in] = j;
        int total = 0;
        for (int w = 0; w < kWarps; ++w) total += __float_as_int(sh.red[w]);
        base += total;
        __syncthreads();
      }
      if (tid == 0) {
        sh.nchild = base;
        sh.next = -1;
        sh.nS = 0;
        sh.Mt = rowM[cur];
        sh.iZt = __frcp_rn(rowZ[cur]);
        sh.Md = rowM[N + cur];
        sh.iZd = __frcp_rn(rowZ[N + cur]);
      }
    }
    __syncthreads();
    // the children's token logits: the first kThreads into registers before the slice is staged,
    // so that their loads overlap the staging's, stored once it is done
    const int nc = sh.nchild;
    float lt0 = 0.f, ld0 = 0.f;
    bool have0 = false;
    if (tid < nc) {
      const int c = ch[tid];
      const int x = SPEC_CHECK(p, c > cur && c < N) ? tok[c] : 0;
      if (SPEC_CHECK(p, x >= 0 && x < V && tid < SPEC_MAX_NODES)) {
        lt0 = ld_elem<E>(P + x);
        ld0 = ld_elem<E>(Q + x);
        have0 = true;
      }
    }
    tsc_stage<E>(P, Q, V, k_lo, nsl * (kSeg / 8), sh.Mt, sh.iZt, sh.Md, sh.iZd, c2, ps, qs);
    if (have0) {
      sh.lt[tid] = lt0;
      sh.ld[tid] = ld0;
    }
    for (int i = tid + kThreads; i < nc; i += kThreads) {
      const int c = ch[i];
      const int x = SPEC_CHECK(p, c > cur && c < N) ? tok[c] : 0;
      if (!SPEC_CHECK(p, x >= 0 && x < V && i < SPEC_MAX_NODES)) continue;
      sh.lt[i] = ld_elem<E>(P + x);
      sh.ld[i] = ld_elem<E>(Q + x);
    }
    __syncthreads();
    for (int i = 0; i < nc; ++i) {
      // the test of child i (the same on every thread of every CTA)
      const int c = ch[i];
      const float px = __fmul_rn(ex2_shift(sh.lt[i], sh.Mt, c2), sh.iZt);
      const float qx = __fmul_rn(ex2_shift(sh.ld[i], sh.Md, c2), sh.iZd);
      const float rx = ts_weight(px, qx, sh.invS, sh.nS);
      const float ratio = qx > 0.f ? __fdiv_rn(rx, qx) : (rx > 0.f ? INFINITY : 0.f);
      const float uc = p.uniforms[bN + c];
      if (uc <= ratio) {
        if (tid == 0) sh.next = c;
        break;
      }
      // rejected: the mass of max(0, r - q) over the vocabulary, for the next sibling's test
      const float mine = tsc_slice_pass(ps, qs, nsl, sh, true, nullptr, sh.red);
      const float St = tsc_allreduce(mine, pass & 1, cs, S, rank);
      ++pass;
      if (St > 0.f && tid == 0 && sh.nS < kTsMaxUpdates) {
        sh.invS[sh.nS] = __frcp_rn(St);
        sh.nS = sh.nS + 1;
      }
      __syncthreads();
    }
    __syncthreads();
    const int next = sh.next;
    if (next >= 0) {
      if (tid == 0 && SPEC_CHECK(p, next < N && sh.depth + 1 < N)) {
        const int d = sh.depth + 1;
        if (rank == 0) {
          pn[d] = next;
          ot[d - 1] = tok[next];
        }
        sh.depth = d;
        sh.cur = next;
      }
      __syncthreads();
      continue;
    }
    // the draw from r with u0: slice totals and segment sums, the slices' prefix in rank order
    const float mine = tsc_slice_pass(ps, qs, nsl, sh, false, segsum, sh.red);
    const int buf = pass & 1;
    const float Stot = tsc_allreduce(mine, buf, cs, S, rank);
    float off = 0.f;
    for (int r = 0; r < rank; ++r) off = __fadd_rn(off, cs.tot[buf][r]);
    const float t = __fmul_rn(sh.u0, Stot);
    // the CTA whose slice holds the crossing (ex <= t < in), else (rounding: no crossing) the
    // highest rank with mass, which takes the last element with r > 0
    int owner = -1, mode = 0;
    {
      float acc = 0.f;
      for (int r = 0; r < S; ++r) {
        const float nx = __fadd_rn(acc, cs.tot[buf][r]);
        if (t < Stot && acc <= t && t < nx) { owner = r; break; }
        acc = nx;
      }
      if (owner < 0) {
        mode = 1;
        for (int r = S - 1; r >= 0; --r)
          if (cs.tot[buf][r] > 0.f) { owner = r; break; }
        if (owner < 0) owner = 0;
      }
    }
    if (rank != owner) return;
    // the segment of the crossing within this slice (one thread scans the segment sums)
    if (tid == 0) {
      int seg = -1;
      float base = off;
      if (mode == 0) {
        float acc = off;
        for (int j = 0; j < nsl; ++j) {
          const float nx = __fadd_rn(acc, segsum[j]);
          if (nx > t) { seg = j; base = acc; break; }
          acc = nx;
        }
      }
      if (seg < 0) {
        mode = 1;
        for (int j = nsl - 1; j >= 0; --j)
          if (segsum[j] > 0.f) { seg = j; break; }
        if (seg < 0) seg = 0;
      }
      sh.seg = seg;
      sh.base = base;
      sh.mode = mode;
    }
    __syncthreads();
    if (warp == 0 && SPEC_CHECK(p, sh.seg >= 0 && sh.seg < nsl)) {
      const int seg = sh.seg;
      const float4 *pa = reinterpret_cast<const float4 *>(ps + seg * kSeg + lane * 8);
      const float4 *qa = reinterpret_cast<const float4 *>(qs + seg * kSeg + lane * 8);
      const float4 p0 = pa[0], p1 = pa[1], q0 = qa[0], q1 = qa[1];
      const float pp[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      const float qq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
      float r[8], ls = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        r[e] = ts_weight(pp[e], qq[e], sh.invS, sh.nS);
        ls = __fadd_rn(ls, r[e]);
      }
      const int k0 = k_lo + seg * kSeg + lane * 8;
      int tk = segment_pick(r, ls, k0, sh.base, t, sh.mode, lane);
      if (tk < 0 || tk >= V) tk = V - 1;   // unreachable: the segment holds mass
      if (lane == 0 && SPEC_CHECK(p, sh.depth < N)) {
        pn[0] = 0;
        ot[sh.depth] = tk;
        p.accept_len[b] = sh.depth;
      }
    }
    return;
  }
}

}  // namespace specv

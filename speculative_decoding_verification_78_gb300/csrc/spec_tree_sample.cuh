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

}  // namespace specv

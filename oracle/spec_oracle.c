/*
 * spec_oracle.c -- CPU oracle of the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's CPU-baseline leg
 * load this file's library; the product path (the CUDA library and its Python binding) never
 * does. It shares no code, header, table or constant with the CUDA library.
 *
 * Plain, slow, single-threaded C in double precision, written as the method reads, one step
 * after another, so that it can be checked against the pages by eye:
 *
 *   "Fast Inference from Transformers via Speculative Decoding" (Leviathan, Kalman, Matias;
 *   pith.science review, sections "The pith", "Core claim", "What carries the argument",
 *   "Desk Editor's Note", "Referee Report: Significance", "Circularity Check") describes the
 *   step: a draft model proposes gamma tokens, the target model scores all of them in one
 *   parallel pass, the longest prefix that passes a rejection-sampling test on the target's
 *   own probabilities is accepted, and a distribution-preserving correction makes the output
 *   an exact sample of the target.
 *
 *   The precise rule (the standard one that makes that claim true, and the one this build
 *   takes): p = softmax(target logits / T), q = softmax(draft logits / T); draft token x_i is
 *   accepted while u_i <= p_i(x_i) / q_i(x_i); at the first rejection n the emitted token is
 *   drawn from norm(max(0, p_n - q_n)); if all gamma drafts pass, one more token is drawn
 *   from p_gamma.
 *
 *   "Falcon: Faster and Parallel Inference of Large Language Models through Enhanced
 *   Semi-Autoregressive Drafting and Custom-Designed Decoding Tree" (pith.science review,
 *   sections "What carries the argument", "Core claim", Figure 3 "SAR decoding tree
 *   attention", Figure 4 "greedy (temperature=0)") verifies a tree of drafts in one pass
 *   under greedy decoding: a node survives when its token equals the target's argmax at its
 *   parent and its parent survives; the deepest surviving node's root path is accepted.
 *
 * Readings taken where the pages are silent (each is also listed in the design notes):
 *   - accept on equality (u <= ratio); uniforms lie strictly in (0,1);
 *   - q(x) = 0: ratio = +inf if p(x) > 0, else 0 (so a token neither model allows is rejected);
 *   - inverse CDF: the first index whose inclusive running sum strictly exceeds u * S;
 *   - a residual whose sum is exactly 0 falls back to p_n;
 *   - T = 0: p and q are one-hot at the lowest-index argmax; the draft logits are not used
 *     (x_i is accepted iff it equals the target argmax, the correction and the bonus token
 *     are target argmaxes);
 *   - a logits row is invalid if it holds NaN or +inf or has no finite entry (-inf entries,
 *     i.e. masked tokens, are allowed); a draft token outside [0, V) is invalid; an invalid
 *     batch row reports accept_len = -1 and all its out_tokens = -1;
 *   - tree: parents[0] = -1 and 0 <= parents[i] < i; node 0 is the committed root; ties in
 *     depth go to the smallest node index; the bonus token is the argmax at the deepest
 *     accepted node.
 *
 * Margins: for every draw the oracle reports how close it was to a decision boundary, so
 * tests can separate draws that any correct fp32 implementation must reproduce from the
 * rare ones that rounding may legitimately flip:
 *   decision margin  |u_i - ratio_i| / max(ratio_i, 1e-300)
 *   CDF margin       min(c_k - t, t - c_{k-1}) / P at the chosen index k, t = u * S, where P
 *                    is the scale of the operands the CDF is built from: P = sum of p_n over
 *                    the indices where r > 0 (for the bonus draw r = p_gamma, so P = S = 1).
 *                    The residual r = max(0, p_n - q_n) is a difference of two unit-mass
 *                    distributions; rounding in p and q moves its CDF by an amount that scales
 *                    with P, not with the residual's own mass S, which can be far smaller.
 * A batch row's margin is the minimum over its draws (+inf when it made none, e.g. T = 0).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_OK 0
#define ORC_ERR_ROW (-1)    /* NaN / +inf / no finite logit in a row      */
#define ORC_ERR_TOKEN (-2)  /* draft or node token outside [0, V)          */
#define ORC_ERR_PARENT (-3) /* tree parent index not in [0, i), or root != -1 */
#define ORC_ERR_ARG (-4)    /* bad sizes or temperature                    */
#define ORC_ERR_MEM (-5)

/* ------------------------------------------------------------------ logits access */

/* Value of element idx of a logits tensor, as a double. bf16 is widened exactly: its 16 bits
 * are the upper half of the fp32 with the same value. */
static double logit_at(const void *base, int dtype, size_t idx) {
  if (dtype == ORC_F32) return (double)((const float *)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* 1 if the row [off, off+V) has no NaN, no +inf and at least one finite value. */
static int row_valid(const void *base, int dtype, size_t off, long V) {
  int any_finite = 0;
  for (long k = 0; k < V; ++k) {
    double v = logit_at(base, dtype, off + (size_t)k);
    if (isnan(v) || v == INFINITY) return 0;
    if (isfinite(v)) any_finite = 1;
  }
  return any_finite;
}

/* Lowest index holding the row maximum. */
static long argmax_row(const void *base, int dtype, size_t off, long V) {
  long best = 0;
  double bv = logit_at(base, dtype, off);
  for (long k = 1; k < V; ++k) {
    double v = logit_at(base, dtype, off + (size_t)k);
    if (v > bv) { bv = v; best = k; }
  }
  return best;
}

/* Temperature softmax of one (valid) row: p[k] = exp((l[k]-m)/T) / sum_j exp((l[j]-m)/T),
 * m = max_k l[k], sums in index order. T == 0: one-hot at the lowest-index argmax. */
static void softmax_row(const void *base, int dtype, size_t off, long V, double T, double *p) {
  if (T == 0.0) {
    long g = argmax_row(base, dtype, off, V);
    for (long k = 0; k < V; ++k) p[k] = 0.0;
    p[g] = 1.0;
    return;
  }
  double m = -INFINITY;
  for (long k = 0; k < V; ++k) {
    double v = logit_at(base, dtype, off + (size_t)k);
    if (v > m) m = v;
  }
  double Z = 0.0;
  for (long k = 0; k < V; ++k) {
    p[k] = exp((logit_at(base, dtype, off + (size_t)k) - m) / T);
    Z += p[k];
  }
  for (long k = 0; k < V; ++k) p[k] /= Z;
}

/* Inverse-CDF draw from the unnormalised weights r[0..V): the first k whose inclusive running
 * sum c_k strictly exceeds t = u * S, S = sum r (index order). If rounding leaves no such k,
 * the last k with r[k] > 0. Writes the CDF margin relative to `scale` (see Margins above). */
static long inverse_cdf(const double *r, long V, double u, double scale, double *margin) {
  double S = 0.0;
  for (long k = 0; k < V; ++k) S += r[k];
  double t = u * S;
  double c = 0.0;
  for (long k = 0; k < V; ++k) {
    double prev = c;
    c += r[k];
    if (c > t) {
      double a = c - t, b = t - prev;
      *margin = (a < b ? a : b) / scale;
      return k;
    }
  }
  *margin = 0.0;
  for (long k = V - 1; k >= 0; --k)
    if (r[k] > 0.0) return k;
  return V - 1;
}

/* ------------------------------------------------------------------ public: probabilities */

/* out[rows, V] = temperature softmax of each logits row (one-hot at the argmax for T == 0).
 * Invalid rows are filled with NaN. Returns 0, or ORC_ERR_ROW if any row was invalid. */
int oracle_probs(const void *logits, int dtype, long rows, long V, double T, double *out) {
  if (rows < 0 || V < 1 || !(T >= 0.0) || isinf(T)) return ORC_ERR_ARG;
  int rc = ORC_OK;
  for (long r = 0; r < rows; ++r) {
    size_t off = (size_t)r * (size_t)V;
    if (!row_valid(logits, dtype, off, V)) {
      for (long k = 0; k < V; ++k) out[off + (size_t)k] = NAN;
      rc = ORC_ERR_ROW;
      continue;
    }
    softmax_row(logits, dtype, off, V, T, out + off);
  }
  return rc;
}

/* Lowest-index argmax of each row; -1 for an invalid row. */
int oracle_argmax(const void *logits, int dtype, long rows, long V, int32_t *out) {
  if (rows < 0 || V < 1) return ORC_ERR_ARG;
  int rc = ORC_OK;
  for (long r = 0; r < rows; ++r) {
    size_t off = (size_t)r * (size_t)V;
    if (!row_valid(logits, dtype, off, V)) { out[r] = -1; rc = ORC_ERR_ROW; continue; }
    out[r] = (int32_t)argmax_row(logits, dtype, off, V);
  }
  return rc;
}

/* ------------------------------------------------------------------ public: chain verify */

static void fail_row(int32_t *accept_len, int32_t *out_tokens, long b, long gamma) {
  accept_len[b] = -1;
  for (long j = 0; j <= gamma; ++j) out_tokens[b * (gamma + 1) + j] = -1;
}

/*
 * Batched chain verify.
 *   target   [B, gamma+1, V] logits of the target at positions 0..gamma
 *   draft    [B, gamma, V]   logits of the draft at positions 0..gamma-1 (unused at T == 0)
 *   tokens   [B, gamma]      draft tokens x_0..x_{gamma-1}
 *   uniforms [B, gamma+1]    u_0..u_{gamma-1} acceptance tests, u_gamma the final draw
 * Outputs: accept_len[B] = n (number of accepted drafts), out_tokens[B, gamma+1] =
 * x_0..x_{n-1}, then the correction (n < gamma) or bonus (n == gamma) token, then -1;
 * margin[B] (may be NULL). Returns 0 or the first error code met.
 */
int oracle_verify_chain(const void *target, const void *draft, int dtype, const int32_t *tokens,
                        const float *uniforms, long B, long gamma, long V, double T,
                        int32_t *accept_len, int32_t *out_tokens, double *margin) {
  if (B < 0 || gamma < 0 || V < 1 || !(T >= 0.0) || isinf(T)) return ORC_ERR_ARG;
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  double *r = (double *)malloc(sizeof(double) * (size_t)V);
  if (!p || !q || !r) { free(p); free(q); free(r); return ORC_ERR_MEM; }
  int rc = ORC_OK;
  for (long b = 0; b < B; ++b) {
    const size_t trow0 = (size_t)b * (size_t)(gamma + 1);
    const size_t drow0 = (size_t)b * (size_t)gamma;
    const int32_t *x = tokens + (size_t)b * (size_t)gamma;
    const float *u = uniforms + (size_t)b * (size_t)(gamma + 1);
    if (margin) margin[b] = INFINITY;

    /* validate the whole batch row before any decision */
    int err = ORC_OK;
    for (long i = 0; i <= gamma && !err; ++i)
      if (!row_valid(target, dtype, (trow0 + (size_t)i) * (size_t)V, V)) err = ORC_ERR_ROW;
    if (T > 0.0)
      for (long i = 0; i < gamma && !err; ++i)
        if (!row_valid(draft, dtype, (drow0 + (size_t)i) * (size_t)V, V)) err = ORC_ERR_ROW;
    for (long i = 0; i < gamma && !err; ++i)
      if (x[i] < 0 || x[i] >= V) err = ORC_ERR_TOKEN;
    if (err) {
      fail_row(accept_len, out_tokens, b, gamma);
      if (rc == ORC_OK) rc = err;
      continue;
    }

    long n = gamma;
    long token;
    if (T == 0.0) {
      /* greedy: accept x_i iff it is the target argmax at position i */
      for (long i = 0; i < gamma; ++i) {
        long g = argmax_row(target, dtype, (trow0 + (size_t)i) * (size_t)V, V);
        if (x[i] != g) { n = i; break; }
      }
      token = argmax_row(target, dtype, (trow0 + (size_t)n) * (size_t)V, V);
    } else {
      double mg = INFINITY;
      for (long i = 0; i < gamma; ++i) {
        softmax_row(target, dtype, (trow0 + (size_t)i) * (size_t)V, V, T, p);
        softmax_row(draft, dtype, (drow0 + (size_t)i) * (size_t)V, V, T, q);
        double px = p[x[i]], qx = q[x[i]];
        double ratio = (qx > 0.0) ? px / qx : (px > 0.0 ? INFINITY : 0.0);
        double ui = (double)u[i];
        if (isfinite(ratio)) {
          double m = fabs(ui - ratio) / (ratio > 1e-300 ? ratio : 1e-300);
          if (m < mg) mg = m;
        }
        if (ui > ratio) { n = i; break; } /* first rejection ends the step */
      }
      double scale = 1.0;
      if (n < gamma) {
        /* p and q still hold position n: residual max(0, p - q) */
        double S = 0.0;
        scale = 0.0;
        for (long k = 0; k < V; ++k) {
          double d = p[k] - q[k];
          r[k] = d > 0.0 ? d : 0.0;
          S += r[k];
          if (r[k] > 0.0) scale += p[k];
        }
        if (S == 0.0) {
          for (long k = 0; k < V; ++k) r[k] = p[k];
          scale = 1.0;
        }
      } else {
        softmax_row(target, dtype, (trow0 + (size_t)gamma) * (size_t)V, V, T, r);
      }
      double cm;
      token = inverse_cdf(r, V, (double)u[gamma], scale, &cm);
      if (cm < mg) mg = cm;
      if (margin) margin[b] = mg;
    }

    accept_len[b] = (int32_t)n;
    int32_t *o = out_tokens + (size_t)b * (size_t)(gamma + 1);
    for (long j = 0; j < n; ++j) o[j] = x[j];
    o[n] = (int32_t)token;
    for (long j = n + 1; j <= gamma; ++j) o[j] = -1;
  }
  free(p); free(q); free(r);
  return rc;
}

/*
 * The band of one inverse-CDF draw: with c_k the inclusive running sums of r (index order,
 * c_{-1} = 0), S = c_{V-1} and t = u * S, the tokens k whose CDF cell [c_{k-1}, c_k] comes
 * within band * scale of t: c_k >= t - band * scale and c_{k-1} <= t + band * scale. The cells
 * are consecutive, so this is the index interval [*lo, *hi]; it holds the drawn token. A token
 * outside it needs a cumulative-sum error above band * scale to be drawn.
 */
static void cdf_band(const double *r, long V, double u, double scale, double band, long *lo,
                     long *hi) {
  double S = 0.0;
  for (long k = 0; k < V; ++k) S += r[k];
  const double t = u * S, w = band * scale;
  *lo = V - 1;
  *hi = 0;
  int seen = 0;
  double c = 0.0;
  for (long k = 0; k < V; ++k) {
    double prev = c;
    c += r[k];
    if (c >= t - w && prev <= t + w) {
      if (!seen) *lo = k;
      *hi = k;
      seen = 1;
    }
  }
}

/*
 * Per-position detail of batched chain verify, for tests that compare an implementation working
 * in fp32 with this one. oracle_verify_chain follows one path, the one the uniforms select;
 * here every batch row is evaluated at every position, as if the step had reached it, so that
 * a run whose path left the oracle's at a near-boundary decision can still be checked decision
 * by decision and draw by draw:
 *   accept[b, i]   i < gamma: 1 if u_i <= p_i(x_i) / q_i(x_i) (T == 0: x_i == argmax of target
 *                  row i), else 0
 *   dmargin[b, i]  |u_i - ratio_i| / ratio_i, as in oracle_verify_chain (+inf when the ratio is
 *                  +inf or 0, and at T == 0)
 *   tok[b, j]      j <= gamma: the token the step emits if it stops at position j -- for j <
 *                  gamma the correction drawn with u_gamma from norm(max(0, p_j - q_j)) (p_j if
 *                  that sums to 0), for j == gamma the bonus drawn from p_gamma (T == 0: the
 *                  argmax of target row j)
 *   cmargin[b, j]  the CDF margin of that draw (relative to P, as in oracle_verify_chain; +inf
 *                  at T == 0)
 *   lo[b, j], hi[b, j]  the draw's band (cdf_band) for the given band width (T == 0: the token)
 * The path oracle_verify_chain takes is n = the first i with accept[b, i] == 0 (or gamma);
 * its outputs are tok[b, n] after x_0..x_{n-1}. An invalid batch row gets accept = 0, margins
 * +inf and tok = lo = hi = -1. Returns 0 or the first error code met.
 */
int oracle_verify_chain_detail(const void *target, const void *draft, int dtype,
                               const int32_t *tokens, const float *uniforms, long B, long gamma,
                               long V, double T, double band, int32_t *accept, double *dmargin,
                               int32_t *tok, double *cmargin, int32_t *lo, int32_t *hi) {
  if (B < 0 || gamma < 0 || V < 1 || !(T >= 0.0) || isinf(T) || !(band >= 0.0))
    return ORC_ERR_ARG;
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  double *r = (double *)malloc(sizeof(double) * (size_t)V);
  if (!p || !q || !r) { free(p); free(q); free(r); return ORC_ERR_MEM; }
  int rc = ORC_OK;
  for (long b = 0; b < B; ++b) {
    const size_t trow0 = (size_t)b * (size_t)(gamma + 1);
    const size_t drow0 = (size_t)b * (size_t)gamma;
    const int32_t *x = tokens + (size_t)b * (size_t)gamma;
    const float *u = uniforms ? uniforms + (size_t)b * (size_t)(gamma + 1) : NULL;
    int32_t *acc_b = accept + drow0;
    double *dm_b = dmargin + drow0;
    int32_t *tok_b = tok + trow0, *lo_b = lo + trow0, *hi_b = hi + trow0;
    double *cm_b = cmargin + trow0;
    for (long i = 0; i < gamma; ++i) { acc_b[i] = 0; dm_b[i] = INFINITY; }
    for (long j = 0; j <= gamma; ++j) {
      tok_b[j] = lo_b[j] = hi_b[j] = -1;
      cm_b[j] = INFINITY;
    }

    int err = ORC_OK;   /* the same validation as oracle_verify_chain */
    for (long i = 0; i <= gamma && !err; ++i)
      if (!row_valid(target, dtype, (trow0 + (size_t)i) * (size_t)V, V)) err = ORC_ERR_ROW;
    if (T > 0.0)
      for (long i = 0; i < gamma && !err; ++i)
        if (!row_valid(draft, dtype, (drow0 + (size_t)i) * (size_t)V, V)) err = ORC_ERR_ROW;
    for (long i = 0; i < gamma && !err; ++i)
      if (x[i] < 0 || x[i] >= V) err = ORC_ERR_TOKEN;
    if (err) {
      if (rc == ORC_OK) rc = err;
      continue;
    }

    for (long j = 0; j <= gamma; ++j) {
      const size_t toff = (trow0 + (size_t)j) * (size_t)V;
      if (T == 0.0) {
        long g = argmax_row(target, dtype, toff, V);
        if (j < gamma) acc_b[j] = (x[j] == g);
        tok_b[j] = lo_b[j] = hi_b[j] = (int32_t)g;
        continue;
      }
      softmax_row(target, dtype, toff, V, T, p);
      double scale = 1.0;
      if (j < gamma) {
        softmax_row(draft, dtype, (drow0 + (size_t)j) * (size_t)V, V, T, q);
        double px = p[x[j]], qx = q[x[j]];
        double ratio = (qx > 0.0) ? px / qx : (px > 0.0 ? INFINITY : 0.0);
        double uj = (double)u[j];
        acc_b[j] = !(uj > ratio);
        if (isfinite(ratio))
          dm_b[j] = fabs(uj - ratio) / (ratio > 1e-300 ? ratio : 1e-300);
        /* the correction this position would draw: residual max(0, p - q) */
        double S = 0.0;
        scale = 0.0;
        for (long k = 0; k < V; ++k) {
          double d = p[k] - q[k];
          r[k] = d > 0.0 ? d : 0.0;
          S += r[k];
          if (r[k] > 0.0) scale += p[k];
        }
        if (S == 0.0) {
          for (long k = 0; k < V; ++k) r[k] = p[k];
          scale = 1.0;
        }
      } else {
        for (long k = 0; k < V; ++k) r[k] = p[k];
      }
      double cm;
      long lk, hk;
      tok_b[j] = (int32_t)inverse_cdf(r, V, (double)u[gamma], scale, &cm);
      cm_b[j] = cm;
      cdf_band(r, V, (double)u[gamma], scale, band, &lk, &hk);
      lo_b[j] = (int32_t)lk;
      hi_b[j] = (int32_t)hk;
    }
  }
  free(p); free(q); free(r);
  return rc;
}

/* ------------------------------------------------------------------ public: tree verify */

/*
 * Batched greedy tree verify.
 *   target   [B, N, V]  target logits at every node
 *   parents  [B, N]     parents[b,0] = -1, 0 <= parents[b,i] < i
 *   tokens   [B, N]     node tokens (node 0's is unused)
 * A node is accepted iff it is the root, or its parent is accepted and its token equals the
 * target argmax at its parent. d* = deepest accepted node (smallest index on ties).
 * Outputs: accept_len[B] = depth(d*); path_nodes[B, N] = root..d*, then -1;
 * out_tokens[B, N] = tokens of path nodes 1..depth, then argmax at d* (bonus), then -1.
 */
int oracle_verify_tree(const void *target, int dtype, const int32_t *parents,
                       const int32_t *tokens, long B, long N, long V, int32_t *accept_len,
                       int32_t *path_nodes, int32_t *out_tokens) {
  if (B < 0 || N < 1 || V < 1) return ORC_ERR_ARG;
  long *g = (long *)malloc(sizeof(long) * (size_t)N);
  int *acc = (int *)malloc(sizeof(int) * (size_t)N);
  long *depth = (long *)malloc(sizeof(long) * (size_t)N);
  long *path = (long *)malloc(sizeof(long) * (size_t)N);
  if (!g || !acc || !depth || !path) {
    free(g); free(acc); free(depth); free(path);
    return ORC_ERR_MEM;
  }
  int rc = ORC_OK;
  for (long b = 0; b < B; ++b) {
    const int32_t *par = parents + (size_t)b * (size_t)N;
    const int32_t *tok = tokens + (size_t)b * (size_t)N;
    int32_t *pn = path_nodes + (size_t)b * (size_t)N;
    int32_t *ot = out_tokens + (size_t)b * (size_t)N;
    for (long j = 0; j < N; ++j) { pn[j] = -1; ot[j] = -1; }

    int err = ORC_OK;
    if (par[0] != -1) err = ORC_ERR_PARENT;
    for (long i = 1; i < N && !err; ++i)
      if (par[i] < 0 || par[i] >= i) err = ORC_ERR_PARENT;
    for (long i = 1; i < N && !err; ++i)
      if (tok[i] < 0 || tok[i] >= V) err = ORC_ERR_TOKEN;
    for (long j = 0; j < N && !err; ++j)
      if (!row_valid(target, dtype, ((size_t)b * (size_t)N + (size_t)j) * (size_t)V, V))
        err = ORC_ERR_ROW;
    if (err) {
      accept_len[b] = -1;
      if (rc == ORC_OK) rc = err;
      continue;
    }

    for (long j = 0; j < N; ++j)
      g[j] = argmax_row(target, dtype, ((size_t)b * (size_t)N + (size_t)j) * (size_t)V, V);
    acc[0] = 1;
    depth[0] = 0;
    for (long i = 1; i < N; ++i) {
      long pa = par[i];
      acc[i] = acc[pa] && (long)tok[i] == g[pa];
      depth[i] = depth[pa] + 1;
    }
    long best = 0;
    for (long i = 1; i < N; ++i)
      if (acc[i] && depth[i] > depth[best]) best = i;

    long D = depth[best];
    long v = best;
    for (long j = D; j >= 0; --j) { path[j] = v; v = (j > 0) ? par[v] : -1; }
    for (long j = 0; j <= D; ++j) pn[j] = (int32_t)path[j];
    for (long j = 0; j < D; ++j) ot[j] = tok[path[j + 1]];
    ot[D] = (int32_t)g[best];
    accept_len[b] = (int32_t)D;
  }
  free(g); free(acc); free(depth); free(path);
  return rc;
}

/*
 * Batched stochastic (T > 0) tree verify: the tree's walk by sequential per-sibling rejection
 * sampling. The pages verify Falcon's tree only greedily (Falcon review, Figure 4, "greedy
 * (temperature=0)"); for sampling this build takes the rejection rule of chain verification
 * ("Fast Inference from Transformers via Speculative Decoding", pith.science review, "The pith",
 * "Desk Editor's Note": accept while u <= p/q, correct a rejection from norm(max(0, p - q)))
 * and applies it to the siblings of a node one after another, the residual of each rejection
 * becoming the target of the next sibling's test. When every child of a node was drafted
 * independently from the drafter's distribution q at that node, each emitted token is an exact
 * sample of the target given the tokens before it.
 *   target   [B, N, V]  target logits at every node (p_i: the next token after node i's path)
 *   draft    [B, N, V]  draft logits at every node (q_i: the distribution node i's children
 *                       were drafted from)
 *   parents  [B, N]     parents[b,0] = -1, 0 <= parents[b,i] < i
 *   tokens   [B, N]     node tokens (node 0's is unused)
 *   uniforms [B, N]     u[b,0]: the final draw; u[b,i], i >= 1: node i's acceptance test
 * Per batch row, from cur = the root:
 *   r = p_cur, q = q_cur;
 *   for each child c of cur, in increasing index: x = tokens[c],
 *     ratio = r(x) / q(x) (q(x) = 0: +inf if r(x) > 0, else 0);
 *     u[c] <= ratio: accept c (emit x, cur = c, start again at c);
 *     else r = norm(max(0, r - q)) (unchanged if that sums to 0);
 *   no child accepted (or none): draw the last token from r with u[b,0] (inverse CDF, first k
 *   whose running sum strictly exceeds u * sum(r)).
 * T == 0 is greedy tree verification (oracle_verify_tree; draft logits and uniforms unused).
 * Outputs as oracle_verify_tree: accept_len = accepted tokens (the final node's depth),
 * path_nodes = root .. final node, out_tokens = accepted tokens then the drawn token, then -1.
 * margin[B] (may be NULL): the minimum over the walk's decisions and its draw, each relative to
 * the rounding amplification A of the residual it used: A = product over its updates of P/S
 * (P = the previous r's mass on the new support, S = the mass of max(0, r - q)); a decision
 * |u - ratio| / (ratio A), the draw min(c_k - t, t - c_{k-1}) / A (A = 1 with no update, as for
 * the chain's bonus draw; one update gives the chain's P/S).
 */
/*
 * The walk of oracle_verify_tree_sample with its two kinds of margin apart (each may be NULL):
 * dmargin[b] the smallest over the walk's decisions, cmargin[b] the final draw's, and the
 * draw's band [lo[b], hi[b]] (cdf_band, width band * A in the normalised residual). T == 0:
 * margins +inf, the band the drawn token.
 */
int oracle_verify_tree_sample_detail(const void *target, const void *draft, int dtype,
                                     const int32_t *parents, const int32_t *tokens,
                                     const float *uniforms, long B, long N, long V, double T,
                                     double band, int32_t *accept_len, int32_t *path_nodes,
                                     int32_t *out_tokens, double *dmargin, double *cmargin,
                                     int32_t *lo, int32_t *hi) {
  if (B < 0 || N < 1 || V < 1 || !(T >= 0.0) || isinf(T) || !(band >= 0.0)) return ORC_ERR_ARG;
  if (T == 0.0) {
    int rc0 = oracle_verify_tree(target, dtype, parents, tokens, B, N, V, accept_len, path_nodes,
                                 out_tokens);
    for (long b = 0; b < B; ++b) {
      const int32_t a = accept_len[b];
      const int32_t t = a >= 0 ? out_tokens[(size_t)b * (size_t)N + (size_t)a] : -1;
      if (dmargin) dmargin[b] = INFINITY;
      if (cmargin) cmargin[b] = INFINITY;
      if (lo) lo[b] = t;
      if (hi) hi[b] = t;
    }
    return rc0;
  }
  double *r = (double *)malloc(sizeof(double) * (size_t)V);
  double *q = (double *)malloc(sizeof(double) * (size_t)V);
  double *w = (double *)malloc(sizeof(double) * (size_t)V);
  if (!r || !q || !w) { free(r); free(q); free(w); return ORC_ERR_MEM; }
  int rc = ORC_OK;
  for (long b = 0; b < B; ++b) {
    const int32_t *par = parents + (size_t)b * (size_t)N;
    const int32_t *tok = tokens + (size_t)b * (size_t)N;
    const float *u = uniforms + (size_t)b * (size_t)N;
    int32_t *pn = path_nodes + (size_t)b * (size_t)N;
    int32_t *ot = out_tokens + (size_t)b * (size_t)N;
    for (long j = 0; j < N; ++j) { pn[j] = -1; ot[j] = -1; }
    if (dmargin) dmargin[b] = INFINITY;
    if (cmargin) cmargin[b] = INFINITY;
    if (lo) lo[b] = -1;
    if (hi) hi[b] = -1;

    int err = ORC_OK;   /* the same validation as greedy tree verify, plus the draft rows */
    if (par[0] != -1) err = ORC_ERR_PARENT;
    for (long i = 1; i < N && !err; ++i)
      if (par[i] < 0 || par[i] >= i) err = ORC_ERR_PARENT;
    for (long i = 1; i < N && !err; ++i)
      if (tok[i] < 0 || tok[i] >= V) err = ORC_ERR_TOKEN;
    for (long j = 0; j < N && !err; ++j) {
      const size_t off = ((size_t)b * (size_t)N + (size_t)j) * (size_t)V;
      if (!row_valid(target, dtype, off, V) || !row_valid(draft, dtype, off, V))
        err = ORC_ERR_ROW;
    }
    if (err) {
      accept_len[b] = -1;
      if (rc == ORC_OK) rc = err;
      continue;
    }

    double mg = INFINITY;
    long cur = 0, depth = 0;
    pn[0] = 0;
    for (;;) {
      const size_t off = ((size_t)b * (size_t)N + (size_t)cur) * (size_t)V;
      softmax_row(target, dtype, off, V, T, r);
      softmax_row(draft, dtype, off, V, T, q);
      double A = 1.0;
      long next = -1;
      for (long c = cur + 1; c < N && next < 0; ++c) {
        if (par[c] != cur) continue;
        const long x = tok[c];
        double ratio = (q[x] > 0.0) ? r[x] / q[x] : (r[x] > 0.0 ? INFINITY : 0.0);
        double uc = (double)u[c];
        if (isfinite(ratio)) {
          double m = fabs(uc - ratio) / fmax(ratio * A, 1e-300);
          if (m < mg) mg = m;
        }
        if (uc <= ratio) { next = c; break; }
        /* rejected: the residual becomes the target of the next sibling's test */
        double S = 0.0, P = 0.0;
        for (long k = 0; k < V; ++k) {
          double d = r[k] - q[k];
          w[k] = d > 0.0 ? d : 0.0;
          S += w[k];
          if (w[k] > 0.0) P += r[k];
        }
        if (S > 0.0) {
          for (long k = 0; k < V; ++k) r[k] = w[k] / S;
          A *= P / S;
        }
      }
      if (next >= 0) {
        ++depth;
        pn[depth] = (int32_t)next;
        ot[depth - 1] = tok[next];
        cur = next;
        continue;
      }
      double cm;
      const long t = inverse_cdf(r, V, (double)u[0], A, &cm);
      long lk, hk;
      cdf_band(r, V, (double)u[0], A, band, &lk, &hk);
      if (cmargin) cmargin[b] = cm;
      if (lo) lo[b] = (int32_t)lk;
      if (hi) hi[b] = (int32_t)hk;
      ot[depth] = (int32_t)t;
      break;
    }
    accept_len[b] = (int32_t)depth;
    if (dmargin) dmargin[b] = mg;
  }
  free(r); free(q); free(w);
  return rc;
}

int oracle_verify_tree_sample(const void *target, const void *draft, int dtype,
                              const int32_t *parents, const int32_t *tokens, const float *uniforms,
                              long B, long N, long V, double T, int32_t *accept_len,
                              int32_t *path_nodes, int32_t *out_tokens, double *margin) {
  double *cm = margin ? (double *)malloc(sizeof(double) * (size_t)(B > 0 ? B : 1)) : NULL;
  if (margin && !cm) return ORC_ERR_MEM;
  int rc = oracle_verify_tree_sample_detail(target, draft, dtype, parents, tokens, uniforms, B, N,
                                            V, T, 0.0, accept_len, path_nodes, out_tokens, margin,
                                            cm, NULL, NULL);
  for (long b = 0; b < B && margin; ++b)
    if (cm[b] < margin[b]) margin[b] = cm[b];
  free(cm);
  return rc;
}

/* ------------------------------------------------------------------ public: drafter side */

/*
 * Drafter-side sampling, the step before verification: the draft model proposes x_i by
 * sampling its own distribution q_i ("Fast Inference from Transformers via Speculative
 * Decoding", pith.science review, "The pith": the small model proposes tokens that the large
 * model then checks).
 *   out_tokens[r] = the inverse-CDF draw from softmax(logits[r] / T) with uniform u[r]: the first
 *   k whose running sum of p exceeds u (sums in index order); T == 0: the lowest-index argmax;
 *   -1 for an invalid row. margin[r] (may be NULL): the CDF margin of the draw (+inf at T == 0).
 */
int oracle_sample(const void *logits, int dtype, long rows, long V, double T,
                  const float *uniforms, int32_t *out_tokens, double *margin) {
  if (rows < 0 || V < 1 || !(T >= 0.0) || isinf(T)) return ORC_ERR_ARG;
  double *p = (double *)malloc(sizeof(double) * (size_t)V);
  if (!p) return ORC_ERR_MEM;
  int rc = ORC_OK;
  for (long r = 0; r < rows; ++r) {
    size_t off = (size_t)r * (size_t)V;
    if (margin) margin[r] = INFINITY;
    if (!row_valid(logits, dtype, off, V)) {
      out_tokens[r] = -1;
      if (rc == ORC_OK) rc = ORC_ERR_ROW;
      continue;
    }
    if (T == 0.0) {
      out_tokens[r] = (int32_t)argmax_row(logits, dtype, off, V);
      continue;
    }
    softmax_row(logits, dtype, off, V, T, p);
    double mg = 0.0;
    out_tokens[r] = (int32_t)inverse_cdf(p, V, (double)uniforms[r], 1.0, &mg);
    if (margin) margin[r] = mg;
  }
  free(p);
  return rc;
}

/*
 * Top-n candidates per row, for building a draft tree: Falcon expands each node of its decoding
 * tree with the drafter's most likely tokens at that node ("Falcon: Faster and Parallel
 * Inference of Large Language Models through Enhanced Semi-Autoregressive Drafting and
 * Custom-Designed Decoding Tree", pith.science review, "What carries the argument": deeper
 * branches for higher-probability tokens).
 *   out_idx[r, 0..k) = the indices of the k largest logits of row r, largest first, equal values
 *   in increasing index order (so out_idx[r, 0] is the lowest-index argmax); a logit's rank does
 *   not depend on the temperature. -1 everywhere for an invalid row. 1 <= k <= V.
 */
int oracle_topk(const void *logits, int dtype, long rows, long V, long k, int32_t *out_idx) {
  if (rows < 0 || V < 1 || k < 1 || k > V) return ORC_ERR_ARG;
  char *taken = (char *)malloc((size_t)V);
  if (!taken) return ORC_ERR_MEM;
  int rc = ORC_OK;
  for (long r = 0; r < rows; ++r) {
    size_t off = (size_t)r * (size_t)V;
    int32_t *o = out_idx + (size_t)r * (size_t)k;
    if (!row_valid(logits, dtype, off, V)) {
      for (long j = 0; j < k; ++j) o[j] = -1;
      if (rc == ORC_OK) rc = ORC_ERR_ROW;
      continue;
    }
    memset(taken, 0, (size_t)V);
    for (long j = 0; j < k; ++j) {   /* repeated selection of the best remaining element */
      long best = -1;
      double bv = 0.0;
      for (long q = 0; q < V; ++q) {
        if (taken[q]) continue;
        double v = logit_at(logits, dtype, off + (size_t)q);
        if (best < 0 || v > bv) { best = q; bv = v; }
      }
      taken[best] = 1;
      o[j] = (int32_t)best;
    }
  }
  free(taken);
  return rc;
}

/*
 * Tree-attention mask: in Falcon's decoding tree every node attends to itself and its
 * ancestors only (Falcon review, Figure 3, "SAR decoding tree attention").
 *   words[b, i, w] (W = ceil(N / 32) words per node) has bit j % 32 of word j / 32 set iff node j
 *   is node i or an ancestor of node i. parents as for oracle_verify_tree; an invalid tree gets
 *   an all-zero mask and ORC_ERR_PARENT.
 */
int oracle_tree_mask(const int32_t *parents, long B, long N, uint32_t *words) {
  if (B < 0 || N < 1) return ORC_ERR_ARG;
  long W = (N + 31) / 32;
  int rc = ORC_OK;
  for (long b = 0; b < B; ++b) {
    const int32_t *par = parents + (size_t)b * (size_t)N;
    uint32_t *m = words + (size_t)b * (size_t)N * (size_t)W;
    for (long q = 0; q < N * W; ++q) m[q] = 0u;
    int bad = par[0] != -1;
    for (long i = 1; i < N && !bad; ++i)
      if (par[i] < 0 || par[i] >= i) bad = 1;
    if (bad) {
      if (rc == ORC_OK) rc = ORC_ERR_PARENT;
      continue;
    }
    for (long i = 0; i < N; ++i)   /* walk from the node up to the root */
      for (long j = i; j >= 0; j = (j > 0) ? par[j] : -1)
        m[(size_t)i * (size_t)W + (size_t)(j / 32)] |= 1u << (j % 32);
  }
  return rc;
}

/*
 * LM-head logits as stored by the fused producer: the last layer of the target's (and the
 * drafter's) scoring pass, logits = hidden . head^T ("Fast Inference from Transformers via
 * Speculative Decoding", pith.science review, "The pith": the target scores every drafted
 * position in one parallel pass), stored in bf16. The dot products are taken by the Python
 * wrapper (a float64 matrix product); this is the rounding of each exact-or-nearly value to
 * the nearest bf16, ties to the even significand (IEEE 754 roundTiesToEven), straight from
 * double so that no intermediate float rounds it twice. NaN -> 0x7FC0; magnitudes at or above
 * 2^128 after rounding -> infinity; below 2^-126 the spacing stays 2^-133 (bf16 subnormals).
 */
int oracle_round_bf16(const double *x, long n, uint16_t *out) {
  if (n < 0 || (n > 0 && (!x || !out))) return ORC_ERR_ARG;
  for (long i = 0; i < n; ++i) {
    const double v = x[i];
    if (isnan(v)) { out[i] = 0x7FC0; continue; }
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) { out[i] = sign; continue; }
    if (isinf(a)) { out[i] = sign | 0x7F80; continue; }
    int e;
    frexp(a, &e);                 /* a = f 2^e, 0.5 <= f < 1: the leading bit is 2^(e-1) */
    int q = e - 8;                /* 8 significant bits: the spacing is 2^(e-8) */
    if (q < -133) q = -133;
    a = ldexp(nearbyint(ldexp(a, -q)), q);   /* exact scalings; nearest, ties to even */
    if (a >= ldexp(1.0, 128)) { out[i] = sign | 0x7F80; continue; }
    /* a has at most 8 significant bits and lies in float's range: exact as a float, whose
       upper 16 bits are then its bf16 pattern */
    const float f = (float)a;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    out[i] = (uint16_t)(sign | (u >> 16));
  }
  return ORC_OK;
}

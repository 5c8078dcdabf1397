"""Pins the CPU oracle to facts that do not come from the oracle itself.

What the pages fix about the verify step, and how each is checked here:

* Exactness -- speculative decoding produces exact samples of the target distribution ("Fast
  Inference from Transformers via Speculative Decoding", pith.science review: "Core claim",
  "Desk Editor's Note": rejection sampling that keeps the exact target distribution).
  Checked (a) exactly, by treating the oracle as a black box in the uniforms and measuring,
  to float32 resolution, the set of uniforms that yields each output, and (b) statistically,
  with a chi-squared test over 10^6 seeded steps. The target distribution is known in closed
  form because the logits are ln(w) at T = 1, so p = w / sum(w) needs no softmax code.
* Acceptance rate -- the probability that a draft token passes is sum_x min(p(x), q(x)); the
  mean number of tokens per step is (1 - a^(gamma+1)) / (1 - a) for identical positions, and
  sum_k prod_{i<k} a_i in general. This is what the review's "What would settle it" statistic
  (average accepted tokens per step) measures.
* Greedy identity -- at temperature 0 the output is identical to greedy decoding of the target
  (the pages' "identical outputs"; Falcon review, "Editorial extensions: decoding is lossless"
  and Figure 4, greedy temperature 0): checked against a separate greedy loop written with
  numpy's argmax, and against the T -> 0 limit of the sampling branch.
* Tree -- a node is accepted when its whole root path matches the target argmaxes (Falcon
  review, "What carries the argument"): checked against brute-force enumeration of every root
  path, and against chain verification on path-shaped trees.
* Probabilities -- special cases with closed forms (ln-weights, power-of-two temperature
  scaling, shifts, masked entries, exact bf16 widening).
"""

import math

import numpy as np
import pytest

from workloads import BF16, F32, bf16_to_f32, f32_to_bf16, make_uniforms

# --------------------------------------------------------------------------- helpers


def ln_logits(w):
    w = np.asarray(w, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.where(w > 0, np.log(np.where(w > 0, w, 1.0)), -np.inf).astype(np.float32)


def norm(w):
    w = np.asarray(w, dtype=np.float64)
    return w / w.sum()


TINY_U = np.float32(np.finfo(np.float32).tiny)       # smallest normal float32 > 0
TOP_U = np.float32(1.0) - np.float32(2.0 ** -24)      # largest float32 below 1


def _bits(u):
    return int(np.float32(u).view(np.uint32))


def _from_bits(b):
    return np.uint32(b).view(np.float32)


def step_outcomes(orc, tgt_rows, drf_rows, x, u_batch, T=1.0):
    """Run the oracle once per row of u_batch on the same logits/draft tokens.
    Returns (accept_len [G], out_tokens [G, gamma+1])."""
    G = u_batch.shape[0]
    tgt = np.broadcast_to(tgt_rows, (G,) + tgt_rows.shape).copy()
    drf = np.broadcast_to(drf_rows, (G,) + drf_rows.shape).copy()
    tok = np.broadcast_to(np.asarray(x, np.int32), (G, len(x))).copy()
    acc, out, _, rc = orc.verify_chain(tgt, drf, F32, tok, u_batch.astype(np.float32), T)
    assert rc == 0
    return acc, out


def measure_1d(f, grid=2048):
    """Measure, over u in (0,1), the set on which the integer-valued black box f(u) takes
    each value. f maps a float32 array to an int array. Returns {value: measure}."""
    us = np.concatenate([[TINY_U], ((np.arange(grid) + 0.5) / grid).astype(np.float32), [TOP_U]])
    vals = f(us)
    cache = {}

    def ev(b):
        if b not in cache:
            cache[b] = int(f(np.asarray([_from_bits(b)], np.float32))[0])
        return cache[b]

    bounds = []  # (u_boundary, value_left, value_right)

    def find(lo_b, hi_b, vlo, vhi):
        # outcomes at bit patterns lo_b < hi_b differ; locate every change in between
        if hi_b - lo_b <= 1:
            bounds.append((float(_from_bits(hi_b)), vlo, vhi))
            return
        mid = (lo_b + hi_b) // 2
        vm = ev(mid)
        if vm != vlo:
            find(lo_b, mid, vlo, vm)
        if vm != vhi:
            find(mid, hi_b, vm, vhi)

    for i in range(len(us) - 1):
        if vals[i] != vals[i + 1]:
            find(_bits(us[i]), _bits(us[i + 1]), int(vals[i]), int(vals[i + 1]))
    bounds.sort()
    meas = {}
    left, cur = 0.0, int(vals[0])
    for ub, vl, vr in bounds:
        assert vl == cur
        meas[cur] = meas.get(cur, 0.0) + (ub - left)
        left, cur = ub, vr
    meas[cur] = meas.get(cur, 0.0) + (1.0 - left)
    return meas


# --------------------------------------------------------------------------- exactness


def _exact_case(gamma, V, seed):
    rng = np.random.default_rng(seed)
    wp = [rng.integers(1, 9, V).astype(float) for _ in range(gamma + 1)]
    wq = [rng.integers(1, 9, V).astype(float) for _ in range(gamma)]
    # zero-mass entries exercise ratio = +inf (q = 0 < p) and ratio = 0 (p = 0 < q)
    if gamma >= 1:
        wp[0][0] = 0.0
        wq[0][1] = 0.0
    return wp, wq


@pytest.mark.parametrize("gamma,V,seed", [(1, 5, 11), (2, 4, 12), (2, 6, 13)])
def test_emitted_tokens_are_exact_target_samples(orc, gamma, V, seed):
    """For every position j the token emitted there, given the step reached j, is
    distributed exactly as p_j -- measured without sampling error."""
    wp, wq = _exact_case(gamma, V, seed)
    p = [norm(w) for w in wp]
    q = [norm(w) for w in wq]
    tgt = np.stack([ln_logits(w) for w in wp])               # [gamma+1, V]
    drf = np.stack([ln_logits(w) for w in wq]) if gamma else np.zeros((0, V), np.float32)

    def reachable_token(i):   # a token accepted with probability > 0 at position i
        return int(np.argmax(p[i] / np.maximum(q[i], 1e-300)))

    def rejectable_token(i):  # a token with p(x)/q(x) < 1 - 2^-24, i.e. rejectable
        return int(np.argmax(q[i] - p[i]))

    for j in range(gamma + 1):
        # uniforms for positions before j: TINY accepts any reachable token
        base_x = [reachable_token(i) for i in range(gamma)]
        dist = np.zeros(V)
        if j < gamma:
            rej_mass = 0.0
            for x in range(V):
                if q[j][x] == 0:
                    continue
                xs = list(base_x)
                xs[j] = x

                def acc_f(u, xs=xs):
                    ub = np.full((len(u), gamma + 1), 0.5, np.float32)
                    ub[:, :j] = TINY_U
                    ub[:, j] = u
                    a, _ = step_outcomes(orc, tgt, drf, xs, ub)
                    return (a > j).astype(int)

                A = measure_1d(acc_f).get(1, 0.0)
                dist[x] += q[j][x] * A
                rej_mass += q[j][x] * (1.0 - A)
            # the correction draw after a rejection at j depends on u_gamma only
            xs = list(base_x)
            xs[j] = rejectable_token(j)

            def res_f(u, xs=xs):
                ub = np.full((len(u), gamma + 1), 0.5, np.float32)
                ub[:, :j] = TINY_U
                ub[:, j] = TOP_U
                ub[:, gamma] = u
                a, o = step_outcomes(orc, tgt, drf, xs, ub)
                assert np.all(a == j)
                return o[:, j]

            for k, m in measure_1d(res_f).items():
                dist[k] += rej_mass * m
        else:
            def bonus_f(u):
                ub = np.full((len(u), gamma + 1), TINY_U, np.float32)
                ub[:, gamma] = u
                a, o = step_outcomes(orc, tgt, drf, base_x, ub)
                assert np.all(a == gamma)
                return o[:, gamma]

            for k, m in measure_1d(bonus_f).items():
                dist[k] += m
        # float32 ln(w) logits perturb p by ~1e-7 relative; uniforms resolve to 2^-24
        np.testing.assert_allclose(dist, p[j], rtol=0, atol=2e-6,
                                   err_msg=f"position {j} of gamma={gamma}")


def test_chi_squared_first_token_and_acceptance_rates(orc):
    """10^6 seeded steps, V=8, gamma=2, drafts x_i ~ q_i: the first emitted token follows p_0
    (chi-squared), and the acceptance rate at positions 0 and 1 is sum_x min(p_i, q_i)."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(20240601)
    V, gamma, n = 8, 2, 1_000_000
    wp = [np.array([5, 1, 3, 8, 2, 7, 4, 6.]), np.array([1, 1, 9, 2, 4, 4, 3, 1.]),
          np.array([2, 3, 2, 3, 2, 3, 2, 3.])]
    wq = [np.array([3, 6, 3, 4, 4, 2, 8, 1.]), np.array([2, 1, 5, 5, 1, 4, 3, 6.])]
    p = [norm(w) for w in wp]
    q = [norm(w) for w in wq]
    tgt = np.broadcast_to(np.stack([ln_logits(w) for w in wp]), (n, gamma + 1, V)).copy()
    drf = np.broadcast_to(np.stack([ln_logits(w) for w in wq]), (n, gamma, V)).copy()
    x = np.stack([rng.choice(V, size=n, p=q[i]) for i in range(gamma)], axis=1).astype(np.int32)
    u = make_uniforms(rng, (n, gamma + 1))
    acc, out, _, rc = orc.verify_chain(tgt, drf, F32, x, u, 1.0)
    assert rc == 0
    counts = np.bincount(out[:, 0], minlength=V)
    assert chisquare(counts, n * p[0]).pvalue > 1e-3
    for i in range(gamma):
        reached = acc >= i
        alpha = np.minimum(p[i], q[i]).sum()
        rate = (acc[reached] > i).mean()
        sd = math.sqrt(alpha * (1 - alpha) / reached.sum())
        assert abs(rate - alpha) < 4 * sd, (i, rate, alpha)
    # token emitted at position 1 (given it was reached) follows p_1 too
    sel = acc >= 1
    c1 = np.bincount(out[sel, 1], minlength=V)
    assert chisquare(c1, sel.sum() * p[1]).pvalue > 1e-3
    # a deliberately wrong target (p_1 in place of p_0) must be rejected by the same test
    assert chisquare(counts, n * p[1]).pvalue < 1e-6


def test_mean_tokens_per_step_closed_form(orc):
    """Identical p, q at every position: E[emitted tokens] = (1 - a^(g+1)) / (1 - a)."""
    rng = np.random.default_rng(7)
    V, gamma, n = 8, 4, 400_000
    wp = np.array([4, 1, 3, 8, 2, 7, 4, 6.])
    wq = np.array([3, 6, 3, 4, 4, 2, 8, 1.])
    p, q = norm(wp), norm(wq)
    alpha = np.minimum(p, q).sum()
    tgt = np.broadcast_to(ln_logits(wp), (n, gamma + 1, V)).copy()
    drf = np.broadcast_to(ln_logits(wq), (n, gamma, V)).copy()
    x = rng.choice(V, size=(n, gamma), p=q).astype(np.int32)
    u = make_uniforms(rng, (n, gamma + 1))
    acc, out, _, rc = orc.verify_chain(tgt, drf, F32, x, u, 1.0)
    assert rc == 0
    emitted = acc + 1
    expect = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    sd = emitted.std() / math.sqrt(n)
    assert abs(emitted.mean() - expect) < 4 * sd, (emitted.mean(), expect)
    # emitted tokens per row: exactly n accepted drafts then one more, then -1
    assert np.all((out >= 0).sum(axis=1) == emitted)


def test_mean_tokens_general_product_form(orc):
    """Position-dependent p_i, q_i on the tiny fp32 workload's distributions:
    E[emitted] = sum_k prod_{i<k} a_i, averaged over rows."""
    from workloads import chain_tiny
    ci = chain_tiny(B=1000)
    B, g, V = ci.B, ci.gamma, ci.V
    reps = 40
    rng = np.random.default_rng(3)
    pt, rc1 = orc.probs(ci.target, F32, 1.0)
    qd, rc2 = orc.probs(ci.draft, F32, 1.0)
    assert rc1 == 0 and rc2 == 0
    alpha = np.minimum(pt[:, :g], qd).sum(axis=2)                    # [B, g]
    expect = np.ones(B)
    run = np.ones(B)
    for k in range(1, g + 1):
        run = run * alpha[:, k - 1]
        expect += run
    tot = np.zeros(B)
    sq = np.zeros(B)
    for _ in range(reps):
        # fresh drafts x_i ~ q_i and fresh uniforms
        cdf = np.cumsum(qd, axis=2)
        r = rng.random((B, g, 1))
        x = np.minimum((cdf < r).sum(axis=2), V - 1).astype(np.int32)
        u = make_uniforms(rng, (B, g + 1))
        acc, _, _, rc = orc.verify_chain(ci.target, ci.draft, F32, x, u, 1.0)
        assert rc == 0
        tot += acc + 1
        sq += (acc + 1) ** 2
    mean_emit = tot.sum() / (B * reps)
    var = sq.sum() / (B * reps) - mean_emit ** 2
    sd = math.sqrt(var / (B * reps))
    assert abs(mean_emit - expect.mean()) < 4 * sd + 1e-3, (mean_emit, expect.mean())


# --------------------------------------------------------------------------- greedy


def _tie_logits(rng, shape):
    """Small-integer logits (many exact ties), stored as bf16."""
    return f32_to_bf16(rng.integers(-3, 4, size=shape).astype(np.float32))


def test_greedy_equals_target_greedy_decoding(orc):
    rng = np.random.default_rng(5)
    B, g, V = 400, 5, 16
    tgt = _tie_logits(rng, (B, g + 1, V))
    drf = _tie_logits(rng, (B, g, V))
    tv = bf16_to_f32(tgt)
    # drafts: the target's greedy token 70% of the time
    greedy = np.argmax(tv, axis=2)          # numpy: lowest index on ties
    x = np.where(rng.random((B, g)) < 0.7, greedy[:, :g], rng.integers(0, V, (B, g)))
    x = x.astype(np.int32)
    u = make_uniforms(rng, (B, g + 1))
    acc, out, mg, rc = orc.verify_chain(tgt, drf, BF16, x, u, 0.0)
    assert rc == 0
    assert np.all(np.isinf(mg))
    for b in range(B):
        ys = []
        for j in range(g + 1):
            ys.append(int(np.argmax(tv[b, j])))
            if j < g and x[b, j] != ys[-1]:
                break
        assert acc[b] == len(ys) - 1
        assert list(out[b, :len(ys)]) == ys
        assert np.all(out[b, len(ys):] == -1)
    # the draft logits are not read at T = 0: NaN there changes nothing
    drf_nan = drf.copy()
    drf_nan[:, :, 0] = 0x7FC0
    acc2, out2, _, rc2 = orc.verify_chain(tgt, drf_nan, BF16, x, u, 0.0)
    assert rc2 == 0 and np.array_equal(acc, acc2) and np.array_equal(out, out2)


def test_sampling_branch_reaches_greedy_as_T_goes_to_zero(orc):
    """With a gap of >= 0.1 under each row's maximum, exp((l - m)/T) underflows to exactly 0 at
    T = 1e-4, so the sampling branch must reproduce the greedy branch exactly."""
    rng = np.random.default_rng(9)
    B, g, V = 300, 4, 12
    vals = np.stack([rng.permutation(V) for _ in range(B * (2 * g + 1))]).astype(np.float32)
    vals = (vals * 0.1).reshape(B, 2 * g + 1, V)
    tgt = np.ascontiguousarray(vals[:, :g + 1])
    drf = np.ascontiguousarray(vals[:, g + 1:])
    greedy = np.argmax(tgt, axis=2)
    x = np.where(rng.random((B, g)) < 0.6, greedy[:, :g], rng.integers(0, V, (B, g)))
    x = x.astype(np.int32)
    u = make_uniforms(rng, (B, g + 1))
    a0, o0, _, rc0 = orc.verify_chain(tgt, drf, F32, x, u, 0.0)
    a1, o1, _, rc1 = orc.verify_chain(tgt, drf, F32, x, u, 1e-4)
    assert rc0 == 0 and rc1 == 0
    np.testing.assert_array_equal(a0, a1)
    np.testing.assert_array_equal(o0, o1)


# --------------------------------------------------------------------------- tree


def brute_force_tree(tv, parents, tokens):
    """Every root path checked on its own: node i is accepted iff for every node j on its
    root path (j != root), tokens[j] == argmax(logits at parent(j))."""
    N = len(parents)
    g = np.argmax(tv, axis=1)
    best, best_depth, best_path = 0, 0, [0]
    for i in range(N):
        path = [i]
        while path[-1] != 0:
            path.append(int(parents[path[-1]]))
        path = path[::-1]
        if all(tokens[j] == g[parents[j]] for j in path[1:]):
            d = len(path) - 1
            if d > best_depth:
                best, best_depth, best_path = i, d, path
    out = [int(tokens[j]) for j in best_path[1:]] + [int(g[best])]
    return best_depth, best_path, out


def _random_tree(rng, N):
    return np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)], dtype=np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_tree_matches_brute_force(orc, seed):
    rng = np.random.default_rng(100 + seed)
    B, V = 60, 4
    N = int(rng.integers(2, 13))
    parents = np.stack([_random_tree(rng, N) for _ in range(B)])
    tgt = _tie_logits(rng, (B, N, V))
    tv = bf16_to_f32(tgt)
    g = np.argmax(tv, axis=2)
    tokens = np.where(rng.random((B, N)) < 0.75,
                      np.take_along_axis(g, np.maximum(parents, 0), axis=1),
                      rng.integers(0, V, (B, N))).astype(np.int32)
    acc, path, out, rc = orc.verify_tree(tgt, BF16, parents, tokens)
    assert rc == 0
    for b in range(B):
        d, pth, o = brute_force_tree(tv[b], parents[b], tokens[b])
        assert acc[b] == d
        assert list(path[b, :d + 1]) == pth and np.all(path[b, d + 1:] == -1)
        assert list(out[b, :d + 1]) == o and np.all(out[b, d + 1:] == -1)


def test_path_shaped_tree_equals_greedy_chain(orc):
    rng = np.random.default_rng(77)
    B, g, V = 200, 6, 10
    tgt = _tie_logits(rng, (B, g + 1, V))
    greedy = np.argmax(bf16_to_f32(tgt), axis=2)
    x = np.where(rng.random((B, g)) < 0.8, greedy[:, :g], rng.integers(0, V, (B, g)))
    x = x.astype(np.int32)
    u = make_uniforms(rng, (B, g + 1))
    ca, co, _, rc = orc.verify_chain(tgt, tgt[:, :g], BF16, x, u, 0.0)
    parents = np.tile(np.arange(-1, g, dtype=np.int32), (B, 1))
    tokens = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    ta, tp, to, rt = orc.verify_tree(tgt, BF16, parents, tokens)
    assert rc == 0 and rt == 0
    np.testing.assert_array_equal(ca, ta)
    np.testing.assert_array_equal(co, to)
    for b in range(B):
        assert list(tp[b, :ta[b] + 1]) == list(range(ta[b] + 1))


def test_tree_invalid_inputs(orc):
    V = 4
    tgt = np.zeros((4, 3, V), np.float32)
    parents = np.array([[-1, 0, 1], [0, 0, 1], [-1, 0, 2], [-1, 0, 0]], np.int32)
    tokens = np.array([[0, 0, 0], [0, 0, 0], [0, 0, 0], [0, 0, V]], np.int32)
    acc, path, out, rc = orc.verify_tree(tgt, F32, parents, tokens)
    assert rc == orc.ERR_PARENT
    assert list(acc) == [2, -1, -1, -1]
    assert np.all(path[1:] == -1) and np.all(out[1:] == -1)


# --------------------------------------------------------------------------- probabilities


def test_probs_closed_forms(orc):
    rng = np.random.default_rng(1)
    w = rng.integers(1, 100, size=(50, 37)).astype(np.float64)
    p, rc = orc.probs(ln_logits(w), F32, 1.0)
    assert rc == 0
    np.testing.assert_allclose(p, w / w.sum(axis=1, keepdims=True), rtol=2e-6, atol=0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    # doubling the logits and the temperature changes nothing (scaling by 2 is exact)
    lg = (rng.standard_normal((20, 33)) * 3).astype(np.float32)
    p1, _ = orc.probs(lg, F32, 0.7)
    p2, _ = orc.probs(lg * np.float32(2), F32, 1.4)
    np.testing.assert_allclose(p1, p2, rtol=1e-14, atol=1e-300)
    # an exact shift of bf16-valued logits changes nothing
    lb = bf16_to_f32(f32_to_bf16(lg))
    p3, _ = orc.probs(lb, F32, 1.0)
    p4, _ = orc.probs(lb + np.float32(16.0), F32, 1.0)
    np.testing.assert_allclose(p3, p4, rtol=1e-12, atol=1e-300)
    # bf16 input equals its exact fp32 widening, bit for bit
    p5, _ = orc.probs(f32_to_bf16(lg), BF16, 1.0)
    assert np.array_equal(p5, p3)
    # masked (-inf) entries get probability 0 and the rest renormalise
    lm = lg.copy()
    lm[:, ::3] = -np.inf
    p6, _ = orc.probs(lm, F32, 1.0)
    assert np.all(p6[:, ::3] == 0)
    keep = np.ones(33, bool)
    keep[::3] = False
    p7, _ = orc.probs(np.ascontiguousarray(lg[:, keep]), F32, 1.0)
    np.testing.assert_allclose(p6[:, keep], p7, rtol=1e-14, atol=0)
    # T = 0: one-hot at numpy's argmax (lowest index on ties)
    lt = rng.integers(-2, 3, size=(40, 9)).astype(np.float32)
    p8, _ = orc.probs(lt, F32, 0.0)
    assert np.array_equal(np.argmax(p8, axis=1), np.argmax(lt, axis=1))
    assert np.all(p8.sum(axis=1) == 1.0) and np.all((p8 == 0) | (p8 == 1))
    a, rc = orc.argmax(lt, F32)
    assert rc == 0 and np.array_equal(a, np.argmax(lt, axis=1))


def test_probs_invalid_rows(orc):
    lg = np.zeros((4, 5), np.float32)
    lg[0, 2] = np.nan
    lg[1, 0] = np.inf
    lg[2, :] = -np.inf
    lg[3, 1] = -np.inf          # a masked entry alone is fine
    p, rc = orc.probs(lg, F32, 1.0)
    assert rc == orc.ERR_ROW
    assert np.all(np.isnan(p[:3])) and np.all(np.isfinite(p[3]))
    a, rc = orc.argmax(lg, F32)
    assert list(a) == [-1, -1, -1, 0]


def test_bf16_widening_is_exact():
    vals = np.array([1.0, -2.5, 3.140625, 0.0, -0.0, 65280.0, -np.inf, 2.0 ** -126], np.float32)
    assert np.array_equal(bf16_to_f32(f32_to_bf16(vals)).view(np.uint32), vals.view(np.uint32))
    assert f32_to_bf16(np.array([1.0], np.float32))[0] == 0x3F80
    # round to nearest even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> 1
    assert f32_to_bf16(np.array([1.0 + 2 ** -8], np.float32))[0] == 0x3F80
    assert f32_to_bf16(np.array([1.0 + 3 * 2 ** -8], np.float32))[0] == 0x3F82


# --------------------------------------------------------------------------- chain edge cases


def test_chain_invalid_rows_and_tokens(orc):
    V, g = 6, 2
    tgt = np.zeros((4, g + 1, V), np.float32)
    drf = np.zeros((4, g, V), np.float32)
    x = np.zeros((4, g), np.int32)
    x[1, 1] = V             # token out of range
    tgt[2, 2, 3] = np.nan   # bad target row (even at the bonus position)
    drf[3, 1, 0] = np.inf   # bad draft row
    u = np.full((4, g + 1), 0.5, np.float32)
    acc, out, mg, rc = orc.verify_chain(tgt, drf, F32, x, u, 1.0)
    assert rc in (orc.ERR_TOKEN, orc.ERR_ROW)
    assert list(acc) == [2, -1, -1, -1]
    assert np.all(out[1:] == -1)
    # at T = 0 the bad draft row is not read
    acc0, _, _, _ = orc.verify_chain(tgt, drf, F32, x, u, 0.0)
    assert list(acc0) == [2, -1, -1, 2]


def test_margins_flag_near_boundary_draws(orc):
    """The decision margin is |u - ratio| / ratio and the CDF margin is the distance of
    u * S to the nearest CDF step, relative to P (for this bonus draw P = S = 1; residual draws
    with P != S are pinned by tests/golden/margin_cases.json)."""
    V = 4
    tgt = np.zeros((1, 2, V), np.float32)                     # p_0 = 1/4 each
    drf = np.array([[[0, 0, -np.inf, -np.inf]]], np.float32)  # q_0 = (1/2, 1/2, 0, 0)
    x = np.array([[0]], np.int32)                             # ratio = 1/2
    for u0 in (0.25, 0.49):
        acc, out, mg, rc = orc.verify_chain(tgt, drf, F32, x,
                                            np.array([[u0, 0.6]], np.float32), 1.0)
        assert rc == 0 and acc[0] == 1
        # decision margin |u0 - 1/2| / (1/2); the bonus CDF (1/4, 1/2, 3/4, 1) is 0.1 from
        # t = 0.6 at its nearest step (relative to S = 1)
        assert mg[0] == pytest.approx(min(abs(np.float32(u0) - 0.5) / 0.5, 0.15 - 0.05),
                                      rel=1e-6)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_detail_band_holds_every_draw_within_band(orc, seed):
    """Brute force over the uniform: the band [lo, hi] the detail reports for a draw holds every
    token the oracle draws when t = u * S moves by at most band * P, and its ends are drawn
    when they carry mass. Residual draws (x_0 has p = 0, so position 0 always rejects) and
    bonus draws; a wide band (0.2) so that it spans several tokens."""
    rng = np.random.default_rng(seed)
    V, band = 12, 0.2
    t = (rng.standard_normal((1, 2, V)) * 1.5).astype(np.float32)
    d = t[:, :1] + (rng.standard_normal((1, 1, V)) * 1.0).astype(np.float32)
    t[0, 1, 5] = -np.inf                          # a masked token in the bonus row
    x = np.array([[3]], np.int32)
    t[0, 0, 3] = -np.inf                          # p_0(x_0) = 0: ratio 0, always rejected
    p, _ = orc.probs(t[0], F32, 1.0)
    q, _ = orc.probs(d[0], F32, 1.0)
    r0 = np.maximum(p[0] - q[0], 0.0)
    spans = []
    for j, (S, P) in enumerate([(r0.sum(), p[0][r0 > 0].sum()), (1.0, 1.0)]):
        u = np.float32(0.2 + 0.6 * rng.random())
        det = orc.verify_chain_detail(t, d, F32, x, np.array([[0.5, u]], np.float32), 1.0,
                                      band=band)
        lo, hi = int(det["lo"][0, j]), int(det["hi"][0, j])
        grid = np.linspace(float(u) - band * P / S, float(u) + band * P / S, 4001)
        grid = grid[(grid > 0) & (grid < 1)].astype(np.float32)
        uu = np.stack([np.full(len(grid), 0.5, np.float32), grid], axis=1)
        T_ = np.repeat(t, len(grid), axis=0)
        D_ = np.repeat(d, len(grid), axis=0)
        X_ = np.repeat(x, len(grid), axis=0)
        if j == 0:
            acc, out, _, _ = orc.verify_chain(T_, D_, F32, X_, uu, 1.0)
            assert np.all(acc == 0)
            drawn = out[:, 0]
        else:   # the bonus draw from p_1, reached through a draft that is always accepted
            T2 = T_.copy()
            T2[:, 0, :] = 0.0
            D2 = np.zeros_like(D_)
            acc, out, _, _ = orc.verify_chain(T2, D2, F32, X_, uu, 1.0)
            assert np.all(acc == 1)
            drawn = out[:, 1]
            det = orc.verify_chain_detail(T2[:1], D2[:1], F32, x, np.array([[0.5, u]], np.float32),
                                          1.0, band=band)
            lo, hi = int(det["lo"][0, 1]), int(det["hi"][0, 1])
        assert drawn.min() >= lo and drawn.max() <= hi, (j, lo, hi, np.unique(drawn))
        w = r0 if j == 0 else p[1]
        assert (w[lo] == 0 or lo in drawn) and (w[hi] == 0 or hi in drawn), (j, lo, hi)
        spans.append(hi > lo)
    assert any(spans)           # the wide band spans more than one token at least once

"""Pins of the oracle's stochastic (T > 0) tree verification, each independent of the code it
checks:

- hand-derived dyadic cases (tests/golden/tree_sample_cases.json): the second sibling is tested
  against the residual left by the first, not against p; margins with the rounding
  amplification of each residual update;
- a chain-shaped tree is chain verification: the same accept lengths, tokens and margins as the
  (separately pinned) chain oracle on the same rows and uniforms;
- at T = 0 it is greedy tree verification;
- exactness: with every node's children drafted independently from the drafter's distribution
  at that node, and target distributions that depend only on the token path, the first,
  second and third emitted tokens follow the target given the tokens before them (chi-squared
  over 200000 seeded walks, pre-registered seed, p > 1e-3);
- invalid inputs are reported per tree like greedy tree verification.
"""

import math

import numpy as np
import pytest

from golden_io import tree_sample_cases
from workloads import BF16, F32, f32_to_bf16, make_uniforms, tree_shape


@pytest.mark.parametrize("case", tree_sample_cases(), ids=lambda c: c["name"])
def test_tree_sample_golden(orc, case):
    acc, path, out, mg, rc = orc.verify_tree_sample(case["target"], case["draft"], F32,
                                                    case["parents"], case["tokens"],
                                                    case["uniforms"], case["T"])
    assert rc == 0
    np.testing.assert_array_equal(acc, case["accept_len"])
    np.testing.assert_array_equal(path, case["path_nodes"])
    np.testing.assert_array_equal(out, case["out_tokens"])
    assert mg[0] == pytest.approx(case["margin"], rel=1e-9, abs=1e-15)


@pytest.mark.parametrize("seed,gamma,V,dtype", [(0, 4, 50, F32), (1, 1, 7, F32), (2, 6, 300, BF16),
                                                (3, 3, 2, F32)])
def test_chain_shaped_tree_is_chain_verification(orc, seed, gamma, V, dtype):
    """A tree whose nodes form one path: node i+1 carries draft x_i, node i has the chain's
    target row i and draft row i, node i+1's uniform is u_i and node 0's is the chain's final
    uniform u_gamma."""
    rng = np.random.default_rng(seed)
    B = 400
    t = (rng.standard_normal((B, gamma + 1, V)) * 1.5).astype(np.float32)
    d = (t[:, :gamma] + rng.standard_normal((B, gamma, V)) * 0.7).astype(np.float32)
    d[::5] = t[::5, :gamma]                                    # all-accepting steps
    if dtype == BF16:
        t, d = f32_to_bf16(t), f32_to_bf16(d)
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    u = make_uniforms(rng, (B, gamma + 1))
    acc, out, mg, rc = orc.verify_chain(t, d, dtype, x, u, 1.3)
    assert rc == 0
    N = gamma + 1
    tdraft = np.concatenate([d, d[:, :1]], axis=1)            # the leaf's draft row is unused
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    tok = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    tu = np.concatenate([u[:, gamma:], u[:, :gamma]], axis=1)
    tacc, tpath, tout, tmg, trc = orc.verify_tree_sample(t, tdraft, dtype, par, tok, tu, 1.3)
    assert trc == 0
    np.testing.assert_array_equal(tacc, acc)
    np.testing.assert_array_equal(tout, out)
    for b in range(B):
        np.testing.assert_array_equal(tpath[b, :acc[b] + 1], np.arange(acc[b] + 1))
        assert np.all(tpath[b, acc[b] + 1:] == -1)
    # the tree normalises its residual before the CDF, the chain scans it unnormalised: the
    # same margins up to rounding of the cumulative sums
    np.testing.assert_allclose(tmg, mg, rtol=1e-8)
    assert 0 < acc.mean() < gamma


def test_greedy_limit_is_greedy_tree_verification(orc):
    rng = np.random.default_rng(9)
    B, N, V = 40, 40, 30
    par = np.stack([tree_shape(rng, N) for _ in range(B)])
    x = rng.integers(-3, 3, size=(B, N, V)).astype(np.float32)
    g = np.argmax(x, axis=2)
    tok = np.where(rng.random((B, N)) < 0.8, np.take_along_axis(g, np.maximum(par, 0), 1),
                   rng.integers(0, V, (B, N))).astype(np.int32)
    want = orc.verify_tree(x, F32, par, tok)
    got = orc.verify_tree_sample(x, x, F32, par, tok, None, 0.0)
    for w, g_ in zip(want[:3], got[:3]):
        np.testing.assert_array_equal(g_, w)
    assert want[3] == got[4] == 0


def _chi2_sf(x, k):
    """Survival function of the chi-squared distribution with k degrees of freedom (the
    regularised upper incomplete gamma function, by its series), for the p-values below."""
    a, z = k / 2.0, x / 2.0
    if z <= 0:
        return 1.0
    term = 1.0 / a
    total = term
    for n in range(1, 100000):
        term *= z / (a + n)
        total += term
        if term < total * 1e-15:
            break
    lower = math.exp(-z + a * math.log(z) - math.lgamma(a)) * total
    return max(0.0, 1.0 - lower)


def _chi2_p(counts, probs):
    n = counts.sum()
    keep = probs > 0
    assert np.all(counts[~keep] == 0), "a token of zero target probability was emitted"
    e = n * probs[keep]
    stat = float(((counts[keep] - e) ** 2 / e).sum())
    return _chi2_sf(stat, int(keep.sum()) - 1)


def test_emitted_tokens_follow_the_target(orc):
    """Exactness of the walk by statistics. Tree: the root with 3 children, each with 2 children
    (N = 10). Target and draft logits depend only on the token path (root; root + y; root + y +
    z), so that siblings with equal tokens share their distributions, as a language model's
    would; every node's children are drafted independently from the drafter's distribution at
    that node. Over 200000 walks: the first emitted token follows p(root); the second, given an
    accepted first token y, follows p(y); the third, given accepted y and z, follows p(y, z)."""
    rng = np.random.default_rng(20260101)
    V, T, W = 6, 1.0, 200000
    lt0 = rng.standard_normal(V) * 1.2
    lt1 = rng.standard_normal((V, V)) * 1.2
    lt2 = rng.standard_normal((V, V, V)) * 1.2
    ld0 = lt0 + rng.standard_normal(V) * 0.9
    ld1 = lt1 + rng.standard_normal((V, V)) * 0.9
    sm = lambda l: np.exp(l - l.max(axis=-1, keepdims=True)) / np.exp(
        l - l.max(axis=-1, keepdims=True)).sum(axis=-1, keepdims=True)
    q0, q1 = sm(ld0), sm(ld1)
    par = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], np.int32)
    N = len(par)
    # draft tokens: children of the root from q0, children of node c from q1[token c]
    c1 = np.stack([rng.choice(V, size=W, p=q0) for _ in range(3)], axis=1)
    c2 = np.empty((W, 6), np.int64)
    for j in range(3):
        cum = np.cumsum(q1[c1[:, j]], axis=1)
        for k in range(2):
            r = rng.random(W)[:, None]
            c2[:, 2 * j + k] = np.minimum((r > cum).sum(axis=1), V - 1)
    tok = np.concatenate([np.zeros((W, 1), np.int64), c1, c2], axis=1).astype(np.int32)
    tgt = np.empty((W, N, V), np.float32)
    drf = np.zeros((W, N, V), np.float32)
    tgt[:, 0] = lt0
    drf[:, 0] = ld0
    for c in range(1, 4):
        tgt[:, c] = lt1[tok[:, c]]
        drf[:, c] = ld1[tok[:, c]]
    for c in range(4, 10):
        tgt[:, c] = lt2[tok[:, par[c]], tok[:, c]]
    u = make_uniforms(rng, (W, N))
    acc, path, out, mg, rc = orc.verify_tree_sample(tgt, drf, F32, np.tile(par, (W, 1)), tok, u,
                                                    T)
    assert rc == 0
    # the oracle works in double precision on the fp32 logits: the reference distributions too
    p0 = sm(lt0.astype(np.float32).astype(np.float64))
    assert _chi2_p(np.bincount(out[:, 0], minlength=V), p0) > 1e-3
    pv = []
    for y in range(V):
        sel = (acc >= 1) & (out[:, 0] == y)
        if sel.sum() < 2000:
            continue
        p1 = sm(lt1[y].astype(np.float32).astype(np.float64))
        pv.append(_chi2_p(np.bincount(out[sel, 1], minlength=V), p1))
        for z in range(V):
            sel2 = sel & (acc >= 2) & (out[:, 1] == z)
            if sel2.sum() < 2000:
                continue
            p2 = sm(lt2[y, z].astype(np.float32).astype(np.float64))
            pv.append(_chi2_p(np.bincount(out[sel2, 2], minlength=V), p2))
    assert len(pv) >= 6
    # every conditional test passes at the level that keeps a family of this size at 1e-3
    assert min(pv) > 1e-3 / len(pv), pv
    assert 0.5 < acc.mean() < 2.0


def test_tree_sample_invalid_inputs(orc):
    B, N, V = 4, 5, 8
    par = np.tile(np.array([-1, 0, 0, 1, 1], np.int32), (B, 1))
    t = np.zeros((B, N, V), np.float32)
    d = np.zeros((B, N, V), np.float32)
    tok = np.ones((B, N), np.int32)
    par[1, 4] = 4
    tok[2, 3] = V
    d[3, 2, 0] = np.nan
    u = np.full((B, N), 0.5, np.float32)
    acc, path, out, mg, rc = orc.verify_tree_sample(t, d, F32, par, tok, u, 1.0)
    assert rc in (orc.ERR_PARENT, orc.ERR_TOKEN, orc.ERR_ROW)
    assert list(acc) == [acc[0], -1, -1, -1] and acc[0] >= 0
    assert np.all(out[1:] == -1) and np.all(path[1:] == -1)

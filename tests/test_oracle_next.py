"""Pins of the oracle's drafter-side and tree-attention functions to facts that do not come
from the oracle:

* sampling -- with logits ln(w) for integer weights w at T = 1 (or T * ln(w) at temperature T)
  the distribution is w / sum(w) exactly, so the inverse-CDF token for a uniform u is the first
  k whose integer running sum exceeds u * sum(w), computed here exactly; at T = 0 it is numpy's
  argmax;
* top-n -- numpy's lexicographic sort by (value descending, index ascending);
* tree mask -- a separate walk over parent pointers written here in Python.
"""

import numpy as np
import pytest

from workloads import BF16, F32, f32_to_bf16, make_uniforms


def test_sample_matches_exact_integer_cdf(orc):
    rng = np.random.default_rng(1)
    for V in (1, 2, 5, 64, 1000):
        w = rng.integers(1, 50, size=(40, V)).astype(np.float64)
        w[:, ::7] = 0.0                                     # zero-probability tokens
        w[w.sum(axis=1) == 0, 0] = 1.0
        with np.errstate(divide="ignore"):
            lg = np.where(w > 0, np.log(np.where(w > 0, w, 1.0)), -np.inf).astype(np.float32)
        u = make_uniforms(rng, (40,))
        tok, mg, rc = orc.sample(lg, F32, u, 1.0)
        assert rc == 0
        for r in range(40):
            c = np.cumsum(w[r])
            want = int(np.argmax(c > float(u[r]) * c[-1]))
            if mg[r] > 1e-9:   # float32 logits of ln(w) round w itself by ~1e-7 relative
                assert tok[r] == want, (V, r)
            assert w[r, tok[r]] > 0


def test_sample_distribution_on_a_uniform_grid(orc):
    """Weights summing to 64, uniforms at the midpoints of a 1/4096 grid: each token is drawn
    for exactly w_k / 64 of the grid."""
    w = np.array([5, 0, 11, 16, 3, 29], np.float64)
    lg = np.tile(np.log(np.where(w > 0, w, 1.0)).astype(np.float32), (4096, 1))
    lg[:, 1] = -np.inf
    u = ((np.arange(4096) + 0.5) / 4096).astype(np.float32)
    for T in (1.0, 0.5):
        tok, _, rc = orc.sample((lg * np.float32(T)).astype(np.float32), F32, u, T)
        assert rc == 0
        np.testing.assert_array_equal(np.bincount(tok, minlength=6), w * 64)


def test_sample_greedy_and_invalid_rows(orc):
    rng = np.random.default_rng(2)
    x = rng.integers(-3, 4, size=(30, 77)).astype(np.float32)   # many ties
    tok, _, rc = orc.sample(x, F32, np.full(30, 0.5, np.float32), 0.0)
    assert rc == 0
    np.testing.assert_array_equal(tok, np.argmax(x, axis=1))
    x[3, 5] = np.nan
    x[7, :] = -np.inf
    tok, _, rc = orc.sample(x, F32, np.full(30, 0.5, np.float32), 1.0)
    assert rc != 0 and tok[3] == -1 and tok[7] == -1


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_topk_matches_numpy_lexsort(orc, dtype):
    rng = np.random.default_rng(3)
    for V, k in ((1, 1), (9, 9), (100, 4), (3001, 16), (5000, 1)):
        x = rng.integers(-6, 6, size=(25, V)).astype(np.float32)   # ties everywhere
        x[:, 1::11] = -np.inf                                       # masked tokens
        lg = f32_to_bf16(x) if dtype == BF16 else x
        idx, rc = orc.topk(lg, dtype, k)
        assert rc == 0
        for r in range(25):
            order = np.lexsort((np.arange(V), -x[r].astype(np.float64)))
            np.testing.assert_array_equal(idx[r], order[:k])


def test_topk_invalid_rows(orc):
    x = np.zeros((3, 10), np.float32)
    x[0, 2] = np.inf
    x[1, :] = -np.inf
    idx, rc = orc.topk(x, F32, 3)
    assert rc != 0
    assert np.all(idx[:2] == -1) and list(idx[2]) == [0, 1, 2]


def _ancestor_mask(par):
    N = len(par)
    W = (N + 31) // 32
    m = np.zeros((N, W), np.uint32)
    for i in range(N):
        j = i
        while j != -1:
            m[i, j // 32] |= np.uint32(1 << (j % 32))
            j = par[j]
    return m


def test_tree_mask_matches_parent_walk(orc):
    from workloads import tree_shape
    rng = np.random.default_rng(4)
    for N in (1, 2, 31, 32, 33, 64, 100, 1024):
        pars = [tree_shape(rng, N) if N <= 64 else
                np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)], np.int32)
                for _ in range(3)]
        par = np.stack(pars).astype(np.int32)
        m, rc = orc.tree_mask(par)
        assert rc == 0
        for b in range(3):
            np.testing.assert_array_equal(m[b], _ancestor_mask(par[b]))


def test_tree_mask_invalid_tree(orc):
    par = np.array([[-1, 0, 1], [0, 0, 1], [-1, 2, 0]], np.int32)
    m, rc = orc.tree_mask(par)
    assert rc != 0
    np.testing.assert_array_equal(m[0, :, 0], [1, 3, 7])
    assert np.all(m[1] == 0) and np.all(m[2] == 0)

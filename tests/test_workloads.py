"""The seeded input generators: determinism, shapes, value recipes and tree structure."""

import numpy as np

from workloads import (BF16, F32, as_f32, chain_32k, chain_tiny, make_uniforms, tree_32k,
                       tree_shape)


def test_uniforms_open_interval_and_exact():
    u = make_uniforms(np.random.default_rng(0), 100000)
    assert u.dtype == np.float32
    assert u.min() > 0 and u.max() < 1
    k = (u.astype(np.float64) * 2 ** 24 - 1) / 2
    assert np.all(k == np.round(k))          # every value is (2k+1)/2^24 exactly


def test_generators_are_deterministic():
    a, b = chain_tiny(B=20), chain_tiny(B=20)
    assert np.array_equal(a.target, b.target) and np.array_equal(a.tokens, b.tokens)
    assert np.array_equal(a.uniforms, b.uniforms)
    c = chain_tiny(seed=99, B=20)
    assert not np.array_equal(a.target, c.target)


def test_chain_shapes_and_recipe():
    ci = chain_32k(B=4, gamma=3, V=4000)
    assert ci.target.shape == (4, 4, 4000) and ci.draft.shape == (4, 3, 4000)
    assert ci.dtype == BF16 and ci.target.dtype == np.uint16
    assert ci.tokens.shape == (4, 3) and ci.tokens.min() >= 0 and ci.tokens.max() < 4000
    t = as_f32(ci.target, BF16)
    # 50 peaked ids per (row, position) sit about 8 above the N(0, 3^2) bulk
    assert np.all((t > 8 + 3 * 3.5).sum(axis=2) <= 50 + 5)
    tiny = chain_tiny(B=8)
    assert tiny.dtype == F32 and tiny.target.dtype == np.float32
    d = tiny.draft - tiny.target[:, :4]
    assert abs(d.std() - 0.5) < 0.02


def test_tree_shape_rule():
    rng = np.random.default_rng(0)
    for _ in range(20):
        p = tree_shape(rng, 64)
        assert len(p) == 64 and p[0] == -1
        assert np.all(p[1:] >= 0) and np.all(p[1:] < np.arange(1, 64))
        depth = np.zeros(64, int)
        for i in range(1, 64):
            depth[i] = depth[p[i]] + 1
        assert depth.max() == 6
        # breadth-first numbering: depth never decreases with the node index
        assert np.all(np.diff(depth) >= 0)
        # branching limits per depth {4, 3, 2, 2, 1, 1}
        kids = np.bincount(p[1:], minlength=64)
        for i in range(64):
            assert kids[i] <= (4, 3, 2, 2, 1, 1, 0)[depth[i]]


def test_tree_tokens_follow_designated_argmax():
    ti = tree_32k(B=3, N=64, V=3000)
    t = as_f32(ti.target, BF16)
    g = np.argmax(t, axis=2)
    assert np.array_equal(g, ti.meta["designated"])      # designated id is the strict max
    par = ti.parents
    follow = ti.tokens[:, 1:] == np.take_along_axis(g, par[:, 1:], axis=1)
    assert 0.5 < follow.mean() < 0.9

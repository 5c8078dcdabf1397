"""GPU parity of stochastic (T > 0) tree verification (spec_verify_tree_sample, through the C
ABI) against the oracle's walk: hand-derived cases exactly, chain-shaped trees against chain
verification, configuration 4's trees with sampled drafts at full size, ragged and unaligned
rows, wide and deep trees, T = 0 (greedy), and invalid trees."""

import numpy as np
import pytest
import torch

from golden_io import tree_sample_cases
from gpu_util import compare_chain, compare_tree_sample, dev, run_chain, run_tree_sample
from workloads import (BF16, F32, ChainInputs, TreeInputs, f32_to_bf16, make_uniforms,
                       tree_sample_32k, tree_shape)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_78_gb300 as sv
    sv.load_library()


@pytest.mark.parametrize("case", tree_sample_cases(), ids=lambda c: c["name"])
def test_golden_tree_sample(orc, case):
    """Dyadic probabilities: the kernels' fp32 arithmetic is exact on them."""
    ti = TreeInputs(case["name"], case["target"], F32, case["parents"], case["tokens"])
    acc, path, out, st = run_tree_sample(ti, case["draft"], case["uniforms"],
                                         float(np.float32(case["T"])))
    assert st == 0
    np.testing.assert_array_equal(acc, case["accept_len"])
    np.testing.assert_array_equal(path, case["path_nodes"])
    np.testing.assert_array_equal(out, case["out_tokens"])


@pytest.mark.parametrize("offset", [0, 1])
def test_tree_sample_32k_full_size(orc, offset):
    """Configuration 4's shape (32 trees x 64 nodes x 32000 bf16) with sampled drafts, T = 1."""
    ti = tree_sample_32k()
    draft, u = ti.meta["draft"], ti.meta["uniforms"]
    gpu = run_tree_sample(ti, draft, u, 1.0, offset_elems=offset)
    assert gpu[3] == 0
    compare_tree_sample(orc, ti, draft, u, 1.0, gpu, name=ti.name)
    assert gpu[0].max() >= 1


# V = 300001 fp32: a vocabulary slice per CTA no longer fits in shared memory even across a
# cluster of eight, so the walk runs one CTA per tree reading the rows from L2 (the other cases
# take the cluster walk with p and q in shared memory)
@pytest.mark.parametrize("dtype,V,N,T", [(F32, 1000, 12, 0.8), (BF16, 4099, 64, 1.0),
                                         (F32, 7, 30, 2.0), (BF16, 70001, 20, 0.6),
                                         (F32, 1, 5, 1.0), (F32, 300001, 6, 1.0)])
def test_tree_sample_shapes(orc, dtype, V, N, T):
    ti = tree_sample_32k(seed=7 + V, B=24, N=N, V=V, dtype=dtype, temperature=T,
                         peaked=min(50, max(1, V // 4)))
    draft, u = ti.meta["draft"], ti.meta["uniforms"]
    for off in (0, 1):
        gpu = run_tree_sample(ti, draft, u, T, offset_elems=off)
        assert gpu[3] == 0
        compare_tree_sample(orc, ti, draft, u, T, gpu, name=ti.name)


def test_tree_sample_many_trees(orc):
    """300 trees of 16 nodes over V=32000 bf16: more trees than SMs, so the walk's clusters shrink
    to the two CTAs a slice of p and q needs to fit, in several waves."""
    ti = tree_sample_32k(seed=88, B=300, N=16, V=32000)
    draft, u = ti.meta["draft"], ti.meta["uniforms"]
    gpu = run_tree_sample(ti, draft, u, 1.0)
    assert gpu[3] == 0
    compare_tree_sample(orc, ti, draft, u, 1.0, gpu, name=ti.name)


@pytest.mark.parametrize("kind", ["star", "chain", "wide_deep"])
def test_tree_sample_structures(orc, kind):
    """A star of 200 children of the root (up to 199 residual updates at one node), a 300-node
    path, and 1024-node random trees."""
    rng = np.random.default_rng({"star": 1, "chain": 2, "wide_deep": 3}[kind])
    B, V = 6, 300
    N = {"star": 201, "chain": 300, "wide_deep": 1024}[kind]
    if kind == "star":
        par = np.tile(np.array([-1] + [0] * (N - 1), np.int32), (B, 1))
    elif kind == "chain":
        par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    else:
        par = np.stack([np.array([-1] + [int(rng.integers(max(0, i - 8), i)) for i in range(1, N)])
                        for _ in range(B)]).astype(np.int32)
    t = (rng.standard_normal((B, N, V)) * 1.5).astype(np.float32)
    d = (t + rng.standard_normal((B, N, V)) * 0.6).astype(np.float32)
    if kind == "star":   # a root whose children are mostly rejected: the drafter is far off
        d[:, 0] = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    qd = np.exp(d - d.max(axis=2, keepdims=True))
    qd /= qd.sum(axis=2, keepdims=True)
    tok = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(1, N):
            tok[b, i] = rng.choice(V, p=qd[b, par[b, i]])
    u = make_uniforms(rng, (B, N))
    ti = TreeInputs(kind, t, F32, par, tok)
    gpu = run_tree_sample(ti, d, u, 1.0)
    assert gpu[3] == 0
    compare_tree_sample(orc, ti, d, u, 1.0, gpu, name=f"tree_sample_{kind}")


@pytest.mark.parametrize("seed,gamma,V,dtype", [(0, 4, 5000, BF16), (1, 7, 1001, F32)])
def test_chain_shaped_tree_sample_is_chain_verification(orc, seed, gamma, V, dtype):
    """On chain-shaped trees the walk is chain verification: the same outputs as
    spec_verify_chain on the same rows, and both as the oracle."""
    rng = np.random.default_rng(seed)
    B = 64
    t = (rng.standard_normal((B, gamma + 1, V)) * 2).astype(np.float32)
    d = (t[:, :gamma] + rng.standard_normal((B, gamma, V)) * 0.5).astype(np.float32)
    if dtype == BF16:
        t, d = f32_to_bf16(t), f32_to_bf16(d)
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    u = make_uniforms(rng, (B, gamma + 1))
    ci = ChainInputs("chain", t, d, dtype, x, u, 1.0)
    cg = run_chain(ci)
    compare_chain(orc, ci, cg)
    N = gamma + 1
    tdraft = np.concatenate([d, d[:, :1]], axis=1)
    par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
    tok = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    tu = np.concatenate([u[:, gamma:], u[:, :gamma]], axis=1)
    ti = TreeInputs("chain_tree", t, dtype, par, tok)
    tg = run_tree_sample(ti, tdraft, tu, 1.0)
    assert tg[3] == 0
    compare_tree_sample(orc, ti, tdraft, tu, 1.0, tg, name="tree_sample_chain_shaped")
    same = (tg[0] == cg[0]) & np.all(tg[2][:, :gamma + 1] == cg[1], axis=1)
    assert same.mean() > 0.95


def test_tree_sample_greedy_and_errors(orc):
    import speculative_decoding_verification_78_gb300 as sv
    ti = tree_sample_32k(seed=21, B=8, N=40, V=3000, dtype=F32)
    draft = ti.meta["draft"]
    # T = 0: greedy tree verification, draft logits and uniforms not read
    acc, path, out, st = sv.verify_tree_sample(dev(ti.target), None, dev(ti.parents),
                                               dev(ti.tokens), None, 0.0)
    ra, rp, ro, rc = orc.verify_tree(ti.target, F32, ti.parents, ti.tokens)
    assert int(st.item()) == 0 and rc == 0
    np.testing.assert_array_equal(acc.cpu().numpy(), ra)
    np.testing.assert_array_equal(path.cpu().numpy(), rp)
    np.testing.assert_array_equal(out.cpu().numpy(), ro)
    # invalid trees, one kind each, the others unaffected
    for what, want in (("parent", sv.SPEC_ERR_PARENT), ("token", sv.SPEC_ERR_TOKEN),
                       ("target", sv.SPEC_ERR_NONFINITE), ("draft", sv.SPEC_ERR_NONFINITE)):
        t, d = ti.target.copy(), draft.copy()
        par, tok = ti.parents.copy(), ti.tokens.copy()
        if what == "parent":
            par[3, 10] = 10
        elif what == "token":
            tok[3, 7] = 3000
        elif what == "target":
            t[3, 5, 11] = np.inf
        else:
            d[3, 0, 2] = np.nan
        bad = TreeInputs(what, t, F32, par, tok)
        gpu = run_tree_sample(bad, d, ti.meta["uniforms"], 1.0)
        assert gpu[3] == want, (what, gpu[3])
        assert gpu[0][3] == -1 and np.all(gpu[2][3] == -1) and np.all(gpu[1][3] == -1)
        compare_tree_sample(orc, bad, d, ti.meta["uniforms"], 1.0, gpu, name=f"invalid_{what}")

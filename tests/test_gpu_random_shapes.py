"""Seeded random shapes through every entry point against the oracle: batch sizes, draft
lengths, vocabularies (ragged, unaligned row bases, single- and multi-unit rows, cluster and
CTA draws), dtypes and temperatures drawn from a fixed seed, so that the launch plans and their
boundaries (one-warp finishers, clusters of 1-8 CTAs, lane groups of 1-32 per row, trees of
1-64 nodes and deeper CTA trees, the stochastic walk's cluster and single-CTA forms, the fused
LM head's tile counts and hidden sizes) are all exercised with inputs no hand-written case
chose."""

import numpy as np
import pytest
import torch

from gpu_util import compare_chain, dev, run_chain, run_tree
from workloads import (BF16, F32, ChainInputs, TreeInputs, f32_to_bf16, gumbel_draft_tokens,
                       make_uniforms, tree_shape)

pytestmark = pytest.mark.gpu

VOCABS = [1, 7, 255, 1000, 1031, 2048, 4097, 8191, 32000, 50257, 65536, 100003]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_78_gb300 as sv
    sv.load_library()


def _logits(rng, shape, dtype, scale):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    if rng.random() < 0.3:
        x[..., 1::int(rng.integers(3, 17))] = -np.inf          # masked entries (never all)
    return f32_to_bf16(x) if dtype == BF16 else x


def _f32(a, dtype):
    return (a.astype(np.uint32) << 16).view(np.float32) if dtype == BF16 else a


@pytest.mark.parametrize("seed", range(24))
def test_random_chain(orc, seed):
    rng = np.random.default_rng(1000 + seed)
    dtype = BF16 if rng.random() < 0.5 else F32
    V = int(rng.choice(VOCABS))
    B = int(rng.choice([1, 3, 17, 64, 200]))
    gamma = int(rng.integers(0, 9))
    T = float(rng.choice([0.0, 0.3, 1.0, 2.5]))
    B = max(1, min(B, 60_000_000 // ((2 * gamma + 1) * V)))   # keeps the oracle to seconds
    tgt = _logits(rng, (B, gamma + 1, V), dtype, 3.0)
    drf = _logits(rng, (B, gamma, V), dtype, 3.0) if gamma else np.zeros((B, 0, V), tgt.dtype)
    if gamma and rng.random() < 0.5:       # drafts close to the target: long accepted prefixes
        drf = tgt[:, :gamma].copy()
    tok = (gumbel_draft_tokens(rng, _f32(drf, dtype), max(T, 1e-3)) if gamma
           else np.zeros((B, 0), np.int32))
    ci = ChainInputs(f"random{seed}", tgt, drf, dtype, tok.astype(np.int32),
                     make_uniforms(rng, (B, gamma + 1)), T)
    off = int(rng.integers(0, 2))
    gpu = run_chain(ci, offset_elems=off)
    assert gpu[2] == 0
    compare_chain(orc, ci, gpu)


@pytest.mark.parametrize("seed", range(12))
def test_random_tree(orc, seed):
    rng = np.random.default_rng(2000 + seed)
    dtype = BF16 if rng.random() < 0.5 else F32
    V = int(rng.choice([2, 300, 1031, 32000, 65536]))
    B = int(rng.choice([1, 5, 32, 77]))
    N = int(rng.choice([1, 2, 9, 31, 33, 64, 65, 200]))
    if N <= 64 and rng.random() < 0.5:
        pars = np.stack([tree_shape(rng, N) if N > 1 else np.array([-1]) for _ in range(B)])
    else:                                   # random recursive trees, some of them chains
        lag = int(rng.choice([1, 3, N]))
        pars = np.stack([np.array([-1] + [int(rng.integers(max(0, i - lag), i))
                                          for i in range(1, N)]) for _ in range(B)])
    pars = pars.astype(np.int32)
    tgt = _logits(rng, (B, N, V), dtype, 2.0)
    g = np.argmax(_f32(tgt, dtype), axis=-1)
    tok = np.where(rng.random((B, N)) < 0.8, np.take_along_axis(g, np.maximum(pars, 0), 1),
                   rng.integers(0, V, (B, N))).astype(np.int32)
    ti = TreeInputs(f"rtree{seed}", tgt, dtype, pars, tok)
    acc, path, out, st = run_tree(ti, offset_elems=int(rng.integers(0, 2)))
    ra, rp, ro, rc = orc.verify_tree(tgt, dtype, pars, tok)
    assert st == 0 and rc == 0
    np.testing.assert_array_equal(acc, ra)
    np.testing.assert_array_equal(path, rp)
    np.testing.assert_array_equal(out, ro)


@pytest.mark.parametrize("seed", range(12))
def test_random_probs_sample_topk(orc, seed):
    import speculative_decoding_verification_78_gb300 as sv
    rng = np.random.default_rng(3000 + seed)
    dtype = BF16 if rng.random() < 0.5 else F32
    V = int(rng.choice(VOCABS))
    rows = int(rng.choice([1, 9, 100, 400]))
    T = float(rng.choice([0.0, 0.5, 1.0]))
    lg = _logits(rng, (rows, V), dtype, 3.0)
    off = int(rng.integers(0, 2))
    pr, st = sv.probs(dev(lg, off), T)
    po, rc = orc.probs(lg, dtype, T)
    assert int(st.item()) == 0 and rc == 0
    assert np.abs(pr.cpu().numpy().astype(np.float64) - po).max() <= 2e-6
    u = make_uniforms(rng, (rows,))
    tok, st = sv.sample(dev(lg, off), T, dev(u))
    want, mg, rc = orc.sample(lg, dtype, u, T)
    assert int(st.item()) == 0 and rc == 0
    tok = tok.cpu().numpy()
    close = mg < 1e-5
    np.testing.assert_array_equal(tok[~close], want[~close])
    assert all(po[r, tok[r]] > 0 for r in range(rows))
    k = int(rng.integers(1, min(16, V) + 1))
    idx, st = sv.topk(dev(lg, off), k)
    iw, rc = orc.topk(lg, dtype, k)
    assert int(st.item()) == 0 and rc == 0
    np.testing.assert_array_equal(idx.cpu().numpy(), iw)


@pytest.mark.parametrize("seed", range(12))
def test_random_tree_sample(orc, seed):
    """Stochastic tree walks over seeded shapes: tree sizes, vocabularies (clusters of 1-8 CTAs,
    slices that fit in shared memory or not), batch sizes, dtypes, temperatures and draft
    distances, with ragged and unaligned rows."""
    from gpu_util import compare_tree_sample, run_tree_sample
    from workloads import tree_sample_32k
    rng = np.random.default_rng(4000 + seed)
    dtype = BF16 if rng.random() < 0.5 else F32
    V = int(rng.choice([2, 300, 1031, 32000, 65536, 250007]))
    N = int(rng.choice([2, 9, 33, 64]))
    B = int(rng.choice([1, 7, 40, 160]))
    B = max(1, min(B, 40_000_000 // (2 * N * V)))
    T = float(rng.choice([0.4, 1.0, 2.0]))
    ti = tree_sample_32k(seed=5000 + seed, B=B, N=N, V=V, dtype=dtype, temperature=T,
                         draft_sigma=float(rng.choice([0.3, 1.0, 3.0])),
                         peaked=min(50, max(1, V // 4)))
    draft, u = ti.meta["draft"], ti.meta["uniforms"]
    gpu = run_tree_sample(ti, draft, u, T, offset_elems=int(rng.integers(0, 2)))
    assert gpu[3] == 0
    compare_tree_sample(orc, ti, draft, u, T, gpu, name=f"rtree_sample{seed}")


@pytest.mark.parametrize("seed", range(8))
def test_random_lmhead(orc, seed):
    """The fused LM-head call over seeded shapes (batch, draft length, vocabulary, both hidden
    sizes, temperature) on integer-grid inputs: logits bit-exact, verification draw by draw."""
    import speculative_decoding_verification_78_gb300 as sv
    from workloads import bf16_to_f32, lmhead_grid
    rng = np.random.default_rng(6000 + seed)
    B = int(rng.choice([1, 3, 20, 70]))
    gamma = int(rng.choice([1, 2, 5, 9, 16]))
    V = 256 * int(rng.choice([1, 3, 8, 33, 130]))
    Ht = 64 * int(rng.choice([1, 2, 5, 12]))
    Hd = 64 * int(rng.choice([1, 3, 7]))
    T = float(rng.choice([0.3, 1.0, 1.7]))
    li = lmhead_grid(seed=7000 + seed, B=B, gamma=gamma, V=V, Ht=Ht, Hd=Hd, temperature=T)
    lt_ref, _ = orc.lm_head_logits(li.hidden_t, li.head_t)
    ld_ref, _ = orc.lm_head_logits(li.hidden_d, li.head_d)
    tok = gumbel_draft_tokens(rng, bf16_to_f32(ld_ref).reshape(B, gamma, V), T).astype(np.int32)
    acc, out, st, lt, ld = sv.verify_chain_lmhead(dev(li.hidden_t), dev(li.head_t),
                                                  dev(li.hidden_d), dev(li.head_d), dev(tok),
                                                  dev(li.uniforms), T)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    np.testing.assert_array_equal(bits(lt), lt_ref)
    np.testing.assert_array_equal(bits(ld), ld_ref)
    ci = ChainInputs(f"rlmhead{seed}", lt_ref.reshape(B, gamma + 1, V),
                     ld_ref.reshape(B, gamma, V), BF16, tok, li.uniforms, T)
    compare_chain(orc, ci, (acc.cpu().numpy(), out.cpu().numpy(), 0))

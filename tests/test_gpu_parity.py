"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle on the same
seeded inputs and the same uniforms.

Accept lengths, emitted tokens and tree paths must be bit-exact, except for chain draws whose
oracle margin to a decision or CDF boundary is below 1e-5 relative (counted, reported, and
bounded). Tree and greedy results have no such exemption: argmax compares identical stored
values. Probabilities must agree within 1e-5 absolute (fp32 logits) and 2e-3 (bf16 logits).
"""

import numpy as np
import pytest
import torch

from golden_io import chain_cases, margin_cases, tree_cases
from gpu_util import compare_chain, dev, run_chain, run_tree
from workloads import (BF16, F32, ChainInputs, TreeInputs, bf16_to_f32, chain_128k, chain_32k,
                       chain_tiny, f32_to_bf16, make_uniforms, sweep_152k, tree_32k, tree_shape)

pytestmark = pytest.mark.gpu

PROB_TOL = {F32: 1e-5, BF16: 2e-3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_78_gb300 as sv
    sv.load_library()


# --------------------------------------------------------------------------- golden fixtures


@pytest.mark.parametrize("case", chain_cases(), ids=lambda c: c["name"])
def test_golden_chain(case):
    ci = ChainInputs(case["name"], case["target"], case["draft"], F32, case["tokens"],
                     case["uniforms"], case["T"])
    acc, out, st = run_chain(ci)
    assert st == 0
    np.testing.assert_array_equal(acc, case["accept_len"])
    np.testing.assert_array_equal(out, case["out_tokens"])


@pytest.mark.parametrize("case", margin_cases(), ids=lambda c: c["name"])
def test_golden_margin_cases(orc, case):
    """The hand-derived boundary cases (dyadic probabilities: the kernels' fp32 arithmetic is
    exact on them): the emitted tokens must be the hand-derived ones, and the per-draw
    comparison with the oracle must pass."""
    ci = ChainInputs(case["name"], case["target"], case["draft"], F32, case["tokens"],
                     case["uniforms"], float(np.float32(case["T"])))
    gpu = run_chain(ci)
    assert gpu[2] == 0
    np.testing.assert_array_equal(gpu[0], case["accept_len"])
    np.testing.assert_array_equal(gpu[1], case["out_tokens"])
    compare_chain(orc, ci, gpu)


@pytest.mark.parametrize("case", tree_cases(), ids=lambda c: c["name"])
def test_golden_tree(case):
    ti = TreeInputs(case["name"], case["target"], F32, case["parents"], case["tokens"])
    acc, path, out, st = run_tree(ti)
    assert st == 0
    np.testing.assert_array_equal(acc, case["accept_len"])
    np.testing.assert_array_equal(path, case["path_nodes"])
    np.testing.assert_array_equal(out, case["out_tokens"])


# --------------------------------------------------------------------------- the workloads


@pytest.mark.parametrize("offset", [0, 1])
def test_chain_tiny_1000_steps(orc, offset):
    """1000 B=1 steps batched, gamma=4, V=1000 fp32 (with offset=1 every row starts 4 bytes
    past a 16-byte boundary)."""
    ci = chain_tiny()
    gpu = run_chain(ci, offset_elems=offset)
    assert gpu[2] == 0
    flagged, fdiff, oa = compare_chain(orc, ci, gpu)
    assert 0 < oa.mean() < 4


def test_chain_32k_bf16(orc):
    ci = chain_32k()
    gpu = run_chain(ci)
    assert gpu[2] == 0
    compare_chain(orc, ci, gpu)


@pytest.mark.parametrize("sigma", [0.25, 1.0, 4.0])
def test_chain_128k_bf16_sigma_sweep(orc, sigma):
    """Full-size call (B=256, gamma=8, V=128256, bf16, T=0.7); the oracle checks every row for
    sigma = 1 and a 64-row sample otherwise."""
    ci = chain_128k(sigma=sigma)
    gpu = run_chain(ci)
    assert gpu[2] == 0
    rows = None if sigma == 1.0 else np.arange(0, ci.B, 4)
    compare_chain(orc, ci, gpu, rows=rows)


@pytest.mark.parametrize("B,gamma", [(1, 3), (1, 7), (16, 3), (16, 7), (128, 3), (128, 7)])
def test_sweep_152k_fp32(orc, B, gamma):
    ci = sweep_152k(B=B, gamma=gamma)
    gpu = run_chain(ci)
    assert gpu[2] == 0
    rows = None if B <= 16 else np.arange(0, B, B // 16)
    compare_chain(orc, ci, gpu, rows=rows)


@pytest.mark.parametrize("gamma", [3, 7])
def test_sweep_152k_fp32_largest(orc, gamma):
    """B=1024, V=152064 fp32: 4.4 GB (gamma 3) and 9.3 GB (gamma 7) of logits in one call;
    16 rows checked draw by draw."""
    ci = sweep_152k(B=1024, gamma=gamma)
    gpu = run_chain(ci)
    assert gpu[2] == 0
    compare_chain(orc, ci, gpu, rows=np.arange(0, 1024, 64))
    del ci


def test_tree_32k_bf16(orc):
    ti = tree_32k()
    acc, path, out, st = run_tree(ti)
    ra, rp, ro, rc = orc.verify_tree(ti.target, BF16, ti.parents, ti.tokens)
    assert st == 0 and rc == 0
    np.testing.assert_array_equal(acc, ra)
    np.testing.assert_array_equal(path, rp)
    np.testing.assert_array_equal(out, ro)
    assert acc.max() >= 2


def test_tree_32k_bf16_ties_at_the_maximum(orc):
    """Full-size tree call (32 trees x 64 nodes x 32000 bf16) whose every node holds its maximum
    at five ids: the lowest, the next element of the same 16-byte vector, one 600 ids on (same
    4 KB unit, another lane), one 2100 on (the next unit) and one 9000 on (four units later).
    Argmaxes, paths and bonus tokens bit-exact against the oracle (lowest index wins)."""
    ti = tree_32k(seed=40, tie_offsets=(1, 600, 2100, 9000))
    acc, path, out, st = run_tree(ti)
    ra, rp, ro, rc = orc.verify_tree(ti.target, BF16, ti.parents, ti.tokens)
    assert st == 0 and rc == 0
    np.testing.assert_array_equal(acc, ra)
    np.testing.assert_array_equal(path, rp)
    np.testing.assert_array_equal(out, ro)
    assert acc.max() >= 2
    # the bonus token is the lowest of the tied ids at the deepest accepted node
    des = ti.meta["designated"]
    best = path[np.arange(ti.B), acc]
    np.testing.assert_array_equal(out[np.arange(ti.B), acc], des[np.arange(ti.B), best])


# --------------------------------------------------------------------------- probabilities


@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("V,T", [(32000, 1.0), (1001, 0.7), (5, 100.0), (4097, 0.01),
                                 (3000, 0.0), (70001, 0.9), (70001, 0.0), (200000, 1.0)])
def test_probs(orc, dtype, V, T):
    """Rows held by one CTA, by clusters of 2..8 CTAs (V = 70001, and 200000 in bf16), and rows
    too long for a cluster (200000 in fp32), which take the stream kernel and write pass."""
    import speculative_decoding_verification_78_gb300 as sv
    k, _, cluster = sv.spec_launch_shape(sv.SPEC_CALL_PROBS, 37, 1, V, dtype, T)
    epv = 8 if dtype == BF16 else 4
    per_cta = 512 * (16 if dtype == BF16 else 8) * 4          # elements one CTA holds
    want = -(-((V // epv) * epv) // per_cta)
    if want <= 8:
        assert (k, cluster) == (1, max(want, 1))
    else:
        assert k == 2 and V == 200000 and dtype == F32
    rng = np.random.default_rng(V)
    x = (rng.standard_normal((37, V)) * 3).astype(np.float32)
    x[::5, ::7] = -np.inf      # masked entries
    lg = f32_to_bf16(x) if dtype == BF16 else x
    for off in (0, 1):
        pr, st = sv.probs(dev(lg, off), T)
        torch.cuda.synchronize()
        po, rc = orc.probs(lg, dtype, T)
        assert int(st.item()) == 0 and rc == 0
        err = np.abs(pr.cpu().numpy().astype(np.float64) - po).max()
        assert err <= PROB_TOL[dtype], err
        assert err <= 2e-6     # what the kernel actually reaches (fp32 arithmetic)


@pytest.mark.parametrize("dtype,V,rows", [(BF16, 32000, 700), (F32, 70001, 130), (F32, 3000, 1000)])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_probs_more_rows_than_resident(orc, dtype, V, rows, T):
    """More rows (or clusters) than the GPU holds at once at two CTAs per SM, so the launch runs
    in several waves. Rows 0 and 600 / 30 / 900 are invalid (NaN, all -inf): a flagged row in
    the first and in a later wave; unaligned rows (offset 1) exercise the head and tail
    elements."""
    import speculative_decoding_verification_78_gb300 as sv
    _, grid, cluster = sv.spec_launch_shape(sv.SPEC_CALL_PROBS, rows, 1, V, dtype, T)
    assert grid == rows * cluster
    rng = np.random.default_rng(V + rows)
    x = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    x[::3, ::11] = -np.inf
    bad = (0, rows - 100)
    x[bad[0], 5] = np.nan
    x[bad[1], :] = -np.inf
    lg = f32_to_bf16(x) if dtype == BF16 else x
    po, _ = orc.probs(lg, dtype, T)
    good = np.setdiff1d(np.arange(rows), bad)
    for off in (0, 1):
        pr, st = sv.probs(dev(lg, off), T)
        pr = pr.cpu().numpy()
        assert int(st.item()) == sv.SPEC_ERR_NONFINITE
        assert np.all(np.isnan(pr[list(bad)]))
        err = np.abs(pr[good].astype(np.float64) - po[good]).max()
        assert err <= 2e-6, err


@pytest.mark.parametrize("V", [300, 40000, 200000])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_probs_invalid_rows(V, T):
    """NaN, +inf and all -inf rows (one CTA, a cluster, the two-kernel path; sampling and
    greedy) are written as NaN and reported; the valid row is untouched."""
    import speculative_decoding_verification_78_gb300 as sv
    x = np.zeros((4, V), np.float32)
    x[0, V - 7] = np.nan
    x[1, V // 2] = np.inf
    x[2, :] = -np.inf
    pr, st = sv.probs(dev(x), T)
    p = pr.cpu().numpy()
    assert int(st.item()) == sv.SPEC_ERR_NONFINITE
    assert np.all(np.isnan(p[:3]))
    if T > 0:
        assert np.allclose(p[3], 1 / V)
    else:
        assert p[3, 0] == 1.0 and np.all(p[3, 1:] == 0.0)


# --------------------------------------------------------------------------- edge cases


def _chain_from(tgt, drf, tok, u, T, dtype=F32, name="edge"):
    return ChainInputs(name, tgt, drf, dtype, np.asarray(tok, np.int32), np.asarray(u, np.float32),
                       T)


def test_gamma_zero_and_vocab_one(orc):
    rng = np.random.default_rng(0)
    for V in (1, 2, 7, 300):
        tgt = (rng.standard_normal((50, 1, V)) * 2).astype(np.float32)
        ci = _chain_from(tgt, np.zeros((50, 0, V), np.float32), np.zeros((50, 0)),
                         make_uniforms(rng, (50, 1)), 1.0)
        gpu = run_chain(ci)
        assert gpu[2] == 0 and np.all(gpu[0] == 0)
        compare_chain(orc, ci, gpu)
    # V = 1: every draft is token 0 with p = q = 1, always accepted, bonus 0
    tgt = np.zeros((3, 4, 1), np.float32)
    ci = _chain_from(tgt, np.zeros((3, 3, 1), np.float32), np.zeros((3, 3)),
                     np.full((3, 4), 0.999, np.float32), 1.0)
    acc, out, st = run_chain(ci)
    assert st == 0 and np.all(acc == 3) and np.all(out == 0)


@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("V,offset", [(1001, 0), (1001, 1), (4099, 3), (257, 0)])
def test_ragged_vocab_and_unaligned_rows(orc, dtype, V, offset):
    ci = chain_32k(seed=11, B=40, gamma=3, V=V, dtype=dtype, peaked=5)
    gpu = run_chain(ci, offset_elems=offset)
    assert gpu[2] == 0
    compare_chain(orc, ci, gpu)


@pytest.mark.parametrize("T", [0.01, 0.3, 100.0])
def test_temperatures(orc, T):
    ci = chain_32k(seed=12, B=48, gamma=4, V=5000, temperature=T)
    gpu = run_chain(ci)
    assert gpu[2] == 0
    compare_chain(orc, ci, gpu)


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_greedy_chain_with_ties(orc, dtype):
    """T = 0 with small-integer logits (many exact ties, also across units far apart)."""
    rng = np.random.default_rng(3)
    B, g, V = 64, 6, 9000
    x = rng.integers(-4, 4, size=(B, g + 1, V)).astype(np.float32)
    x[:, :, [17, 4000, 8999]] = 9.0          # equal maxima in different units: lowest wins
    x[::3, :, 17] = 0.0                      # ... or the next one
    tgt = f32_to_bf16(x) if dtype == BF16 else x
    greedy = np.argmax(x, axis=2)
    tok = np.where(rng.random((B, g)) < 0.8, greedy[:, :g], rng.integers(0, V, (B, g)))
    ci = _chain_from(tgt, tgt[:, :g].copy(), tok, make_uniforms(rng, (B, g + 1)), 0.0, dtype)
    acc, out, st = run_chain(ci)
    oa, oo, _, rc = orc.verify_chain(tgt, None, dtype, ci.tokens, ci.uniforms, 0.0)
    assert st == 0 and rc == 0
    np.testing.assert_array_equal(acc, oa)
    np.testing.assert_array_equal(out, oo)


def test_all_accept_and_first_reject(orc):
    rng = np.random.default_rng(4)
    B, g, V = 32, 5, 3000
    t = (rng.standard_normal((B, g + 1, V)) * 2).astype(np.float32)
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    # draft == target: every ratio is 1, all drafts accepted
    ci = _chain_from(t, t[:, :g].copy(), tok, make_uniforms(rng, (B, g + 1)), 1.0)
    acc, out, st = run_chain(ci)
    assert st == 0 and np.all(acc == g)
    compare_chain(orc, ci, (acc, out, st))
    # the target gives the first draft token probability 0: rejected at position 0
    t2 = t.copy()
    t2[np.arange(B), 0, tok[:, 0]] = -np.inf
    ci2 = _chain_from(t2, t[:, :g].copy(), tok, ci.uniforms, 1.0)
    acc2, out2, st2 = run_chain(ci2)
    assert st2 == 0 and np.all(acc2 == 0)
    assert np.all(out2[:, 0] != tok[:, 0])
    compare_chain(orc, ci2, (acc2, out2, st2))


def test_long_draft_gamma_40(orc):
    ci = chain_32k(seed=13, B=8, gamma=40, V=2000, peaked=3)
    # a near-copy draft so that acceptance runs past 32 positions
    ci.draft = ci.target[:, :40].copy()
    gpu = run_chain(ci)
    assert gpu[2] == 0
    compare_chain(orc, ci, gpu)
    assert gpu[0].max() > 32


@pytest.mark.parametrize("gamma,V,dtype,kernels", [(4, 1000, F32, 2), (15, 2000, BF16, 2),
                                                   (20, 500, F32, 2), (31, 1024, F32, 2)])
def test_single_unit_rows(orc, gamma, V, dtype, kernels):
    """Rows of one unit, up to 63 rows per batch row: the stream kernel plus the one-warp
    finish, ragged and unaligned."""
    import speculative_decoding_verification_78_gb300 as sv
    B = 200
    assert sv.spec_launch_shape(sv.SPEC_CALL_CHAIN, B, 2 * gamma + 1, V, dtype,
                                1.0)[0] == kernels
    ci = chain_32k(seed=17 + gamma, B=B, gamma=gamma, V=V, dtype=dtype, peaked=4, boost=3.0)
    ci.draft = (ci.draft if gamma < 20 else ci.target[:, :gamma].copy())
    for off in (0, 1):
        gpu = run_chain(ci, offset_elems=off)
        assert gpu[2] == 0
        compare_chain(orc, ci, gpu)


def test_largest_vocab(orc):
    rng = np.random.default_rng(5)
    V = 1 << 20
    t = (rng.standard_normal((2, 2, V)) * 2).astype(np.float32)
    d = t[:, :1] + (rng.standard_normal((2, 1, V)) * 0.5).astype(np.float32)
    ci = _chain_from(t, d, rng.integers(0, V, (2, 1)), make_uniforms(rng, (2, 2)), 1.0)
    gpu = run_chain(ci)
    assert gpu[2] == 0
    compare_chain(orc, ci, gpu)


def test_invalid_rows_report_and_isolate(orc):
    import speculative_decoding_verification_78_gb300 as sv
    ci = chain_32k(seed=14, B=6, gamma=3, V=700, dtype=F32)
    ci.target[1, 3, 5] = np.nan          # NaN in the bonus row: the whole step is invalid
    ci.draft[2, 0, 9] = np.inf
    ci.target[3, 1, :] = -np.inf         # no finite value
    ci.tokens[4, 2] = 700                # token out of range
    acc, out, st = run_chain(ci)
    oa, oo, _, _ = orc.verify_chain(ci.target, ci.draft, F32, ci.tokens, ci.uniforms, 1.0)
    assert st in (sv.SPEC_ERR_NONFINITE, sv.SPEC_ERR_TOKEN)
    assert list(acc[1:5]) == [-1, -1, -1, -1] and np.all(out[1:5] == -1)
    np.testing.assert_array_equal(acc, oa)
    for b in (0, 5):
        np.testing.assert_array_equal(out[b], oo[b])


def test_tree_shapes_and_errors(orc):
    import speculative_decoding_verification_78_gb300 as sv
    rng = np.random.default_rng(6)
    V = 600
    for N, kind in [(1, "root"), (9, "chain"), (12, "star"), (64, "rule"), (1024, "random"),
                    (300, "chain"), (33, "random"), (63, "chain"), (65, "random"), (64, "chain")]:
        B = 6
        if kind == "root":
            par = np.full((B, 1), -1, np.int32)
        elif kind == "chain":
            par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (B, 1))
        elif kind == "star":
            par = np.tile(np.array([-1] + [0] * (N - 1), np.int32), (B, 1))
        elif kind == "rule":
            par = np.stack([tree_shape(rng, N) for _ in range(B)])
        else:
            par = np.stack([np.array([-1] + [int(rng.integers(0, i)) for i in range(1, N)])
                            for _ in range(B)]).astype(np.int32)
        x = rng.integers(-3, 3, size=(B, N, V)).astype(np.float32)
        tgt = f32_to_bf16(x)
        g = np.argmax(bf16_to_f32(tgt), axis=2)
        tok = np.where(rng.random((B, N)) < 0.85, np.take_along_axis(g, np.maximum(par, 0), 1),
                       rng.integers(0, V, (B, N))).astype(np.int32)
        if kind == "star":
            tok[:, 1:] = g[:, :1]          # duplicate siblings, all accepted: node 1 wins
        ti = TreeInputs(kind, tgt, BF16, par, tok)
        acc, path, out, st = run_tree(ti)
        ra, rp, ro, rc = orc.verify_tree(tgt, BF16, par, tok)
        assert st == 0 and rc == 0, kind
        np.testing.assert_array_equal(acc, ra)
        np.testing.assert_array_equal(path, rp)
        np.testing.assert_array_equal(out, ro)
    # invalid parents / tokens / rows: reported per row, others unaffected
    par = np.tile(np.array([-1, 0, 0, 1], np.int32), (5, 1))
    tgt = np.zeros((5, 4, 50), np.float32)
    tok = np.zeros((5, 4), np.int32)
    par[1, 0] = 0
    par[2, 3] = 3
    tok[3, 2] = 50
    tgt[4, 2, 1] = np.nan
    ti = TreeInputs("bad", tgt, F32, par, tok)
    acc, path, out, st = run_tree(ti)
    ra, rp, ro, _ = orc.verify_tree(tgt, F32, par, tok)
    assert st in (sv.SPEC_ERR_PARENT, sv.SPEC_ERR_TOKEN, sv.SPEC_ERR_NONFINITE)
    assert list(acc) == [2, -1, -1, -1, -1]
    np.testing.assert_array_equal(acc, ra)
    np.testing.assert_array_equal(path[0], rp[0])
    assert np.all(path[1:] == -1) and np.all(out[1:] == -1)
    # one kind of error at a time, in a small (<= 64 nodes) and a large tree: the exact code
    for N in (4, 80):
        for what, want in (("parent", sv.SPEC_ERR_PARENT), ("token", sv.SPEC_ERR_TOKEN),
                           ("row", sv.SPEC_ERR_NONFINITE)):
            par = np.tile(np.arange(-1, N - 1, dtype=np.int32), (3, 1))
            tgt = np.zeros((3, N, 50), np.float32)
            tok = np.zeros((3, N), np.int32)
            if what == "parent":
                par[1, N - 1] = N - 1
            elif what == "token":
                tok[1, N - 2] = -5
            else:
                tgt[1, N - 1, 7] = np.inf
            acc, path, out, st = run_tree(TreeInputs(what, tgt, F32, par, tok))
            ra, rp, ro, _ = orc.verify_tree(tgt, F32, par, tok)
            assert st == want, (N, what, st)
            np.testing.assert_array_equal(acc, ra)
            np.testing.assert_array_equal(path, rp)
            np.testing.assert_array_equal(out, ro)


def test_deterministic_and_workspace_reuse(orc):
    """The workspace is scratch: whatever it holds before a call (here garbage bytes, then the
    previous call's leftovers) does not change the result."""
    import speculative_decoding_verification_78_gb300 as sv
    ci = chain_32k(seed=15, B=32, gamma=5, V=8000)
    ws = sv.new_workspace(ci.B, 2 * ci.gamma + 1, ci.V, sv.SPEC_BF16)
    ws.fill_(0xA5)
    first = run_chain(ci, workspace=ws)
    for k in range(3):
        if k == 1:
            ws.fill_(0xFF)   # NaN bit patterns everywhere
        again = run_chain(ci, workspace=ws)
        assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])
        assert again[2] == 0
    compare_chain(orc, ci, first)


# --------------------------------------------------------------------------- more chain shapes


@pytest.mark.parametrize("B,gamma,V,dtype,T", [
    (1, 5, 32000, BF16, 0.7),      # one batch row
    (3, 15, 4096, BF16, 1.3),      # 31 rows per batch row
    (16, 2, 32000, F32, 1.0),
    (40, 1, 8, BF16, 1.0),         # one 16-byte vector per row
    (7, 3, 6000, F32, 0.05),       # near-greedy temperature
])
def test_chain_shapes_masked_and_all_accepting(orc, B, gamma, V, dtype, T):
    """Chain shapes with masked (-inf) entries in every row and every fourth step accepting all
    its drafts (draft == target), at an aligned and an unaligned base, against the oracle draw
    by draw."""
    ci = chain_32k(seed=50 + gamma, B=B, gamma=gamma, V=V, dtype=dtype, temperature=T,
                   peaked=min(50, V // 4))
    if V > 16:
        t = bf16_to_f32(ci.target) if dtype == BF16 else ci.target
        t[:, :, 3::11] = -np.inf                 # masked tokens in every row
        ci.target = f32_to_bf16(t) if dtype == BF16 else t
        ci.tokens[:, :] = np.where(ci.tokens % 11 == 3, (ci.tokens + 1) % V, ci.tokens)
    ci.draft[::4] = ci.target[::4, :gamma]       # every fourth step accepts all its drafts
    for off in (0, 1):
        gpu = run_chain(ci, offset_elems=off)
        assert gpu[2] == 0
        compare_chain(orc, ci, gpu)
        assert gpu[0][::4].min() == gamma


def test_chain_invalid_rows_and_repeats(orc):
    """Invalid batch rows (NaN in the bonus row, +inf in a draft row, a target row with no
    finite value, a token out of range) report -1 and a status; the other rows are unaffected,
    and repeated calls are bit-identical."""
    import speculative_decoding_verification_78_gb300 as sv
    ci = chain_32k(seed=61, B=12, gamma=5, V=4096, dtype=F32)
    ci.target[1, 5, 100] = np.nan
    ci.draft[2, 0, 4000] = np.inf
    ci.target[3, 1, :] = -np.inf
    ci.tokens[4, 3] = 4096
    first = run_chain(ci)
    assert first[2] in (sv.SPEC_ERR_NONFINITE, sv.SPEC_ERR_TOKEN)
    assert list(first[0][1:5]) == [-1, -1, -1, -1] and np.all(first[1][1:5] == -1)
    good = np.array([0] + list(range(5, 12)))
    compare_chain(orc, ci, first, rows=good)
    for _ in range(2):
        again = run_chain(ci)
        np.testing.assert_array_equal(again[0], first[0])
        np.testing.assert_array_equal(again[1], first[1])


def test_concurrent_calls_on_separate_streams(orc):
    """Two chain calls and a greedy-tree call in flight at once on three streams, each with its
    own workspace and outputs, launched back to back three times over: every result equals the
    oracle's (no state is shared between calls beyond cached device attributes)."""
    import speculative_decoding_verification_78_gb300 as sv
    a = chain_32k(seed=61, B=48, gamma=5, V=32000)
    c = chain_tiny(seed=62, B=400, gamma=4)
    t = tree_32k(seed=63, B=16, N=64, V=32000)
    streams = [torch.cuda.Stream() for _ in range(3)]
    ins_a = (dev(a.target), dev(a.draft), dev(a.tokens), dev(a.uniforms))
    ins_c = (dev(c.target), dev(c.draft), dev(c.tokens), dev(c.uniforms))
    ins_t = (dev(t.target), dev(t.parents), dev(t.tokens))
    torch.cuda.synchronize()
    results = []
    for _ in range(3):
        with torch.cuda.stream(streams[0]):
            ra = sv.verify_chain(*ins_a, a.temperature, stream=streams[0])
        with torch.cuda.stream(streams[1]):
            rc = sv.verify_chain(*ins_c, c.temperature, stream=streams[1])
        with torch.cuda.stream(streams[2]):
            rt = sv.verify_tree(*ins_t, stream=streams[2])
        results.append((ra, rc, rt))
    torch.cuda.synchronize()
    oa = orc.verify_tree(t.target, BF16, t.parents, t.tokens)
    for ra, rc, rt in results:
        for ci, r in ((a, ra), (c, rc)):
            assert int(r[2].item()) == 0
            compare_chain(orc, ci, (r[0].cpu().numpy(), r[1].cpu().numpy(), 0))
        assert int(rt[3].item()) == 0 and oa[3] == 0
        for got, want in zip(rt[:3], oa[:3]):
            np.testing.assert_array_equal(got.cpu().numpy(), want)

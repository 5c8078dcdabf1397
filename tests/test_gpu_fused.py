"""GPU parity of the fused single-kernel path (one thread-block cluster per batch row) against
the CPU oracle, for every cluster size it uses, ragged and unaligned rows, long drafts, greedy
chains, small and large trees, and invalid rows. Each case first asserts through
spec_launch_shape that the call really takes the fused path (and, on a 152-SM GB300, with the
cluster size the case was chosen for)."""

import numpy as np
import pytest
import torch

from gpu_util import compare_chain, run_chain, run_tree
from workloads import BF16, F32, ChainInputs, TreeInputs, chain_32k, tree_32k

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_78_gb300 as sv
    sv.load_library()


def _sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _assert_fused(kind, B, rows, V, dtype, T, cluster):
    import speculative_decoding_verification_78_gb300 as sv
    k, g, c = sv.spec_launch_shape(kind, B, rows, V, dtype, T)
    assert k == 1, (B, rows, V, "not fused")
    assert g == B * c
    if _sm_count() == 152:
        assert c == cluster, (B, rows, V, c)


# (B, gamma, V, dtype, T, row offset, cluster on 152 SMs)
CHAIN_CASES = [
    (24, 3, 20000, BF16, 1.0, 0, 8),
    (60, 2, 9000, F32, 0.7, 0, 4),
    (100, 4, 4099, BF16, 1.0, 1, 2),
    (160, 6, 2500, F32, 1.3, 0, 1),
    (80, 60, 4096, BF16, 1.0, 0, 2),
    (24, 5, 20000, BF16, 0.0, 0, 8),
    (160, 3, 3001, F32, 0.0, 1, 1),
]


@pytest.mark.parametrize("B,gamma,V,dtype,T,offset,cluster", CHAIN_CASES)
def test_fused_chain(orc, B, gamma, V, dtype, T, offset, cluster):
    import speculative_decoding_verification_78_gb300 as sv
    _assert_fused(sv.SPEC_CALL_CHAIN, B, 2 * gamma + 1, V, dtype, T, cluster)
    ci = chain_32k(seed=100 + B + gamma, B=B, gamma=gamma, V=V, dtype=dtype, temperature=T,
                   peaked=min(50, V // 8))
    # draft tokens in the rows' unaligned head and tail elements as well
    tok = ci.tokens.copy()
    tok[::3, 0] = np.arange(0, B, 3) % 7
    if gamma > 1:
        tok[1::3, 1] = V - 1 - (np.arange(1, B, 3) % 4)
    ci = ChainInputs(ci.name, ci.target, ci.draft if T > 0 else ci.draft[:, :0], dtype, tok,
                     ci.uniforms, T, ci.meta)
    gpu = run_chain(ci, offset_elems=offset)
    assert gpu[2] == 0
    compare_chain(orc, ci, gpu)


# (B, N, V, dtype, cluster on 152 SMs): N <= 64 takes the warp finish, N > 64 the CTA one
TREE_CASES = [
    (20, 64, 20000, BF16, 8),
    (20, 100, 20000, BF16, 8),
    (40, 9, 12000, F32, 4),
    (160, 33, 2051, BF16, 1),
]


@pytest.mark.parametrize("B,N,V,dtype,cluster", TREE_CASES)
def test_fused_tree(orc, B, N, V, dtype, cluster):
    import speculative_decoding_verification_78_gb300 as sv
    _assert_fused(sv.SPEC_CALL_TREE, B, N, V, dtype, 0.0, cluster)
    ti = tree_32k(seed=200 + N, B=B, N=N, V=V, dtype=dtype, peaked=min(50, V // 8))
    acc, path, out, st = run_tree(ti, offset_elems=1 if V % 8 else 0)
    ra, rp, ro, rc = orc.verify_tree(ti.target, dtype, ti.parents, ti.tokens)
    assert st == 0 and rc == 0
    np.testing.assert_array_equal(acc, ra)
    np.testing.assert_array_equal(path, rp)
    np.testing.assert_array_equal(out, ro)
    assert acc.max() >= 2


def test_fused_invalid_rows_isolated(orc):
    """A NaN logit, a +inf logit, a draft token outside [0, V) and an all -inf row, each in its
    own batch row of a fused call: those rows report -1, every other row matches the oracle."""
    import speculative_decoding_verification_78_gb300 as sv
    B, gamma, V = 24, 3, 20000
    _assert_fused(sv.SPEC_CALL_CHAIN, B, 2 * gamma + 1, V, F32, 1.0, 8)
    ci = chain_32k(seed=321, B=B, gamma=gamma, V=V, dtype=F32)
    tgt, drf, tok = ci.target.copy(), ci.draft.copy(), ci.tokens.copy()
    tgt[2, 1, 17] = np.nan
    drf[5, 0, V - 1] = np.inf
    tok[9, 2] = V
    tgt[13, gamma, :] = -np.inf
    ci = ChainInputs("bad", tgt, drf, F32, tok, ci.uniforms, 1.0, ci.meta)
    acc, out, st = run_chain(ci)
    assert st in (sv.SPEC_ERR_NONFINITE, sv.SPEC_ERR_TOKEN)
    bad = [2, 5, 9, 13]
    assert all(acc[b] == -1 and np.all(out[b] == -1) for b in bad)
    good = np.array([b for b in range(B) if b not in bad])
    compare_chain(orc, ci, (acc, out, st), rows=good)


def test_fused_tree_errors(orc):
    import speculative_decoding_verification_78_gb300 as sv
    B, N, V = 20, 64, 20000
    _assert_fused(sv.SPEC_CALL_TREE, B, N, V, BF16, 0.0, 8)
    ti = tree_32k(seed=77, B=B, N=N, V=V)
    par, tok, tgt = ti.parents.copy(), ti.tokens.copy(), ti.target.copy()
    par[3, 10] = 10
    tok[7, 5] = -1
    tgt[11, 40, 123] = 0x7fc0   # a bf16 NaN
    acc, path, out, st = run_tree(TreeInputs("bad", tgt, BF16, par, tok))
    ra, rp, ro, _ = orc.verify_tree(tgt, BF16, par, tok)
    assert st in (sv.SPEC_ERR_PARENT, sv.SPEC_ERR_TOKEN, sv.SPEC_ERR_NONFINITE)
    np.testing.assert_array_equal(acc, ra)
    np.testing.assert_array_equal(path, rp)
    np.testing.assert_array_equal(out, ro)
    assert list(acc[[3, 7, 11]]) == [-1, -1, -1]

"""GPU parity of the drafter-side helpers against the oracle: sampling (tokens bit-exact except
draws within 1e-5 of a CDF boundary, which must still be valid tokens), top-n candidates and the
tree-attention mask (bit-exact), including ragged, unaligned and invalid rows."""

import numpy as np
import pytest
import torch

from gpu_util import compare_sample, dev
from workloads import BF16, F32, f32_to_bf16, make_uniforms, tree_shape

pytestmark = pytest.mark.gpu

MARGIN = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_78_gb300 as sv
    sv.load_library()


@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("V,T", [(5, 1.0), (1000, 0.7), (32000, 1.0), (128256, 0.7),
                                 (3001, 0.0), (70000, 1.0)])
def test_sample(orc, dtype, V, T):
    import speculative_decoding_verification_78_gb300 as sv
    rng = np.random.default_rng(V + int(10 * T))
    rows = 64
    x = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    x[:, 1::9] = -np.inf
    lg = f32_to_bf16(x) if dtype == BF16 else x
    u = make_uniforms(rng, (rows,))
    _, _, rc = orc.sample(lg, dtype, u, T)
    assert rc == 0
    for off in (0, 1):
        tok, st = sv.sample(dev(lg, off), T, dev(u))
        torch.cuda.synchronize()
        tok = tok.cpu().numpy()
        assert int(st.item()) == 0
        # a draw within MARGIN of a CDF boundary (common for long, flat rows) must land in the
        # oracle's band for it; every other draw must match exactly
        flagged = compare_sample(orc, lg, dtype, u, T, tok)
        assert flagged <= rows // 2


def test_sample_invalid_rows(orc):
    import speculative_decoding_verification_78_gb300 as sv
    x = np.zeros((4, 500), np.float32)
    x[0, 3] = np.nan
    x[2, :] = -np.inf
    u = np.full(4, 0.3137, np.float32)   # u * 500 falls between two CDF steps
    tok, st = sv.sample(dev(x), 1.0, dev(u))
    tok = tok.cpu().numpy()
    assert int(st.item()) == sv.SPEC_ERR_NONFINITE
    want, _, _ = orc.sample(x, F32, u, 1.0)
    np.testing.assert_array_equal(tok, want)


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_sample_invalid_rows_multi_unit(orc, dtype):
    """Rows of several units on 16-byte boundaries (the one-warp-per-row sampling finisher):
    a NaN, an all -inf and a +inf row are flagged, the other rows still sampled."""
    import speculative_decoding_verification_78_gb300 as sv
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((6, 40000)) * 3).astype(np.float32)
    x[1, 17] = np.nan
    x[3, :] = -np.inf
    x[4, 39999] = np.inf
    lg = f32_to_bf16(x) if dtype == BF16 else x
    u = make_uniforms(rng, (6,))
    tok, st = sv.sample(dev(lg), 1.0, dev(u))
    tok = tok.cpu().numpy()
    assert int(st.item()) == sv.SPEC_ERR_NONFINITE
    assert list(tok[[1, 3, 4]]) == [-1, -1, -1]
    compare_sample(orc, lg, dtype, u, 1.0, tok)


@pytest.mark.parametrize("dtype", [F32, BF16])
@pytest.mark.parametrize("V,k", [(16, 16), (1001, 3), (32000, 8), (152064, 16), (5, 1),
                                 (40000, 5)])
def test_topk(orc, dtype, V, k):
    import speculative_decoding_verification_78_gb300 as sv
    rng = np.random.default_rng(V * 17 + k)
    rows = 48
    x = rng.integers(-40, 40, size=(rows, V)).astype(np.float32)   # many ties
    x[:, 1::13] = -np.inf
    x[0, :] = 3.0                                                  # an all-equal row
    lg = f32_to_bf16(x) if dtype == BF16 else x
    want, rc = orc.topk(lg, dtype, k)
    assert rc == 0
    for off in (0, 1):
        idx, st = sv.topk(dev(lg, off), k)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        np.testing.assert_array_equal(idx.cpu().numpy(), want)


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_topk_signed_zero_ties(orc, dtype):
    """-0.0 and +0.0 are equal values: the lower index ranks first, whatever the signs."""
    import speculative_decoding_verification_78_gb300 as sv
    rng = np.random.default_rng(7)
    x = -np.abs(rng.standard_normal((8, 5000))).astype(np.float32) - 1.0
    for r in range(8):
        cols = rng.choice(5000, size=6, replace=False)
        x[r, cols] = np.where(rng.random(6) < 0.5, -0.0, 0.0).astype(np.float32)
    lg = f32_to_bf16(x) if dtype == BF16 else x
    want, rc = orc.topk(lg, dtype, 4)
    assert rc == 0
    idx, st = sv.topk(dev(lg), 4)
    assert int(st.item()) == 0
    np.testing.assert_array_equal(idx.cpu().numpy(), want)


def test_topk_invalid_rows(orc):
    import speculative_decoding_verification_78_gb300 as sv
    x = np.zeros((5, 300), np.float32)
    x[0, 7] = np.nan
    x[1, 0] = np.inf
    x[2, :] = -np.inf
    x[3, 1:] = -np.inf             # one finite value: the rest are ranked by index
    idx, st = sv.topk(dev(x), 4)
    idx = idx.cpu().numpy()
    assert int(st.item()) == sv.SPEC_ERR_NONFINITE
    want, _ = orc.topk(x, F32, 4)
    np.testing.assert_array_equal(idx, want)
    assert list(idx[3]) == [0, 1, 2, 3]


@pytest.mark.parametrize("N", [1, 31, 32, 33, 64, 100, 1024])
def test_tree_mask(orc, N):
    import speculative_decoding_verification_78_gb300 as sv
    rng = np.random.default_rng(N)
    B = 6
    if N <= 64:
        par = np.stack([tree_shape(rng, N) for _ in range(B)])
    else:
        par = np.stack([np.array([-1] + [int(rng.integers(max(0, i - 3), i)) for i in
                                         range(1, N)]) for _ in range(B)])   # deep trees
    par = par.astype(np.int32)
    want, rc = orc.tree_mask(par)
    assert rc == 0
    m, st = sv.tree_mask(dev(par))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    np.testing.assert_array_equal(m.cpu().numpy().view(np.uint32), want)


def test_tree_mask_invalid_tree(orc):
    import speculative_decoding_verification_78_gb300 as sv
    par = np.array([[-1, 0, 1, 1], [0, 0, 1, 2], [-1, 0, 3, 1]], np.int32)
    want, _ = orc.tree_mask(par)
    m, st = sv.tree_mask(dev(par))
    assert int(st.item()) == sv.SPEC_ERR_PARENT
    np.testing.assert_array_equal(m.cpu().numpy().view(np.uint32), want)

"""The checked build (libspec_verify_checked.so: the kernels compiled with SPEC_CHECKED, every
index they compute range-checked before it addresses memory, a violation reported as
SPEC_ERR_CHECK through the status word and the access skipped) on small cases of every entry
point: no check may fire, and every output must equal the normal library's. Stands in for a
memory sanitizer, which this GPU pool does not offer."""

import numpy as np
import pytest
import torch

from gpu_util import dev
from workloads import (BF16, F32, chain_32k, chain_tiny, make_uniforms, tree_32k,
                       tree_sample_32k)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def both():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_78_gb300._binding as bnd
    return bnd, bnd.load_library(), bnd.load_library(checked=True)


def _run(bnd, lib, fn, *args, **kw):
    """Calls binding function `fn` with the given library loaded in place of the normal one."""
    saved = bnd.load_library
    bnd.load_library = lambda checked=False: lib
    try:
        return fn(*args, **kw)
    finally:
        bnd.load_library = saved


def _np(ts):
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in ts]


@pytest.mark.parametrize("case", ["chain_bf16", "chain_fp32_unaligned", "chain_greedy",
                                  "chain_single_unit", "chain_gamma0"])
def test_checked_chain(both, case):
    bnd, lib, clib = both
    off = 0
    if case == "chain_bf16":
        ci = chain_32k(seed=71, B=12, gamma=5, V=9000)
    elif case == "chain_fp32_unaligned":
        ci = chain_32k(seed=72, B=9, gamma=3, V=4099, dtype=F32)
        off = 1
    elif case == "chain_greedy":
        ci = chain_32k(seed=73, B=10, gamma=4, V=7000, temperature=0.0)
    elif case == "chain_single_unit":
        ci = chain_tiny(seed=74, B=50, gamma=4)
    else:
        ci = chain_32k(seed=75, B=20, gamma=0, V=5000)
    args = (dev(ci.target, off), dev(ci.draft, off) if ci.draft.size else None,
            dev(ci.tokens) if ci.tokens.size else None, dev(ci.uniforms), ci.temperature)
    want = _np(_run(bnd, lib, bnd.verify_chain, *args))
    got = _np(_run(bnd, clib, bnd.verify_chain, *args))
    assert int(got[2][0]) == 0, bnd.spec_status_string(int(got[2][0]))
    np.testing.assert_array_equal(got[0], want[0])
    np.testing.assert_array_equal(got[1], want[1])


@pytest.mark.parametrize("N", [64, 150])
def test_checked_trees(both, N):
    bnd, lib, clib = both
    ti = tree_32k(seed=76, B=4, N=N, V=3000)
    args = (dev(ti.target), dev(ti.parents), dev(ti.tokens))
    want = _np(_run(bnd, lib, bnd.verify_tree, *args))
    got = _np(_run(bnd, clib, bnd.verify_tree, *args))
    assert int(got[3][0]) == 0
    for g, w in zip(got[:3], want[:3]):
        np.testing.assert_array_equal(g, w)
    ts = tree_sample_32k(seed=77, B=4, N=N, V=3000)
    args = (dev(ts.target), dev(ts.meta["draft"]), dev(ts.parents), dev(ts.tokens),
            dev(ts.meta["uniforms"]), 1.0)
    want = _np(_run(bnd, lib, bnd.verify_tree_sample, *args))
    got = _np(_run(bnd, clib, bnd.verify_tree_sample, *args))
    assert int(got[3][0]) == 0
    for g, w in zip(got[:3], want[:3]):
        np.testing.assert_array_equal(g, w)
    m = _np(_run(bnd, clib, bnd.tree_mask, dev(ti.parents)))
    w = _np(_run(bnd, lib, bnd.tree_mask, dev(ti.parents)))
    assert int(m[1][0]) == 0
    np.testing.assert_array_equal(m[0], w[0])


@pytest.mark.parametrize("dtype,V,T", [(BF16, 32000, 1.0), (F32, 70001, 0.0), (F32, 200000, 1.0),
                                       (BF16, 1001, 0.7)])
def test_checked_probs_sample_topk(both, dtype, V, T):
    bnd, lib, clib = both
    rng = np.random.default_rng(V)
    x = (rng.standard_normal((9, V)) * 3).astype(np.float32)
    from workloads import f32_to_bf16
    lg = dev(f32_to_bf16(x) if dtype == BF16 else x)
    u = dev(make_uniforms(rng, (9,)))
    for fn, args in ((bnd.probs, (lg, T)), (bnd.sample, (lg, T, u)), (bnd.topk, (lg, 5))):
        want = _np(_run(bnd, lib, fn, *args))
        got = _np(_run(bnd, clib, fn, *args))
        assert int(got[-1][0]) == 0, (fn.__name__, int(got[-1][0]))
        np.testing.assert_array_equal(got[0], want[0])


def test_checked_lmhead(both, orc):
    """The fused LM-head call (tensor-core GEMM epilogue, then the chain finisher) through the
    checked build: no check fires and every output, logits included, equals the plain build's."""
    from workloads import lmhead_grid
    bnd, lib, clib = both
    li = lmhead_grid(seed=9, B=6, gamma=3, V=768, Ht=128, Hd=64)
    rng = np.random.default_rng(9)
    tok = dev(rng.integers(0, 768, (6, 3)).astype(np.int32))
    args = (dev(li.hidden_t), dev(li.head_t), dev(li.hidden_d), dev(li.head_d), tok,
            dev(li.uniforms), 1.0)
    bits = lambda ts: [t.view(torch.int16) if t.dtype == torch.bfloat16 else t for t in ts]
    want = _np(bits(_run(bnd, lib, bnd.verify_chain_lmhead, *args)))
    got = _np(bits(_run(bnd, clib, bnd.verify_chain_lmhead, *args)))
    assert int(got[2][0]) == 0 and int(want[2][0]) == 0
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)

"""spec_verify_chain_static -- chain verification whose scratch is a static device array inside
the library -- against spec_verify_chain with a caller-owned workspace and against the CPU oracle: identical
outputs on calls in a row (different shapes, sampling and greedy, sharing the one static array),
and a call that needs more scratch than the array holds refused before anything is enqueued.
Collected last, and independent of what ran before it."""

import ctypes

import numpy as np
import pytest
import torch

from gpu_util import compare_chain, dev
from workloads import chain_32k, chain_tiny

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_78_gb300 as sv
    sv.load_library()


def _static_call(ci):
    import speculative_decoding_verification_78_gb300 as sv
    tg, dr, tok, uni = dev(ci.target), dev(ci.draft), dev(ci.tokens), dev(ci.uniforms)
    B, g1, V = ci.target.shape
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, g1), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = sv.spec_verify_chain_static(tg, dr, tok, uni, ci.temperature, acc, out, st)
    return rc, (tg, dr, tok, uni), acc, out, st


def test_static_scratch_matches_workspace_entry_point(orc):
    """Sampling (T = 1) and greedy (T = 0) calls, each shape against both the workspace entry
    point (identical outputs) and the oracle (the per-draw comparison of the parity tests)."""
    import speculative_decoding_verification_78_gb300 as sv
    greedy = chain_32k(seed=43, B=16, gamma=4, V=9000, temperature=0.0)
    cases = [chain_32k(seed=41, B=8, gamma=5, V=100000), chain_tiny(seed=42, B=300, gamma=20),
             greedy]
    for ci in cases:   # every shape takes the two-kernel path, which uses the scratch
        B, g1, V = ci.target.shape
        assert sv.spec_launch_shape(sv.SPEC_CALL_CHAIN, B, 2 * g1 - 1, V, ci.dtype,
                                    ci.temperature)[0] == 2
        assert 0 < sv.spec_workspace_bytes(B, 2 * g1 - 1, V, ci.dtype) <= \
            sv.SPEC_STATIC_SCRATCH_BYTES
    # two calls in a row on one stream, the second reusing the static scratch of the first
    runs = [_static_call(ci) for ci in cases]
    torch.cuda.synchronize()
    for ci, (rc, inputs, acc_s, out_s, st_s) in zip(cases, runs):
        assert rc == sv.SPEC_OK
        acc, out, st = sv.verify_chain(*inputs, ci.temperature)
        torch.cuda.synchronize()
        assert int(st_s.item()) == 0 and int(st.item()) == 0
        np.testing.assert_array_equal(acc_s.cpu().numpy(), acc.cpu().numpy())
        np.testing.assert_array_equal(out_s.cpu().numpy(), out.cpu().numpy())
        assert (acc.cpu().numpy() >= 0).all()
        compare_chain(orc, ci, (acc_s.cpu().numpy(), out_s.cpu().numpy(), 0))


def test_static_scratch_refuses_oversized_calls():
    import speculative_decoding_verification_78_gb300 as sv
    B, gamma, V = 1024, 7, 152064
    assert sv.spec_workspace_bytes(B, 2 * gamma + 1, V, sv.SPEC_F32) > \
        sv.SPEC_STATIC_SCRATCH_BYTES
    lib = sv.load_library()
    t = torch.zeros(16, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(t.data_ptr())
    rc = lib.spec_verify_chain_static(p, p, sv.SPEC_F32, p, p, B, gamma, V, ctypes.c_float(1.0),
                                      p, p, p, None)
    assert rc == sv.SPEC_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert float(t.abs().sum().item()) == 0.0   # nothing was written

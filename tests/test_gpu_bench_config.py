"""Parity in the launch configuration the benchmark times: the bench's own CUDA graphs (blocks
of 16 back-to-back calls of each kind over its rotated input copies, consecutive kernels
overlapping through programmatic launches) on the full-size step inputs (chain 64 x 5 x 32000,
tree 32 x 64 x 32000, probabilities of the chain's 384 target rows, all bf16), checked against
the oracle on every copy's outputs."""

import os
import sys

import numpy as np
import pytest
import torch

from gpu_util import compare_chain
from workloads import BF16

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_78_gb300 as sv
    sv.load_library()


def test_bench_block_graphs_match_oracle(orc):
    sys.path.insert(0, ROOT)
    import bench
    ci, ti = bench.make_inputs(0)
    r = bench.Runner(ci, ti, torch.device("cuda", 0))
    r.capture()
    # poison every output so that only values written by the replay can pass
    for c in r.copies:
        for key in ("acc", "out", "tacc", "tpath", "tout"):
            c[key].fill_(-7)
        c["probs"].fill_(float("nan"))
    with torch.cuda.stream(r.stream):
        for kind in bench.KINDS:
            r.block_graphs[kind].replay()
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    ta, tp, to, rc = orc.verify_tree(ti.target, BF16, ti.parents, ti.tokens)
    assert rc == 0
    po, rc = orc.probs(ci.target.reshape(-1, ci.V), BF16, 1.0)
    assert rc == 0
    used = sorted({j % bench.ROT for j in range(bench.BLOCK)})
    for k in used:
        c = r.copies[k]
        compare_chain(orc, ci, (c["acc"].cpu().numpy(), c["out"].cpu().numpy(), 0))
        np.testing.assert_array_equal(c["tacc"].cpu().numpy(), ta)
        np.testing.assert_array_equal(c["tpath"].cpu().numpy(), tp)
        np.testing.assert_array_equal(c["tout"].cpu().numpy(), to)
        pr = c["probs"].cpu().numpy().reshape(-1, ci.V).astype(np.float64)
        assert np.abs(pr - po).max() <= 2e-6

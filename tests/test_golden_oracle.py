"""The oracle against the hand-derived fixtures in tests/golden/ (exact expected outputs
worked out from the method's definition; see the "about" and "why" fields there)."""

import numpy as np
import pytest

from golden_io import chain_cases, margin_cases, tree_cases
from workloads import F32


@pytest.mark.parametrize("case", chain_cases(), ids=lambda c: c["name"])
def test_chain_golden(orc, case):
    acc, out, mg, rc = orc.verify_chain(case["target"], case["draft"], F32, case["tokens"],
                                        case["uniforms"], case["T"])
    assert rc == 0
    np.testing.assert_array_equal(acc, case["accept_len"])
    np.testing.assert_array_equal(out, case["out_tokens"])


@pytest.mark.parametrize("case", tree_cases(), ids=lambda c: c["name"])
def test_tree_golden(orc, case):
    acc, path, out, rc = orc.verify_tree(case["target"], F32, case["parents"], case["tokens"])
    assert rc == 0
    np.testing.assert_array_equal(acc, case["accept_len"])
    np.testing.assert_array_equal(path, case["path_nodes"])
    np.testing.assert_array_equal(out, case["out_tokens"])


@pytest.mark.parametrize("case", margin_cases(), ids=lambda c: c["name"])
def test_margin_golden(orc, case):
    """Pins the margins and bands of the oracle's per-position detail, and the row margin of
    oracle_verify_chain (the minimum over the draws on its path), to the hand-derived values:
    decision margins relative to the ratio, CDF margins relative to P (not S), bands by the
    cumulative-sum rule."""
    d = orc.verify_chain_detail(case["target"], case["draft"], F32, case["tokens"],
                                case["uniforms"], case["T"], band=case["band"])
    assert d["rc"] == 0
    np.testing.assert_array_equal(d["accept"], case["accept"])
    np.testing.assert_array_equal(d["tok"], case["tok"])
    np.testing.assert_array_equal(d["lo"], case["lo"])
    np.testing.assert_array_equal(d["hi"], case["hi"])
    np.testing.assert_allclose(d["dmargin"], case["dmargin"], rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(d["cmargin"], case["cmargin"], rtol=1e-9, atol=1e-15)
    acc, out, mg, rc = orc.verify_chain(case["target"], case["draft"], F32, case["tokens"],
                                        case["uniforms"], case["T"])
    assert rc == 0
    np.testing.assert_array_equal(acc, case["accept_len"])
    np.testing.assert_array_equal(out, case["out_tokens"])
    for b in range(len(acc)):
        n = int(acc[b])
        on_path = list(case["dmargin"][b, :min(n + 1, case["gamma"])]) + [case["cmargin"][b, n]]
        assert mg[b] == pytest.approx(min(on_path), rel=1e-9, abs=1e-15)

"""The oracle against the hand-derived fixtures in tests/golden/ (exact expected outputs
worked out from the method's definition; see the "about" and "why" fields there)."""

import numpy as np
import pytest

from golden_io import chain_cases, tree_cases
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

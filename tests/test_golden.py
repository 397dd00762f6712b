"""Regression of the oracle against the fixtures written by tests/golden/make_golden.py."""
import json
import os

import numpy as np
import pytest

from tests.golden import make_golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name", sorted(make_golden.CASES))
def test_oracle_matches_golden(name):
    with open(os.path.join(HERE, f"{name}.json")) as f:
        want = json.load(f)
    got = make_golden.summarise(*make_golden.run_case(make_golden.CASES[name]))
    assert got["shape"] == want["shape"]
    assert got["ctx_k_bits_sum"] == want["ctx_k_bits_sum"]
    np.testing.assert_allclose(got["sum"], want["sum"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got["abs_sum"], want["abs_sum"], rtol=1e-12)
    for k, v in want["rows"].items():
        np.testing.assert_allclose(got["rows"][k], v, rtol=1e-12, atol=1e-14)

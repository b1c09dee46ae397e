"""The oracle still reproduces the stored fixtures (written by tests/golden/make_golden.py)."""
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.join(os.path.dirname(__file__), "golden"))
import make_golden  # noqa: E402

import oracle  # noqa: E402
import workloads as wl  # noqa: E402


@pytest.mark.parametrize("name", [f[0] for f in make_golden.FIXTURES])
def test_oracle_matches_fixture(name):
    meta, want = make_golden.read(name)
    x, W, b = wl.make_inputs(meta["M"], meta["N"], meta["K"], meta["seed"], bool(meta["bias"]))
    got = oracle.linear_bf16(wl.bits(x), wl.bits(W), wl.bits(b))
    assert np.array_equal(got, want)

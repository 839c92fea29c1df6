"""The oracle still reproduces its stored output on the pages' own small
test scenarios ("cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs", test
o1_batch_matches_serial_steps; fixtures written by tests/golden/make_golden.py
from the oracle alone)."""
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


@pytest.mark.parametrize("idx", [0, 1])
def test_oracle_matches_golden(idx):
    outs = make_golden.run_case(idx)
    rows = np.loadtxt(os.path.join(HERE, "golden", f"page_case_{idx}.txt"), comments="#")
    got = np.concatenate([o.reshape(-1, o.shape[-1]) for o in outs])
    assert rows.shape[0] == got.shape[0]
    np.testing.assert_allclose(got, rows[:, 3:], rtol=1e-13, atol=1e-15)
    assert np.isfinite(got).all()

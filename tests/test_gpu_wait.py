"""The bounded in-kernel waits running out, on purpose, through the C ABI.

o1_set_wait_limit makes the kernels' first waits give up after a few hundred
clock cycles (long before a copy or a tensor-core tile lands). The kernel
must then raise O1_FLAG_WAIT_EXPIRED, still wait (with the full limit) for
the work it had issued, release what it holds and return, leaving the
context usable: after the flag is cleared and the default limit restored,
the next calls match the oracle again.
  - The tensor-core window kernel stops issuing on expiry: that call's
    output is not valid, only the flag and the return are checked.
  - The one-row path's blocks wait once more for their copies and carry on,
    so its output stays valid whether or not a wait ran out (its copies are
    small and may land before the first look): it is compared with the
    oracle under the tiny limit, and the state after it too.
"""
import numpy as np
import pytest

from sliding_window_landmark_gb300 import synth

import harness

pytestmark = pytest.mark.gpu

TINY_LIMIT = 300   # cycles: far below a TMA round trip


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_landmark_gb300 import build
    build.build()


def test_window_kernel_wait_runs_out_and_recovers():
    from sliding_window_landmark_gb300 import o1
    sh = synth.Shape(groups=1, heads_per_group=2, d=64, dv=64, sinks=4, window=512, landmarks=4)
    c = synth.layer_constants(sh, 41)
    q, k, v, g = synth.layer_rows(sh, 41, 0, 300)
    gpu = harness.GpuLayer(sh, c, max_rows=300)
    try:
        o1.o1_set_wait_limit(TINY_LIMIT)
        gpu.rows(q, k, v, g)   # 300 rows: the tensor-core window path
    finally:
        o1.o1_set_wait_limit(0)
    flags = o1.o1_state_flags(gpu.state, gpu.g, clear=True)
    assert flags & o1.O1_FLAG_WAIT_EXPIRED, flags
    assert o1.o1_state_flags(gpu.state, gpu.g) == 0
    # the context is usable and the default limit is back: a fresh layer is green
    orc = harness.oracle_layer(sh, c)
    want, diag = orc.rows(q, k, v, g, diag=True)
    fresh = harness.GpuLayer(sh, c, max_rows=300)
    harness.assert_outputs(fresh.rows(q, k, v, g), want, diag, "after expiry")
    harness.assert_state(fresh.read(), orc, "after expiry")
    assert o1.o1_state_flags(fresh.state, fresh.g) == 0


def test_token_wait_runs_out_and_output_stays_valid():
    from sliding_window_landmark_gb300 import o1
    sh = synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=2, window=64, landmarks=8)
    c = synth.layer_constants(sh, 42)
    q, k, v, g = synth.layer_rows(sh, 42, 0, 104)
    orc = harness.oracle_layer(sh, c)
    gpu = harness.GpuLayer(sh, c, max_rows=100)
    want, diag = orc.rows(q[:100], k[:100], v[:100], g[:100], diag=True)
    harness.assert_outputs(gpu.rows(q[:100], k[:100], v[:100], g[:100]), want, diag, "prompt")
    want, diag = orc.rows(q[100:], k[100:], v[100:], g[100:], diag=True)
    try:
        o1.o1_set_wait_limit(TINY_LIMIT)
        got = gpu.tokens(q[100:], k[100:], v[100:], g[100:])
    finally:
        o1.o1_set_wait_limit(0)
    flags = o1.o1_state_flags(gpu.state, gpu.g, clear=True)
    assert flags & ~o1.O1_FLAG_WAIT_EXPIRED == 0, flags
    print("one-row steps under the tiny limit: a wait ran out" if flags else
          "one-row steps under the tiny limit: every copy landed before the first look")
    harness.assert_outputs(got, want, diag, "one-row steps under a tiny wait limit")
    harness.assert_state(gpu.read(), orc, "after the steps")

"""The allocation-free one-row entry point (o1_token_attend_noalloc) against
the ordinary one (o1_token_attend), through the C ABI.

o1_token_attend_noalloc serves callers that cannot allocate device memory
(a plugin interface that hands over no workspace, or a decode loop that may
not call cudaMalloc); its scratch is a static device array inside the
library. Two layers start from the same 300-row prompt; each then takes two
decode steps in a row, one layer through each entry point. Both steps'
outputs, and the whole state after them (meta, position, ring, far max,
mass and value sums), must match the serial oracle within the parity
tolerance, and the two entry points must agree with each other. The second
call also shows that what the first call left in the shared array does not
leak into the next."""
import numpy as np
import pytest

from sliding_window_landmark_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-4, 1e-4


def test_noalloc_token_matches_token_attend():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_landmark_gb300 import build
    build.build()
    from sliding_window_landmark_gb300 import o1

    import harness

    sh = synth.Shape(groups=2, heads_per_group=4, d=256, dv=256, sinks=4, window=256, landmarks=32)
    c = synth.layer_constants(sh, 31)
    prompt = 300
    q, k, v, gt = synth.layer_rows(sh, 31, 0, prompt + 2)
    orc = harness.oracle_layer(sh, c)
    orc.rows(q[:prompt], k[:prompt], v[:prompt], gt[:prompt], threads=2)
    ref, noalloc = (harness.GpuLayer(sh, c, max_rows=prompt) for _ in range(2))
    assert 0 < o1.o1_scratch_bytes(ref.g, 1) <= o1.O1_NOALLOC_SCRATCH_BYTES
    for lay in (ref, noalloc):
        lay.rows(q[:prompt], k[:prompt], v[:prompt], gt[:prompt])
    dev = torch.device("cuda")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    for step in range(2):
        r = prompt + step
        want, diag = orc.rows(q[r:r + 1], k[r:r + 1], v[r:r + 1], gt[r:r + 1], diag=True)
        a = ref.tokens(q[r:r + 1], k[r:r + 1], v[r:r + 1], gt[r:r + 1])
        got = torch.full((sh.nh, sh.dv), float("nan"), device=dev)
        o1.check(o1.o1_token_attend_noalloc(noalloc.state, noalloc.g, up(q[r]), up(k[r]), up(v[r]), up(gt[r]),
                                            got))
        torch.cuda.synchronize()
        b = got.cpu().numpy()[None]
        assert np.isfinite(b).all()
        harness.assert_outputs(b, want, diag, f"no-alloc step {step} against the oracle")
        harness.assert_outputs(a, want, diag, f"step {step} against the oracle")
        diff = np.abs(a.astype(np.float64) - b)
        assert (diff <= ATOL + RTOL * np.abs(a)).all(), f"step {step}: max diff {diff.max()}"
    harness.assert_state(noalloc.read(), orc, "no-alloc state after two steps")
    harness.assert_state(ref.read(), orc, "state after two steps")
    ra, rb = ref.read(), noalloc.read()
    np.testing.assert_array_equal(ra["meta"], rb["meta"])
    assert int(ra["pos"][0]) == int(rb["pos"][0]) == prompt + 2


def test_noalloc_rejects_geometry_beyond_its_scratch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_landmark_gb300 import build
    build.build()
    from sliding_window_landmark_gb300 import o1
    g = o1.geom(64, 16, 256, 256, 4, 1024, 64)  # one-row scratch well above 4 MiB
    assert o1.o1_scratch_bytes(g, 1) > o1.O1_NOALLOC_SCRATCH_BYTES
    V = o1._VP
    assert o1.LIB.o1_token_attend_noalloc(V(1 << 20), o1.ctypes.byref(g), V(1 << 21), V(1 << 21), V(1 << 21),
                                          None, V(1 << 22), None) == o1.O1_ERR_UNSUPPORTED

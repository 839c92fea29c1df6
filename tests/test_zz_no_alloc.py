"""The allocation-free one-row entry point (o1_token_attend_noalloc) against
the ordinary one (o1_token_attend), through the C ABI.

o1_token_attend_noalloc serves callers that cannot allocate device memory
(a plugin interface that hands over no workspace, or a decode loop that may
not call cudaMalloc); its scratch is a static device array inside the
library. Two layers start from the same state; each then takes two decode
steps in a row, one layer through each entry point, and the outputs must
agree within the parity tolerance. The second call also shows that what
the first call left in the shared array does not leak into the next."""
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

    sh = synth.Shape(groups=2, heads_per_group=4, d=256, dv=256, sinks=4, window=256, landmarks=32)
    g = o1.geom(sh.groups, sh.heads_per_group, sh.d, sh.dv, sh.sinks, sh.window, sh.landmarks)
    assert 0 < o1.o1_scratch_bytes(g, 1) <= o1.O1_NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda")
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    c = synth.layer_constants(sh, 31)
    consts = [up(c.sink_k), up(c.sink_v), up(c.k_tilde), up(c.q_tilde), up(c.mu)]
    prompt = 300
    q, k, v, gt = (up(x) for x in synth.layer_rows(sh, 31, 0, prompt + 2))
    states = []
    for _ in range(2):
        st = torch.empty(o1.o1_state_bytes(g), dtype=torch.uint8, device=dev)
        o1.check(o1.o1_state_init(st, g, None, *consts, 0))
        scratch = torch.empty(o1.o1_scratch_bytes(g, prompt), dtype=torch.uint8, device=dev)
        pout = torch.empty((prompt, sh.nh, sh.dv), device=dev)
        o1.check(o1.o1_chunk_attend(st, g, scratch, q[:prompt], k[:prompt], v[:prompt], gt[:prompt], prompt, pout))
        states.append(st)
    scratch = torch.empty(o1.o1_scratch_bytes(g, 1), dtype=torch.uint8, device=dev)
    for step in range(2):
        r = prompt + step
        ref = torch.empty((sh.nh, sh.dv), device=dev)
        got = torch.full((sh.nh, sh.dv), float("nan"), device=dev)
        o1.check(o1.o1_token_attend(states[0], g, scratch, q[r], k[r], v[r], gt[r], ref))
        o1.check(o1.o1_token_attend_noalloc(states[1], g, q[r], k[r], v[r], gt[r], got))
        torch.cuda.synchronize()
        a, b = ref.cpu().numpy().astype(np.float64), got.cpu().numpy().astype(np.float64)
        assert np.isfinite(b).all()
        assert (np.abs(a - b) <= ATOL + RTOL * np.abs(a)).all(), f"step {step}: max diff {np.abs(a - b).max()}"
    ra, rb = o1.empty_state_arrays(g), o1.empty_state_arrays(g)
    o1.check(o1.o1_state_read(states[0], g, ra))
    o1.check(o1.o1_state_read(states[1], g, rb))
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

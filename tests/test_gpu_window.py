"""The exact-attention comparator (o1_window_attend) against exact softmax
attention written out in numpy, in double: textbook half-split rotation
with the f32-rounded table, scores over the sinks and each row's window,
softmax, value sum, sigmoid gate. Each row attends to the last
min(window, position + 1) keys ending at its own, and nothing reaches a far
field. From a fresh state with a window of at least the rows, this is full
causal attention (the no-eviction pin); with a shorter window the dropped
keys are simply gone. The state must come out unchanged.
"""
import numpy as np
import pytest

from sliding_window_landmark_gb300 import synth

import harness
import test_oracle_pins as pins

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_landmark_gb300 import build
    build.build()


def _exact(shape, consts, q, k, v, gate, first, scale):
    """Rows first .. first + R - 1 of a stream whose keys are k[0 .. first + R - 1]
    (all of them, from position 0): sinks + the last min(wg, t + 1) keys."""
    R = q.shape[0] - first
    G, hpg = shape.groups, shape.heads_per_group
    wins = shape.group_windows or (shape.window,) * G
    kr = np.stack([pins._rot(k[t], t, shape.rope_base) for t in range(k.shape[0])])   # [T][G][d]
    out = np.empty((R, shape.nh, shape.dv))
    for r in range(R):
        t = first + r
        for gi in range(G):
            lo = max(0, t + 1 - wins[gi])
            keys = kr[lo:t + 1, gi]
            vals = v[lo:t + 1, gi].astype(np.float64)
            if shape.sinks:
                keys = np.concatenate([consts.sink_k[gi].astype(np.float64), keys])
                vals = np.concatenate([consts.sink_v[gi].astype(np.float64), vals])
            qr = np.stack([pins._rot(q[t, gi * hpg + h], t, shape.rope_base) for h in range(hpg)])
            s = scale * qr @ keys.T
            p = np.exp(s - s.max(axis=1, keepdims=True))
            o = (p @ vals) / p.sum(axis=1, keepdims=True)
            out[r, gi * hpg:(gi + 1) * hpg] = o * pins._sigmoid(gate[t, gi * hpg:(gi + 1) * hpg])
    return out


# (shape, rows already pushed by o1_chunk_attend, rows attended)
WINDOW_CASES = [
    # fp32 window kernel: full causal from a fresh state, sinks
    (synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=4, window=256, landmarks=4), 0, 200),
    # sliding: window shorter than the rows, no sinks (the pages' exact path)
    (synth.Shape(groups=1, heads_per_group=4, d=32, dv=32, sinks=0, window=48, landmarks=2), 0, 150),
    # after a prompt: the ring's keys, then this call's rows
    (synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=2, window=96, landmarks=4,
                 group_windows=(96, 40)), 130, 70),
    # tensor-core window kernel: full causal, then sliding after a prompt
    (synth.Shape(groups=1, heads_per_group=2, d=64, dv=64, sinks=0, window=768, landmarks=4), 0, 700),
    (synth.Shape(groups=2, heads_per_group=2, d=128, dv=64, sinks=3, window=512, landmarks=4), 600, 300),
    # a short pass (rows x heads per group <= 64: the key-slice window path),
    # on a tensor-core geometry and on an fp32 one
    (synth.Shape(groups=2, heads_per_group=4, d=64, dv=64, sinks=2, window=512, landmarks=4), 700, 12),
    (synth.Shape(groups=1, heads_per_group=2, d=32, dv=32, sinks=4, window=40, landmarks=2), 90, 5),
]


@pytest.mark.parametrize("case", range(len(WINDOW_CASES)))
def test_window_attend_is_exact_attention(case):
    import torch
    from sliding_window_landmark_gb300 import o1
    shape, pre, rows = WINDOW_CASES[case]
    seed = 80 + case
    c = synth.layer_constants(shape, seed)
    gpu = harness.GpuLayer(shape, c, max_rows=max(rows, pre, 1))
    q, k, v, g = synth.layer_rows(shape, seed, 0, pre + rows)
    if pre:
        gpu.rows(q[:pre], k[:pre], v[:pre], g[:pre])
    before = gpu.state.clone()
    out = torch.empty((rows, shape.nh, shape.dv), dtype=torch.float32, device=gpu.dev)
    o1.check(o1.o1_window_attend(gpu.state, gpu.g, gpu.scratch, gpu.up(q[pre:]), gpu.up(k[pre:]), gpu.up(v[pre:]),
                                 gpu.up(g[pre:]), rows, out), "window")
    torch.cuda.synchronize()
    want = _exact(shape, c, q, k, v, g, pre, float(gpu.g.scale))
    harness.assert_outputs(out.cpu().numpy(), want, None, "exact attention")
    assert torch.equal(gpu.state, before), "the comparator changed the state"

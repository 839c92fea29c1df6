"""Speculative verification against the oracle ("cortiq-engine 0.8.82
src/gpu_metal/o1c.rs": encode with commit = false, then spec_commit over the
accepted rows).

A draft attended by o1_chunk_attend_spec gives the outputs the oracle gives
for those rows after the committed history, and leaves every byte of the
state as it was. o1_spec_commit over the first n accepted rows leaves the
state the oracle has after exactly those rows, and the calls after it keep
matching. The expected values come from two oracle runs: one over the
committed history (advanced by the accepted rows only), and one replaying
that history and then the whole draft.

The meta rewind of looped-layer KV modes (o1_state_back; "cortiq-engine
0.8.77 src/gpu_wgpu/dory.rs", dory_o1_back) is checked the same way against
the oracle's rewind, including a refused rewind.
"""
import numpy as np
import pytest

from sliding_window_landmark_gb300 import synth

import harness

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_landmark_gb300 import build
    build.build()


# (shape, prompt rows, [(draft rows, accepted rows)], scratch rows)
SPEC_CASES = [
    # fp32 window: drafts longer than a 64-row block and than the window
    # (keys pushed and evicted within the draft), a one-row draft, none and
    # all accepted
    (synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=4, window=48, landmarks=8), 100,
     [(8, 5), (1, 1), (70, 0), (12, 12), (70, 70), (3, 2)], 128),
    # tensor-core window (window >= 512), the ring already evicting
    (synth.Shape(groups=1, heads_per_group=2, d=64, dv=64, sinks=2, window=512, landmarks=4), 600,
     [(8, 3), (1, 1), (130, 77), (64, 0)], 256),
    # before the ring fills: no far field yet, then the first evictions
    # inside a committed draft
    (synth.Shape(groups=1, heads_per_group=4, d=32, dv=32, sinks=0, window=64, landmarks=4), 40,
     [(30, 30), (20, 11)], 64),
    # group windows narrower than a short commit: the commit evicts its own
    # rows, whose keys the far insert rotates where it reads them
    (synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=2, window=12, landmarks=4, group_windows=(6, 12)), 30,
     [(16, 14), (10, 9), (4, 1)], 32),
]


@pytest.mark.parametrize("case", range(len(SPEC_CASES)))
def test_spec_verify_then_commit(case):
    import torch
    from sliding_window_landmark_gb300 import o1
    shape, prompt, drafts, scratch_rows = SPEC_CASES[case]
    seed = 40 + case
    c = synth.layer_constants(shape, seed)
    committed = harness.oracle_layer(shape, c)
    gpu = harness.GpuLayer(shape, c, max_rows=scratch_rows)
    q, k, v, g = synth.layer_rows(shape, seed, 0, prompt)
    history = [(q, k, v, g)]
    want, diag = committed.rows(q, k, v, g, diag=True)
    harness.assert_outputs(gpu.rows(q, k, v, g), want, diag, "prompt")
    r0 = prompt
    for i, (n_draft, n_acc) in enumerate(drafts):
        q, k, v, g = synth.layer_rows(shape, seed, r0, n_draft)
        r0 += n_draft
        # expected draft outputs: the committed history, then the whole draft
        replay = harness.oracle_layer(shape, c)
        replay.rows(*[np.concatenate([h[j] for h in history]) for j in range(4)])
        want, diag = replay.rows(q, k, v, g, diag=True)

        before = gpu.state.clone()
        qd, kd, vd, gd = gpu.up(q), gpu.up(k), gpu.up(v), gpu.up(g)
        out = torch.empty((n_draft, shape.nh, shape.dv), dtype=torch.float32, device=gpu.dev)
        o1.check(o1.o1_chunk_attend_spec(gpu.state, gpu.g, gpu.scratch, qd, kd, vd, gd, n_draft, out), "spec")
        torch.cuda.synchronize()
        harness.assert_outputs(out.cpu().numpy(), want, diag, f"draft {i}")
        assert torch.equal(gpu.state, before), f"draft {i}: an attend-only call changed the state"

        o1.check(o1.o1_spec_commit(gpu.state, gpu.g, gpu.scratch, kd[:n_acc].contiguous(),
                                   vd[:n_acc].contiguous(), n_acc), "commit")
        torch.cuda.synchronize()
        if n_acc:
            committed.rows(q[:n_acc], k[:n_acc], v[:n_acc], g[:n_acc])
            history.append((q[:n_acc], k[:n_acc], v[:n_acc], g[:n_acc]))
        else:
            assert torch.equal(gpu.state, before), f"draft {i}: committing no rows changed the state"
        harness.assert_state(gpu.read(), committed, f"after committing {n_acc} of draft {i}")
    # ordinary calls continue from the committed state
    q, k, v, g = synth.layer_rows(shape, seed, r0, 50)
    want, diag = committed.rows(q, k, v, g, diag=True)
    harness.assert_outputs(gpu.rows(q, k, v, g), want, diag, "after the drafts")
    harness.assert_state(gpu.read(), committed, "end")


def test_spec_commit_in_several_passes():
    """A commit longer than the scratch's capacity runs as several passes and
    still lands on the oracle's state."""
    import torch
    from sliding_window_landmark_gb300 import o1
    shape = synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=4, window=96, landmarks=8)
    c = synth.layer_constants(shape, 77)
    orc = harness.oracle_layer(shape, c)
    gpu = harness.GpuLayer(shape, c, max_rows=64)
    q, k, v, g = synth.layer_rows(shape, 77, 0, 300)
    orc.rows(q, k, v, g)
    o1.check(o1.o1_spec_commit(gpu.state, gpu.g, gpu.scratch, gpu.up(k), gpu.up(v), 300), "commit")
    torch.cuda.synchronize()
    harness.assert_state(gpu.read(), orc, "after a 300-row commit through 64-row scratch")


def test_spec_draft_above_capacity_is_refused():
    import torch
    from sliding_window_landmark_gb300 import o1
    shape = synth.Shape(groups=1, heads_per_group=2, d=64, dv=64, sinks=4, window=48, landmarks=4)
    c = synth.layer_constants(shape, 5)
    gpu = harness.GpuLayer(shape, c, max_rows=64)
    q, k, v, g = synth.layer_rows(shape, 5, 0, 4096)
    out = torch.empty((4096, shape.nh, shape.dv), dtype=torch.float32, device=gpu.dev)
    before = gpu.state.clone()
    st = o1.o1_chunk_attend_spec(gpu.state, gpu.g, gpu.scratch, gpu.up(q), gpu.up(k), gpu.up(v), gpu.up(g), 4096,
                                 out)
    assert st == o1.O1_ERR_ARG
    torch.cuda.synchronize()
    assert torch.equal(gpu.state, before)


# (shape, prompt rows, chunk rows, rewind rows)
BACK_CASES = [
    # ring not yet full: the rewind drops the newest entries
    (synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=4, window=256, landmarks=8), 60, 40, 40),
    # full ring with evictions: head and eviction count step back
    (synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=4, window=48, landmarks=8), 150, 70, 30),
    # tensor-core window, group windows of different widths
    (synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=2, window=512, landmarks=4,
                 group_windows=(512, 384)), 700, 130, 100),
]


@pytest.mark.parametrize("case", range(len(BACK_CASES)))
def test_state_back_then_repush(case):
    """o1_state_back against the oracle's rewind (dory.rs dory_o1_back): the
    state after the rewind, then the outputs and state of the rows pushed
    over it, match; a rewind longer than a group can take is refused on the
    device with nothing changed."""
    import torch
    from sliding_window_landmark_gb300 import o1
    shape, prompt, n, back = BACK_CASES[case]
    seed = 60 + case
    c = synth.layer_constants(shape, seed)
    orc = harness.oracle_layer(shape, c)
    gpu = harness.GpuLayer(shape, c, max_rows=max(prompt, n))
    q, k, v, g = synth.layer_rows(shape, seed, 0, prompt + n)
    for a, b in ((0, prompt), (prompt, prompt + n)):
        want, diag = orc.rows(q[a:b], k[a:b], v[a:b], g[a:b], diag=True)
        harness.assert_outputs(gpu.rows(q[a:b], k[a:b], v[a:b], g[a:b]), want, diag, f"rows {a}..{b}")
    assert orc.back(back)
    o1.check(o1.o1_state_back(gpu.state, gpu.g, back), "back")
    torch.cuda.synchronize()
    assert o1.o1_state_flags(gpu.state, gpu.g) == 0
    harness.assert_state(gpu.read(), orc, "after the rewind")
    # other rows pushed over the rewound positions
    q2, k2, v2, g2 = synth.layer_rows(shape, seed + 100, 0, back + 20)
    want, diag = orc.rows(q2, k2, v2, g2, diag=True)
    harness.assert_outputs(gpu.rows(q2, k2, v2, g2), want, diag, "rows after the rewind")
    harness.assert_state(gpu.read(), orc, "after pushing again")
    # refused: more than the position allows
    before = gpu.state.clone()
    too_many = int(orc.pos[0]) + 1
    assert not orc.back(too_many)
    o1.check(o1.o1_state_back(gpu.state, gpu.g, too_many), "back")
    torch.cuda.synchronize()
    assert o1.o1_state_flags(gpu.state, gpu.g, clear=True) == o1.O1_FLAG_BACK_REFUSED
    assert torch.equal(gpu.state, before)


# (shape, prompt rows, rows committed one at a time, rewind + re-commit pairs)
ONE_ROW_CASES = [
    # the ring fills during the one-row commits, then every commit evicts
    (synth.Shape(groups=2, heads_per_group=2, d=64, dv=64, sinks=4, window=24, landmarks=8), 10, 30, 6),
    # the stack's landmark count and widths (m = 64, d = dv = 128), ring evicting
    (synth.Shape(groups=2, heads_per_group=4, d=128, dv=128, sinks=4, window=64, landmarks=64), 80, 12, 6),
]


@pytest.mark.parametrize("case", range(len(ONE_ROW_CASES)))
def test_one_row_commits_and_rewinds(case):
    """o1_spec_commit of one row at a time (the one-row kernel's commit mode:
    the far chunks insert the evicted key, the last CTA pushes the row) lands
    on the oracle's state, across the ring filling and evicting; then one-row
    rewinds each followed by a one-row commit of another row, as a looped
    layer runs them; then attention over that state matches the oracle."""
    import torch
    from sliding_window_landmark_gb300 import o1
    shape, prompt, n, pairs = ONE_ROW_CASES[case]
    seed = 90 + case
    c = synth.layer_constants(shape, seed)
    orc = harness.oracle_layer(shape, c)
    gpu = harness.GpuLayer(shape, c, max_rows=max(prompt, 16))
    q, k, v, g = synth.layer_rows(shape, seed, 0, prompt + n + pairs + 16)
    want, diag = orc.rows(q[:prompt], k[:prompt], v[:prompt], g[:prompt], diag=True)
    harness.assert_outputs(gpu.rows(q[:prompt], k[:prompt], v[:prompt], g[:prompt]), want, diag, "prompt")
    kd, vd = gpu.up(k), gpu.up(v)
    for i in range(prompt, prompt + n):
        orc.rows(q[i:i + 1], k[i:i + 1], v[i:i + 1], g[i:i + 1])   # the oracle's push (its output unused)
        o1.check(o1.o1_spec_commit(gpu.state, gpu.g, gpu.scratch, kd[i:i + 1], vd[i:i + 1], 1), "commit")
    torch.cuda.synchronize()
    assert o1.o1_state_flags(gpu.state, gpu.g) == 0
    harness.assert_state(gpu.read(), orc, f"after {n} one-row commits")
    for j in range(prompt + n, prompt + n + pairs):
        assert orc.back(1)
        o1.check(o1.o1_state_back(gpu.state, gpu.g, 1), "back")
        orc.rows(q[j:j + 1], k[j:j + 1], v[j:j + 1], g[j:j + 1])
        o1.check(o1.o1_spec_commit(gpu.state, gpu.g, gpu.scratch, kd[j:j + 1], vd[j:j + 1], 1), "commit")
    torch.cuda.synchronize()
    assert o1.o1_state_flags(gpu.state, gpu.g) == 0
    harness.assert_state(gpu.read(), orc, f"after {pairs} rewind + one-row commit pairs")
    a = prompt + n + pairs
    want, diag = orc.rows(q[a:a + 16], k[a:a + 16], v[a:a + 16], g[a:a + 16], diag=True)
    harness.assert_outputs(gpu.tokens(q[a:a + 16], k[a:a + 16], v[a:a + 16], g[a:a + 16]), want, diag,
                           "one-row steps after the commits")
    harness.assert_state(gpu.read(), orc, "end")

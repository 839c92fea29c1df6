"""CUDA path against the oracle, element by element, on the same seeded
inputs, through the C ABI.

Cases: the tiny workload (G=1, hpg=2, d=dv=64, 4 sinks, w=16, m=4; ring full
before the measured chunk, so every row evicts), the pages' own test
scenarios, small shapes that span several blocks with a ragged tail (group
windows, rectified mass, shorter windows than a block, many passes, no
sinks, one landmark), chunk == row-by-row, and the full single-layer
workloads (4096-row prompt; 8192-row prompt + 1024 decode steps; 32768-row
prompt with group windows 1024 / 2048).
"""
import numpy as np
import pytest

from sliding_window_landmark_gb300 import synth

import harness
import scenarios

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sliding_window_landmark_gb300 import build
    build.build()


def _run(shape, seed, calls, rect=False, mu_abs=False, consts=None, token=False, gate=True,
         scratch_rows=None, check_state=True):
    """calls: row counts of consecutive calls. Returns per-call stats."""
    c = consts or synth.layer_constants(shape, seed, mu_abs=mu_abs)
    orc = harness.oracle_layer(shape, c, rect=rect)
    gpu = harness.GpuLayer(shape, c, rect=rect, max_rows=max(calls), scratch_rows=scratch_rows)
    r0, stats = 0, []
    for n in calls:
        q, k, v, g = synth.layer_rows(shape, seed, r0, n, gate=gate)
        want, diag = orc.rows(q, k, v, g, threads=shape.groups, diag=True)
        got = gpu.tokens(q, k, v, g) if token else gpu.rows(q, k, v, g)
        stats.append(harness.assert_outputs(got, want, diag, what=f"rows {r0}..{r0 + n}"))
        if check_state:
            harness.assert_state(gpu.read(), orc, what=f"after rows {r0 + n}")
        r0 += n
    return stats


@pytest.mark.parametrize("rope_base", [1e6, 0.0])
@pytest.mark.parametrize("warm", [16, 48])
def test_tiny_workload(rope_base, warm):
    sh = synth.Shape(**{**synth.TINY.__dict__, "rope_base": rope_base})
    st = _run(sh, 0, [warm, 64])
    assert st[1]["have_frac"] > 0.2


def test_tiny_workload_is_deterministic():
    sh = synth.TINY
    c = synth.layer_constants(sh, 0)
    res = []
    for _ in range(2):
        gpu = harness.GpuLayer(sh, c, max_rows=64)
        q, k, v, g = synth.layer_rows(sh, 0, 0, 80)
        o = np.concatenate([gpu.rows(q[:16], k[:16], v[:16], g[:16]), gpu.rows(q[16:], k[16:], v[16:], g[16:])])
        res.append((o, gpu.read()))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    for key in res[0][1]:
        np.testing.assert_array_equal(res[0][1][key], res[1][1][key])


@pytest.mark.parametrize("case", scenarios.PAGE_CASES, ids=[str(c[:7]) for c in scenarios.PAGE_CASES])
def test_page_scenarios(case):
    shape, c, prompt, chunks = scenarios.page_case(*case)
    orc = harness.oracle_layer(shape, c)
    gpu = harness.GpuLayer(shape, c, max_rows=max(case[5], max(case[7])))
    want, diag = orc.rows(*prompt, threads=2, diag=True)
    harness.assert_outputs(gpu.rows(*prompt), want, diag, "prompt")
    harness.assert_state(gpu.read(), orc, "after prompt")
    for i, ch in enumerate(chunks):
        want, diag = orc.rows(*ch, threads=2, diag=True)
        got = gpu.tokens(*ch) if ch[0].shape[0] == 1 else gpu.rows(*ch)
        harness.assert_outputs(got, want, diag, f"chunk {i}")
        harness.assert_state(gpu.read(), orc, f"after chunk {i}")


SMALL = [
    # (G, hpg, d, dv, ns, w, group windows, m, calls, rect, mu_abs, rope, scratch rows)
    (2, 2, 32, 24, 2, 40, (17, 40), 5, (150, 70, 1, 3), False, False, 1e6, None),
    (2, 6, 16, 16, 3, 64, (64, 30), 8, (200, 64, 65), False, True, 1e4, None),
    (1, 16, 8, 4, 1, 9, None, 3, (130,), False, False, 1e6, None),
    (3, 1, 64, 128, 0, 20, (5, 20, 1), 2, (90, 7), True, False, 1e6, None),
    (2, 4, 128, 128, 4, 100, None, 64, (300,), False, False, 1e6, 64),
    (1, 3, 24, 20, 5, 50, None, 1, (77, 77), False, True, 0.0, 33),
    (2, 2, 256, 256, 2, 70, (70, 66), 16, (140,), False, False, 1e6, None),
]


@pytest.mark.parametrize("case", SMALL, ids=[f"small{i}" for i in range(len(SMALL))])
def test_small_shapes(case):
    G, hpg, d, dv, ns, w, gw, m, calls, rect, mu_abs, rope, srows = case
    sh = synth.Shape(groups=G, heads_per_group=hpg, d=d, dv=dv, sinks=ns, window=w, landmarks=m,
                     rope_base=rope, group_windows=gw)
    _run(sh, 100 + d, list(calls), rect=rect, mu_abs=mu_abs, scratch_rows=srows)


# The tensor-core window path (d % 64 == 0, dv % 32 == 0, window >= 512):
# every d chunk count (1, 2, 4), dv from 32 to 256, ragged 128-row tiles,
# tile starts not on a 64-key boundary, one-row passes between chunks, a
# group window shorter than the ring stride, rectified mass, no sinks.
TC = [
    # (G, hpg, d, dv, ns, w, group windows, m, calls, rect, mu_abs, rope)
    (2, 2, 128, 128, 4, 512, (512, 130), 16, (1500, 77), False, False, 1e6),
    (1, 4, 64, 64, 0, 600, None, 8, (130, 900, 1), False, True, 1e6),
    (2, 3, 256, 256, 2, 520, (520, 515), 32, (700,), True, False, 1e4),
    (1, 1, 64, 32, 1, 512, None, 4, (1, 63, 600), False, False, 0.0),
    (1, 2, 192, 96, 3, 700, None, 8, (333, 1000), False, False, 1e6),
]


@pytest.mark.parametrize("case", TC, ids=[f"tc{i}" for i in range(len(TC))])
def test_tensor_core_window_shapes(case):
    G, hpg, d, dv, ns, w, gw, m, calls, rect, mu_abs, rope = case
    sh = synth.Shape(groups=G, heads_per_group=hpg, d=d, dv=dv, sinks=ns, window=w, landmarks=m,
                     rope_base=rope, group_windows=gw)
    st = _run(sh, 300 + d, list(calls), rect=rect, mu_abs=mu_abs)
    print("tensor-core window:", st)


def test_tensor_core_flags():
    """The tensor-core path leaves the state's flags clear on ordinary inputs
    and raises O1_FLAG_FP16_RANGE for a value outside the fp16 range."""
    from sliding_window_landmark_gb300 import o1
    sh = synth.Shape(groups=1, heads_per_group=2, d=64, dv=64, sinks=1, window=512, landmarks=4)
    c = synth.layer_constants(sh, 5)
    gpu = harness.GpuLayer(sh, c, max_rows=256)
    q, k, v, g = synth.layer_rows(sh, 5, 0, 256)
    gpu.rows(q, k, v, g)
    assert o1.o1_state_flags(gpu.state, gpu.g) == 0
    v = v.copy()
    v[100, 0, 3] = 1e5
    gpu.rows(q, k, v, g)
    assert o1.o1_state_flags(gpu.state, gpu.g, clear=True) == o1.O1_FLAG_FP16_RANGE
    assert o1.o1_state_flags(gpu.state, gpu.g) == 0


def test_no_gate_and_empty_call():
    sh = synth.Shape(groups=2, heads_per_group=2, d=16, dv=8, sinks=1, window=10, landmarks=3)
    c = synth.layer_constants(sh, 7)
    gpu = harness.GpuLayer(sh, c, max_rows=50)
    orc = harness.oracle_layer(sh, c)
    import torch
    from sliding_window_landmark_gb300 import o1
    empty = torch.empty(0, device="cuda")
    assert o1.LIB.o1_chunk_attend(o1._VP(gpu.state.data_ptr()), o1.ctypes.byref(gpu.g),
                                  o1._VP(gpu.scratch.data_ptr()), gpu.scratch.numel(), None, None, None, None, 0,
                                  None, None) == o1.O1_OK
    del empty
    q, k, v, _ = synth.layer_rows(sh, 7, 0, 50, gate=False)
    want, diag = orc.rows(q, k, v, None, diag=True)
    harness.assert_outputs(gpu.rows(q, k, v, None), want, diag)
    harness.assert_state(gpu.read(), orc)


def test_chunk_equals_row_by_row():
    """One call over the rows equals the rows one call at a time (the far
    terms referenced to a later max only rescale numerator and denominator
    together), and both equal the oracle."""
    sh = synth.Shape(groups=2, heads_per_group=4, d=64, dv=64, sinks=4, window=48, landmarks=8,
                     group_windows=(48, 20))
    c = synth.layer_constants(sh, 12)
    q, k, v, g = synth.layer_rows(sh, 12, 0, 200)
    a = harness.GpuLayer(sh, c, max_rows=200)
    b = harness.GpuLayer(sh, c, max_rows=200)
    orc = harness.oracle_layer(sh, c)
    want, diag = orc.rows(q, k, v, g, diag=True)
    ca = a.rows(q, k, v, g)
    cb = b.tokens(q, k, v, g)
    harness.assert_outputs(ca, want, diag, "chunk")
    harness.assert_outputs(cb, want, diag, "rows")
    skip = harness.flip_rows(diag)[..., None]
    diff = np.abs(ca.astype(np.float64) - cb)
    i = np.unravel_index(np.argmax(np.where(skip, 0, diff)), diff.shape)
    print("chunk vs rows: max diff", diff[i], "at", i, "oracle", want[i], "chunk", ca[i], "rows", cb[i])
    assert ((diff <= harness.ATOL + harness.RTOL * np.abs(want)) | skip).all()
    sa, sb = a.read(), b.read()
    np.testing.assert_array_equal(sa["meta"], sb["meta"])
    np.testing.assert_array_equal(sa["ring_v"], sb["ring_v"])


# ---------------------------------------------------------- full workloads

def test_qwen_layer_prompt_4096():
    st = _run(synth.QWEN_LAYER, 1, [4096])
    print("4096-row prompt:", st)


def test_qwen_layer_decode_after_8192():
    sh = synth.QWEN_LAYER
    c = synth.layer_constants(sh, 2)
    orc = harness.oracle_layer(sh, c)
    gpu = harness.GpuLayer(sh, c, max_rows=8192)
    q, k, v, g = synth.layer_rows(sh, 2, 0, 8192)
    orc.rows(q, k, v, g, threads=2)
    gpu.rows(q, k, v, g)
    q, k, v, g = synth.layer_rows(sh, 2, 8192, 1024)
    want, diag = orc.rows(q, k, v, g, threads=2, diag=True)
    st = harness.assert_outputs(gpu.tokens(q, k, v, g), want, diag, "decode")
    harness.assert_state(gpu.read(), orc, "after decode")
    print("decode:", st)


def test_qwen_long_prompt_group_windows():
    st = _run(synth.QWEN_LONG, 3, [32768], check_state=True)
    print("32768-row prompt:", st)


def test_qwen_long_prompt_nonnegative_mu():
    """mu >= 0: the far mass cannot cancel (every term is non-negative), so
    no row is flip-adjacent and every row gets the strict tolerance."""
    st = _run(synth.QWEN_LONG, 4, [32768], mu_abs=True)
    assert st[0]["flip_rows"] == 0
    print("32768-row prompt, mu >= 0:", st)


@pytest.mark.parametrize("layer", [0, 23])
def test_stack_layer_prompt(layer):
    """A layer of the 24-layer stack (4 KV groups x 4 heads, d = dv = 128,
    window 1024, 64 landmarks): the 65536-row prompt of its own seed."""
    sh = synth.STACK_LAYER
    seed = 1000 + layer
    c = synth.layer_constants(sh, seed)
    orc = harness.oracle_layer(sh, c)
    gpu = harness.GpuLayer(sh, c, max_rows=16384)
    stats = []
    for r0 in range(0, 65536, 16384):
        q, k, v, g = synth.layer_rows(sh, seed, r0, 16384)
        want, diag = orc.rows(q, k, v, g, threads=sh.groups, diag=True)
        stats.append(harness.assert_outputs(gpu.rows(q, k, v, g), want, diag, f"layer {layer} rows {r0}"))
    harness.assert_state(gpu.read(), orc, f"layer {layer}")
    print(f"stack layer {layer}:", stats)


@pytest.mark.parametrize("layer", [0, 11, 23])
def test_stack_layer_decode(layer):
    """Decode at the stack shape (4 KV groups x 4 heads, d = dv = 128, window
    1024, 64 landmarks per head, the most the library takes): an 1100-row
    prompt through o1_chunk_attend (the ring full and past it), then 256
    one-row steps through o1_token_attend, each evicting a key; every output
    and the final state against the oracle, on the layer's own seed."""
    sh = synth.STACK_LAYER
    seed = 1000 + layer
    c = synth.layer_constants(sh, seed)
    orc = harness.oracle_layer(sh, c)
    gpu = harness.GpuLayer(sh, c, max_rows=1100)
    q, k, v, g = synth.layer_rows(sh, seed, 0, 1100)
    want, diag = orc.rows(q, k, v, g, threads=sh.groups, diag=True)
    harness.assert_outputs(gpu.rows(q, k, v, g), want, diag, f"layer {layer} prompt")
    q, k, v, g = synth.layer_rows(sh, seed, 1100, 256)
    want, diag = orc.rows(q, k, v, g, threads=sh.groups, diag=True)
    st = harness.assert_outputs(gpu.tokens(q, k, v, g), want, diag, f"layer {layer} decode")
    harness.assert_state(gpu.read(), orc, f"layer {layer} after decode")
    print(f"stack layer {layer} decode:", st)


def test_decode_widest_far_block():
    """The one-row far block's shared-memory layout grows as m d + m^2 and is
    largest at d = dv = 256 with 64 landmarks: a prompt past the window, then
    one-row steps, against the oracle."""
    sh = synth.Shape(groups=1, heads_per_group=2, d=256, dv=256, sinks=4, window=64, landmarks=64)
    st = _run(sh, 77, [100, 1, 1, 1, 1, 1, 1, 1, 1], token=True)
    print("widest far block:", st[-1])


def test_timed_stages_and_stream_capture():
    """The timed variant records a begin/end pair per stage (on the stage's
    own stream); a CUDA-graph capture of o1_chunk_attend (whose far-field
    branch runs on the library's second stream) replays to the oracle's
    result."""
    import torch
    from sliding_window_landmark_gb300 import o1
    sh = synth.Shape(groups=1, heads_per_group=2, d=64, dv=64, sinks=2, window=512, landmarks=4)
    c = synth.layer_constants(sh, 9)
    q, k, v, g = synth.layer_rows(sh, 9, 0, 300)
    want, diag = harness.oracle_layer(sh, c).rows(q, k, v, g, diag=True)

    gpu = harness.GpuLayer(sh, c, max_rows=300)
    names = [o1.o1_stage_name(i) for i in range(o1.O1_NUM_STAGES)]
    assert names == ["rope", "far_block", "far_tscan", "side_readout", "gather_tc", "near", "merge", "commit"]
    assert o1.o1_stage_name(o1.O1_NUM_STAGES) is None
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * o1.O1_NUM_STAGES)]
    for e in evs:
        e.record()
    out = torch.empty((300, sh.nh, sh.dv), dtype=torch.float32, device="cuda")
    dq, dk, dvv, dg = gpu.up(q), gpu.up(k), gpu.up(v), gpu.up(g)
    o1.check(o1.o1_chunk_attend_timed(gpu.state, gpu.g, gpu.scratch, dq, dk, dvv, dg, 300, out, evs), "timed")
    torch.cuda.synchronize()
    times = [evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(o1.O1_NUM_STAGES)]
    assert all(np.isfinite(t) and t >= 0 for t in times), times
    harness.assert_outputs(out.cpu().numpy(), want, diag, "timed")
    assert o1.o1_status_string(o1.LIB.o1_chunk_attend_timed(
        o1._VP(gpu.state.data_ptr()), o1.ctypes.byref(gpu.g), o1._VP(gpu.scratch.data_ptr()), gpu.scratch.numel(),
        o1._VP(dq.data_ptr()), o1._VP(dk.data_ptr()), o1._VP(dvv.data_ptr()), None, 300, o1._VP(out.data_ptr()),
        (o1._VP * 3)(), 3, None)) == o1.o1_status_string(o1.O1_ERR_ARG)

    cap = harness.GpuLayer(sh, c, max_rows=300)
    out2 = torch.empty((300, sh.nh, sh.dv), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            o1.check(o1.o1_chunk_attend(cap.state, cap.g, cap.scratch, dq, dk, dvv, dg, 300, out2), "capture")
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    harness.assert_outputs(out2.cpu().numpy(), want, diag, "graph replay")
    orc = harness.oracle_layer(sh, c)
    orc.rows(q, k, v, g)
    harness.assert_state(cap.read(), orc, "graph replay state")


# passes of at most 16 rows take the short far kernel (k_side_short):
# (shape, calls) with short calls after a prompt that fills the ring, so
# that every short row evicts, and one set before it fills
SHORT_CASES = [
    (synth.Shape(groups=2, heads_per_group=4, d=256, dv=256, sinks=4, window=64, landmarks=32), [100, 2, 16, 5, 9, 1, 3]),
    (synth.Shape(groups=2, heads_per_group=4, d=128, dv=128, sinks=4, window=48, landmarks=64), [60, 16, 7, 2, 11]),
    (synth.Shape(groups=1, heads_per_group=2, d=64, dv=64, sinks=0, window=40, landmarks=8), [5, 16, 12, 9, 2]),
]


@pytest.mark.parametrize("case", range(len(SHORT_CASES)))
def test_short_passes(case):
    """Short passes (the far field and sinks row by row in one CTA a head)
    against the oracle: outputs of every call and the state after each."""
    shape, calls = SHORT_CASES[case]
    _run(shape, 120 + case, calls)

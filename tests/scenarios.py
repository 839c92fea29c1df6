"""The pages' own batch-vs-serial test scenarios, replayed.

"cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs", test
o1_batch_matches_serial_steps, and "cortiq-engine 0.8.82 src/gpu_metal/o1c.rs",
test o1c_matches_serial_steps: geometries (d, m, w, sink, hpg, t, w2, chunks),
two KV groups (the second with its own window w2), a prompt of t rows first,
then chunks that continue from the committed state. Data is the pages'
integer pattern jit(a, b) with their per-tensor streams: b = 1, 2, 3 + h
(+20 per group) for the prompt's k, v, q and 5, 6, 7 for the chunks' q, k, v.
The pages build their landmarks with a seal step that is not on them; here
the sinks and landmarks come from further jit streams (b = 8..12, +20 per
group), and the t prompt rows are pushed through the layer from a fresh state.
"""
import numpy as np

from sliding_window_landmark_gb300 import synth

# (d, m, w, sink, hpg, t, w2, chunks)
PAGE_CASES = [
    (8, 4, 64, 2, 2, 100, 64, (70, 9)),
    (8, 4, 64, 2, 2, 100, 128, (70, 40)),
    (256, 32, 128, 4, 6, 300, 512, (64, 64)),
    (256, 32, 128, 4, 6, 300, 128, (5, 1)),
]


def page_case(d, m, w, sink, hpg, t, w2, chunks):
    """Shape, constants and the row stream of one scenario.

    Returns (shape, consts, prompt, chunk_rows): prompt = (q, k, v) of the t
    rows, chunk_rows = list of (q, k, v) per chunk. No gate (the pages' batch
    kernels leave it to a later stage)."""
    G = 2
    nh = G * hpg
    W = max(w, w2)
    shape = synth.Shape(groups=G, heads_per_group=hpg, d=d, dv=d, sinks=sink, window=W, landmarks=m,
                        rope_base=0.0, group_windows=(w, w2))
    J = synth.jit
    sink_k = np.stack([J(np.arange(sink * d), 8 + 20 * g).reshape(sink, d) for g in range(G)])
    sink_v = np.stack([J(np.arange(sink * d), 9 + 20 * g).reshape(sink, d) for g in range(G)])
    kt = np.stack([J(np.arange(m * d), 10 + 20 * g).reshape(m, d) for g in range(G)])
    qt = np.stack([J(np.arange(hpg * m * d), 11 + 20 * g).reshape(hpg, m, d) for g in range(G)])
    mu = np.stack([J(np.arange(hpg * m * m), 12 + 20 * g).reshape(hpg, m, m) for g in range(G)]).reshape(nh, m, m)
    consts = synth.LayerInputs(shape, sink_k, sink_v, kt, qt, mu)
    pk = np.stack([J(np.arange(t * d), 1 + 20 * g).reshape(t, d) for g in range(G)], axis=1)
    pv = np.stack([J(np.arange(t * d), 2 + 20 * g).reshape(t, d) for g in range(G)], axis=1)
    pq = np.stack([np.stack([J(np.arange(t * d), 3 + h + 20 * g).reshape(t, d) for h in range(hpg)], 1)
                   for g in range(G)], axis=1).reshape(t, nh, d)
    chunk_rows = []
    base = 0
    for rows in chunks:
        q = J(np.arange(rows * nh * d) + base * nh * d, 5).reshape(rows, nh, d)
        k = J(np.arange(rows * G * d) + base * G * d, 6).reshape(rows, G, d)
        v = J(np.arange(rows * G * d) + base * G * d, 7).reshape(rows, G, d)
        chunk_rows.append((q, k, v))
        base += rows
    return shape, consts, (pq, pk, pv), chunk_rows

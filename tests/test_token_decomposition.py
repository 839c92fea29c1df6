"""The one-row (decode) path's decomposition, restated in numpy (fp64) and
checked against the serial oracle on the CPU.

The decode kernel does not attend in one sequence. The near set after the
push (sinks, then the ring in logical order, with the pushed slot served
from the row's own key and value) is cut into slices of KC keys, each with
a slice-local softmax (max, mass, value sum); the merge takes every slice
against the largest slice max. The far part is cut into chunks of MB
landmark queries: each applies the evicted key's insert to its (M, Z, T)
and forms its share of the readout under its own exponent (the largest
F + M'_b of the chunk): far mass and numerator; the merge moves the chunks
to their largest exponent and sums them before the sign decision. The two
parts meet under one exponent with the 1e-30 floor, and then the gate. This
test takes one step that way from a snapshot of the oracle's state and
compares it with the oracle's own next row, to fp64 rounding.
"""
import numpy as np
import pytest

from sliding_window_landmark_gb300 import synth

import test_oracle_pins as pins


def _token_step(shape, c, snap, q, k, v, gate, scale, KC, MB):
    G, hpg, m, ns = shape.groups, shape.heads_per_group, shape.landmarks, shape.sinks
    p = snap["pos"]
    out = np.zeros((shape.nh, shape.dv))
    kt = c.k_tilde.astype(np.float64).reshape(G, m, -1)
    qt = c.q_tilde.astype(np.float64).reshape(G, hpg, m, -1)
    mu = c.mu.astype(np.float64).reshape(shape.nh, m, m)
    for gi in range(G):
        ln, head, farl, wg = (int(x) for x in snap["meta"][gi])
        kr = pins._rot(k[gi], p, shape.rope_base)
        evict = ln == wg
        k_e, v_e = snap["ring_k"][gi, head], snap["ring_v"][gi, head]
        len1 = wg if evict else ln + 1
        head1 = (head + 1) % wg if evict else head
        # the near set after the push: sinks, then the ring in logical order;
        # the last logical slot is the row's own key and value
        keys = [c.sink_k[gi].astype(np.float64)] if ns else []
        vals = [c.sink_v[gi].astype(np.float64)] if ns else []
        slots = [(head1 + i) % wg for i in range(len1)]
        rk, rv = snap["ring_k"][gi][slots].copy(), snap["ring_v"][gi][slots].copy()
        rk[-1], rv[-1] = kr, v[gi].astype(np.float64)
        keys, vals = np.concatenate(keys + [rk]), np.concatenate(vals + [rv])
        for hl in range(hpg):
            h = gi * hpg + hl
            qv = pins._rot(q[h], p, shape.rope_base)
            # slices: (max, mass, value sum) each, merged against the largest max
            parts = []
            for i0 in range(0, len(keys), KC):
                s = scale * keys[i0:i0 + KC] @ qv
                ms = s.max()
                e = np.exp(s - ms)
                parts.append((ms, e.sum(), e @ vals[i0:i0 + KC]))
            Mw = max(pt[0] for pt in parts)
            Lw = sum(pt[1] * np.exp(pt[0] - Mw) for pt in parts)
            Aw = sum(pt[2] * np.exp(pt[0] - Mw) for pt in parts)
            # the far part: insert of the evicted key, then the readout
            cf, Df, have, num = -np.inf, 0.0, False, 0.0
            if farl + (1 if evict else 0) > 0:
                Mo, Zo, To = snap["M"][h], snap["Z"][h], snap["T"][h]
                if evict:
                    l = scale * qt[gi, hl] @ k_e
                    Mn = np.maximum(Mo, l)
                    with np.errstate(invalid="ignore"):
                        rho = np.where(Mn == Mo, 1.0, np.exp(Mo - Mn))
                    ee = np.exp(l - Mn)
                    Zn, Tn = Zo * rho + ee, To * rho[:, None] + ee[:, None] * v_e[None, :]
                else:
                    Mn, Zn, Tn = Mo, Zo, To
                f = scale * kt[gi] @ qv
                F = f.max()
                u = np.exp(f - F) @ mu[h]
                cb = F + Mn
                # chunks of MB landmark queries, each under its own exponent
                recs = []
                for b0 in range(0, m, MB):
                    sl = slice(b0, b0 + MB)
                    cl = cb[sl].max()
                    gl = u[sl] * np.exp(cb[sl] - cl)
                    recs.append((cl, gl @ Zn[sl], gl @ Tn[sl]))
                cf = max(r[0] for r in recs)
                Df = sum(r[1] * np.exp(r[0] - cf) for r in recs)
                have = Df >= 0
                num = sum(r[2] * np.exp(r[0] - cf) for r in recs)
            cc = max(Mw, cf)
            al = np.exp(Mw - cc)
            be = np.exp(cf - cc) if have else 0.0
            den = max(be * Df + al * Lw, 1e-30)
            out[h] = (be * num + al * Aw) / den * pins._sigmoid(gate[h])
    return out


@pytest.mark.parametrize("case", [
    # (G, hpg, d, dv, ns, window, m, prompt rows, KC, MB, rope base, seed)
    (2, 2, 16, 8, 3, 24, 4, 60, 8, 4, 1e6, 1),    # full ring: each step evicts; one far chunk
    (2, 2, 16, 8, 3, 24, 7, 60, 8, 3, 1e6, 4),    # far chunks of 3, 3 and 1 landmarks
    (1, 3, 8, 4, 2, 40, 3, 17, 8, 1, 1e4, 2),     # ring still filling: no eviction, no far field yet
    (1, 2, 8, 6, 0, 12, 2, 12, 16, 1, 0.0, 3),    # the first eviction, no sinks, one slice
])
def test_token_decomposition_equals_serial(case):
    G, hpg, d, dv, ns, w, m, prompt, KC, MB, base, seed = case
    sh = synth.Shape(groups=G, heads_per_group=hpg, d=d, dv=dv, sinks=ns, window=w, landmarks=m, rope_base=base)
    lay, c, g = pins._layer(sh, seed)
    q, k, v, gt = synth.layer_rows(sh, seed, 0, prompt + 3)
    lay.rows(q[:prompt], k[:prompt], v[:prompt], gt[:prompt])
    for t in range(prompt, prompt + 3):
        snap = lay.snapshot()
        got = _token_step(sh, c, snap, q[t], k[t], v[t], gt[t], g.scale_f32(), KC, MB)
        want = lay.rows(q[t:t + 1], k[t:t + 1], v[t:t + 1], gt[t:t + 1])[0]
        np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-11)

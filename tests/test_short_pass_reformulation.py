"""A short pass (at most 16 rows), taken in the order the short far kernel
takes it, restated in numpy (fp64) and checked against the serial oracle on
the CPU.

The pages interleave, row after row, the insert of the key a row evicts and
that row's readout. The short far kernel does not. It computes every dot
product of the pass first: the insert logits of the keys the rows evict,
and the far and sink scores of the rows' queries. Then only the recurrence
of M and Z (per landmark: M' = max(M, l), rho, e, Z = rho Z + e) runs row
after row, keeping each row's M and Z. Every row's readout scalars come
from that row's snapshot, independently of the other rows: c_f, the
gains, D and its sign, c_s = max(sink max, c_f), the sink weights and the
side mass. Last, T runs row after row (T = rho T + e v_e) for the side
numerators. The window part is exact per row. The two parts merge under
one exponent with the 1e-30 floor, then the gate. From a snapshot of the
oracle's state, the pass must equal the oracle's next rows to fp64
rounding and leave the same far field. This pins the design, not the
kernel: the kernel is compared with the oracle on the GPU. No CUDA code,
and nothing of the oracle but its public results, is used here.
"""
import numpy as np
import pytest

from sliding_window_landmark_gb300 import synth

import test_oracle_pins as pins


def _short_pass(shape, c, snap, q, k, v, gate, scale, rect):
    G, hpg, m, ns, dv = shape.groups, shape.heads_per_group, shape.landmarks, shape.sinks, shape.dv
    R = q.shape[0]
    p0 = snap["pos"]
    kt = c.k_tilde.astype(np.float64).reshape(G, m, -1)
    qt = c.q_tilde.astype(np.float64).reshape(G, hpg, m, -1)
    mu = c.mu.astype(np.float64).reshape(shape.nh, m, m)
    out = np.zeros((R, shape.nh, dv))
    M1, Z1, T1 = snap["M"].copy(), snap["Z"].copy(), snap["T"].copy()
    for gi in range(G):
        ln, head, farl, wg = (int(x) for x in snap["meta"][gi])
        j0 = wg - ln   # row r evicts X[r - j0] once r >= j0
        # X: the ring in logical order, then this pass's rotated keys
        slots = [(head + i) % wg for i in range(ln)]
        Xk = np.concatenate([snap["ring_k"][gi][slots].reshape(ln, -1),
                             np.stack([pins._rot(k[r, gi], p0 + r, shape.rope_base) for r in range(R)])])
        Xv = np.concatenate([snap["ring_v"][gi][slots].reshape(ln, -1), v[:, gi].astype(np.float64)])
        sk = c.sink_k[gi].astype(np.float64).reshape(ns, shape.d)
        sv = c.sink_v[gi].astype(np.float64).reshape(ns, dv)
        for hl in range(hpg):
            h = gi * hpg + hl
            qv = np.stack([pins._rot(q[r, h], p0 + r, shape.rope_base) for r in range(R)])   # [R][d]
            # 1. every dot product of the pass
            ev = [r for r in range(R) if r >= j0]
            L = {r: scale * qt[gi, hl] @ Xk[r - j0] for r in ev}
            f = scale * qv @ kt[gi].T                                   # [R][m]
            s = scale * qv @ sk.T if ns else np.zeros((R, 0))          # [R][ns]
            # 2. the recurrence of M and Z, each row's M and Z kept
            M, Z = snap["M"][h].copy(), snap["Z"][h].copy()
            rho, e, Ms, Zs = {}, {}, [], []
            for r in range(R):
                if r in L:
                    Mn = np.maximum(M, L[r])
                    with np.errstate(invalid="ignore"):
                        rho[r] = np.where(Mn == M, 1.0, np.exp(M - Mn))
                    e[r] = np.exp(L[r] - Mn)
                    Z = Z * rho[r] + e[r]
                    M = Mn
                Ms.append(M.copy())
                Zs.append(Z.copy())
            F = f.max(axis=1)
            u = np.exp(f - F[:, None]) @ mu[h]
            if rect:
                u = np.maximum(u, 0.0)
            # 3. every row's readout scalars, from its own snapshot
            gains, fs, side, cs = [None] * R, np.zeros(R), np.zeros(R), np.full(R, -np.inf)
            wts = np.zeros((R, ns))
            for r in range(R):
                cf, D, have = -np.inf, 0.0, False
                if farl + max(0, r - j0 + 1) > 0:
                    cb = F[r] + Ms[r]
                    cf = cb.max()
                    gains[r] = u[r] * np.exp(cb - cf)
                    D = gains[r] @ Zs[r]
                    have = D >= 0
                smax = s[r].max() if ns else -np.inf
                cs[r] = max(smax, cf)
                fs[r] = np.exp(cf - cs[r]) if have else 0.0
                wts[r] = np.exp(s[r] - cs[r]) if ns else wts[r]
                side[r] = (fs[r] * D if have else 0.0) + wts[r].sum()
            # 4. T row after row, and the side numerators
            T = snap["T"][h].copy()
            for r in range(R):
                if r in e:
                    T = rho[r][:, None] * T + e[r][:, None] * Xv[r - j0][None, :]
                num = (fs[r] * (gains[r] @ T) if fs[r] != 0.0 else np.zeros(dv)) + (wts[r] @ sv if ns else 0.0)
                # the window part, exact: X[max(0, ln + r + 1 - wg) .. ln + r]
                lo = max(0, ln + r + 1 - wg)
                sw = scale * Xk[lo:ln + r + 1] @ qv[r]
                Mw = sw.max()
                ew = np.exp(sw - Mw)
                cc = max(Mw, cs[r])
                al = np.exp(Mw - cc)
                be = np.exp(cs[r] - cc) if cs[r] > -np.inf else 0.0
                den = max(al * ew.sum() + be * side[r], 1e-30)
                out[r, h] = (al * (ew @ Xv[lo:ln + r + 1]) + be * num) / den * pins._sigmoid(gate[r, h])
            M1[h], Z1[h], T1[h] = M, Z, T
    return out, M1, Z1, T1


@pytest.mark.parametrize("case", [
    # (G, hpg, d, dv, ns, window, group windows, m, prompt rows, pass rows, rope base, rect, seed)
    (2, 2, 16, 8, 3, 24, None, 4, 60, 8, 1e6, False, 1),       # full ring: every row evicts
    (1, 3, 8, 4, 2, 40, None, 5, 30, 16, 1e4, False, 2),       # the ring fills within the pass: j0 = 10
    (1, 2, 8, 6, 0, 12, None, 3, 5, 9, 0.0, False, 3),         # no far field yet, then the first evictions; no sinks
    (2, 2, 16, 8, 2, 12, (5, 12), 4, 30, 14, 1e6, False, 4),   # group windows narrower than the pass: it evicts its own rows
    (1, 2, 16, 8, 4, 20, None, 6, 50, 6, 1e6, True, 5),        # rectified far mass
])
def test_short_pass_equals_serial(case):
    G, hpg, d, dv, ns, w, gw, m, prompt, R, base, rect, seed = case
    sh = synth.Shape(groups=G, heads_per_group=hpg, d=d, dv=dv, sinks=ns, window=w, landmarks=m, rope_base=base,
                     group_windows=gw)
    lay, c, g = pins._layer(sh, seed, rect=rect)
    q, k, v, gt = synth.layer_rows(sh, seed, 0, prompt + 2 * R)
    lay.rows(q[:prompt], k[:prompt], v[:prompt], gt[:prompt])
    for t in (prompt, prompt + R):   # two passes in a row
        snap = lay.snapshot()
        sl = slice(t, t + R)
        got, M1, Z1, T1 = _short_pass(sh, c, snap, q[sl].reshape(R, sh.nh, d), k[sl].reshape(R, G, d),
                                      v[sl].reshape(R, G, dv), gt[sl].reshape(R, sh.nh, dv), g.scale_f32(), rect)
        want = lay.rows(q[sl], k[sl], v[sl], gt[sl])
        np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-11)
        after = lay.snapshot()
        np.testing.assert_allclose(M1, after["M"], rtol=1e-12, atol=0)
        np.testing.assert_allclose(Z1, after["Z"], rtol=1e-9, atol=1e-300)
        np.testing.assert_allclose(T1, after["T"], rtol=1e-9, atol=1e-11)

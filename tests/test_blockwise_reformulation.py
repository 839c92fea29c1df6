"""The chunk pass's reformulation, restated in numpy (fp64) and checked
against the serial oracle on the CPU.

The CUDA chunk pass does not run the pages' serial per-row far insert. It
computes, per 64-row block c of the pass, partials relative to the block's
own max, composes them across blocks by a scan, and reads each row's far
part against the running max M_c after its block. This test writes that
algebra out step by step:
- block partials: logits of the keys the block's rows evict, local max m_c,
  E = e^{l - m_c}, in-block prefix, mass s_c, value-sum increment dT_c;
- the scan: M_c, R_c = e^{M_{c-1} - M_c}, f_c = e^{m_c - M_c}, Z, and the
  value sum entering each block, R_c T_{c-1};
- per row: the landmark readout with gains against M_c, the far mass
  R_c Z_{c-1} + f_c * prefix, the numerator from the entering sum plus the
  in-block coefficients, the sinks, the exact window;
- the merge under one exponent and the gate.

It also checks that the result equals the pages' row-by-row algorithm
(the oracle) to fp64 rounding. This pins the design, not the kernels: the
kernels are compared with the oracle on the GPU. No CUDA code, and nothing
of the oracle but its public results, is used here.
"""
import numpy as np
import pytest

from sliding_window_landmark_gb300 import synth

import test_oracle_pins as pins

BLOCK = 64


def _blockwise(shape, c, q, k, v, gate, scale, rect=False):
    G, hpg, nh, m, ns, w = shape.groups, shape.heads_per_group, shape.nh, shape.landmarks, shape.sinks, shape.window
    R = q.shape[0]
    qr = np.stack([[pins._rot(q[r, h], r, shape.rope_base) for h in range(nh)] for r in range(R)])   # [R][nh][d]
    kr = np.stack([pins._rot(k[r], r, shape.rope_base) for r in range(R)])                             # [R][G][d]
    vv = v.astype(np.float64)
    kt = c.k_tilde.astype(np.float64).reshape(G, m, -1)
    qt = c.q_tilde.astype(np.float64).reshape(G, hpg, m, -1)
    mu = c.mu.astype(np.float64).reshape(nh, m, m)
    out = np.zeros((R, nh, shape.dv))
    nblk = (R + BLOCK - 1) // BLOCK
    j0 = w   # fresh state: row r evicts key X[r - w] once r >= w
    for gi in range(G):
        sk, sv = c.sink_k[gi].astype(np.float64), c.sink_v[gi].astype(np.float64)
        for hl in range(hpg):
            h = gi * hpg + hl
            # block partials
            lmax, lsum = np.full((nblk, m), -np.inf), np.zeros((nblk, m))
            E, P = np.zeros((m, R)), np.zeros((m, R))
            dT = np.zeros((nblk, m, shape.dv))
            for cb in range(nblk):
                rows = np.arange(cb * BLOCK, min(R, cb * BLOCK + BLOCK))
                ev = rows[rows >= j0]
                if len(ev) == 0:
                    continue
                keys, vals = kr[ev - j0, gi], vv[ev - j0, gi]
                l = scale * qt[gi, hl] @ keys.T                        # [m][ev]
                lmax[cb] = l.max(axis=1)
                e = np.exp(l - lmax[cb][:, None])
                E[:, ev], P[:, ev] = e, np.cumsum(e, axis=1)
                lsum[cb] = e.sum(axis=1)
                dT[cb] = e @ vals
            # the scan across blocks
            Mp, Zp, Tp_ = np.full(m, -np.inf), np.zeros(m), np.zeros((m, shape.dv))
            Mc, Rc, Fc, Bc, Tin = [], [], [], [], []
            for cb in range(nblk):
                Mn = np.maximum(Mp, lmax[cb])
                with np.errstate(invalid="ignore"):   # -inf - -inf in the branch np.where discards
                    Rf = np.where(Mn == Mp, 1.0, np.exp(Mp - Mn))
                    f = np.where(np.isneginf(lmax[cb]), 0.0, np.exp(lmax[cb] - Mn))
                Mc.append(Mn), Rc.append(Rf), Fc.append(f), Bc.append(Rf * Zp), Tin.append(Rf[:, None] * Tp_)
                Zp = Rf * Zp + f * lsum[cb]
                Tp_ = Rf[:, None] * Tp_ + f[:, None] * dT[cb]
                Mp = Mn
            # per row: the side part (sinks + far field) and the exact window
            for r in range(R):
                cb = r // BLOCK
                qv = qr[r, h]
                lo = max(0, r + 1 - w)
                s_win = scale * kr[lo:r + 1, gi] @ qv
                s_snk = scale * sk @ qv if ns else np.zeros(0)
                cw = s_win.max()
                farl = max(0, r - j0 + 1)
                cf, have, D, num_far = -np.inf, False, 0.0, 0.0
                if farl > 0:
                    f_a = scale * kt[gi] @ qv
                    F = f_a.max()
                    u = np.exp(f_a - F) @ mu[h]
                    if rect:
                        u = np.maximum(u, 0.0)
                    cb_ = F + Mc[cb]
                    cf = cb_.max()
                    gain = u * np.exp(cb_ - cf)
                    Pr = Bc[cb] + Fc[cb] * P[:, r]
                    D = gain @ Pr
                    have = D >= 0
                    rows = np.arange(cb * BLOCK, r + 1)
                    rows = rows[rows >= j0]
                    coef = (gain * Fc[cb]) @ E[:, rows]                   # in-block coefficients
                    num_far = gain @ Tin[cb] + coef @ vv[rows - j0, gi]
                cs = max(s_snk.max() if ns else -np.inf, cf)
                ws = np.exp(s_snk - cs) if ns else np.zeros(0)
                fs = np.exp(cf - cs) if have else 0.0
                side_num = (ws @ sv if ns else 0.0) + fs * num_far
                side_mass = ws.sum() + fs * D
                # merge under one exponent
                cc = max(cw, cs)
                pw = np.exp(s_win - cw)
                al, be = np.exp(cw - cc), np.exp(cs - cc) if cs > -np.inf else 0.0
                num = al * (pw @ vv[lo:r + 1, gi]) + be * side_num
                den = max(al * pw.sum() + be * side_mass, 1e-30)
                out[r, h] = num / den * pins._sigmoid(gate[r, h])
    return out


@pytest.mark.parametrize("case", [
    # (G, hpg, d, dv, ns, window, m, rows, rope base, rect, seed)
    (1, 2, 8, 4, 2, 5, 3, 150, 1e4, False, 1),      # tiny window: many evictions per block, ragged tail
    (2, 2, 16, 8, 3, 70, 4, 200, 1e6, False, 2),    # first evictions in the middle of block 1
    (1, 3, 8, 6, 0, 64, 2, 130, 0.0, False, 3),     # no sinks, evictions start at a block boundary
    (1, 2, 8, 4, 1, 9, 3, 140, 1e6, True, 4),       # rectified far mass
])
def test_blockwise_chunk_equals_serial(case):
    G, hpg, d, dv, ns, w, m, rows, base, rect, seed = case
    sh = synth.Shape(groups=G, heads_per_group=hpg, d=d, dv=dv, sinks=ns, window=w, landmarks=m, rope_base=base)
    lay, c, g = pins._layer(sh, seed, rect=rect)
    q, k, v, gt = synth.layer_rows(sh, seed, 0, rows)
    want = lay.rows(q, k, v, gt)
    got = _blockwise(sh, c, q, k, v, gt, g.scale_f32(), rect=rect)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-11)

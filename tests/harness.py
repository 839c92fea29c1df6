"""Runs one layer through the CUDA library (C ABI, via the binding) and
through the oracle on the same seeded inputs, and compares them.

Tolerance (per element): |gpu - oracle| <= 2e-4 + 1e-4 |oracle|, fp32 against
the double-precision oracle, on every row-head but the flip-adjacent ones.
Meta, position and ring values are compared bit-exactly; rotated ring keys
within 1e-5 relative (the rotation table is formed differently on each
side).

Flip-adjacent rows. A row's far part enters through its far mass
D = sum_b gain_b Z_b, whose terms carry signed gains and can cancel; the far
part is kept when D >= 0 and dropped otherwise, and the denominator holds D.
An fp32 path knows the far terms to a relative error EPS_FAR: rotated keys
and queries, landmark scores, the products u = e^{f - F} mu and the far
numerator are fp32 (the far mass itself is accumulated and summed in
double). It knows D to about EPS_FAR * A, A = sum_b |gain_b Z_b|: where
|D| <= FLIP_MARGIN * A the sign decision can differ from the oracle's, and
when it agrees the output, whose size grows as A / D, moves by about
EPS_FAR * (A / D) * (|o| + |v|). Measured on the 32768- and 65536-row
prompts: rows just past |D| = 1e-3 A reached 2.3 times the tolerance, an
effective EPS_FAR of about 3.5e-7, and the error fell as D / A rose. So rows
with |D| <= FLIP_MARGIN A = 4e-3 A in the oracle are counted and reported,
not compared: there the result is decided by digits at fp32's resolution
(about 1 % of the row-heads of a long prompt with signed mu, none with
mu >= 0). Every other row is held to the tolerance above.
"""
from __future__ import annotations

import numpy as np

import oracle
from sliding_window_landmark_gb300 import synth

ATOL, RTOL = 2e-4, 1e-4
EPS_FAR = 3.5e-7
FLIP_MARGIN = 4e-3


def oracle_layer(shape: synth.Shape, consts, rect=False, scale=None, pos0=0):
    g = oracle.Geom(shape.groups, shape.heads_per_group, shape.d, shape.dv, shape.sinks, shape.window,
                    shape.landmarks, scale=scale, rope_base=shape.rope_base, rect_far_mass=rect)
    return oracle.OracleLayer(g, consts.sink_k, consts.sink_v, consts.k_tilde, consts.q_tilde, consts.mu,
                              group_windows=shape.group_windows, pos0=pos0)


class GpuLayer:
    """One sealed layer on the GPU, driven through the C ABI."""

    def __init__(self, shape: synth.Shape, consts, rect=False, scale=None, max_rows=4096, pos0=0,
                 scratch_rows=None):
        import torch
        from sliding_window_landmark_gb300 import o1
        self.torch, self.o1, self.shape = torch, o1, shape
        self.g = o1.geom(shape.groups, shape.heads_per_group, shape.d, shape.dv, shape.sinks, shape.window,
                         shape.landmarks, scale=scale, rope_base=shape.rope_base, rect_far_mass=rect)
        dev = torch.device("cuda")
        self.dev = dev
        self.state = torch.empty(o1.o1_state_bytes(self.g), dtype=torch.uint8, device=dev)
        self.scratch = torch.empty(o1.o1_scratch_bytes(self.g, scratch_rows or max_rows), dtype=torch.uint8,
                                   device=dev)
        up = self.up
        self._c = [up(consts.sink_k) if shape.sinks else None, up(consts.sink_v) if shape.sinks else None,
                   up(consts.k_tilde), up(consts.q_tilde), up(consts.mu)]
        o1.check(o1.o1_state_init(self.state, self.g, shape.group_windows, *self._c, pos0), "init")

    def up(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(self.dev)

    def rows(self, q, k, v, gate=None):
        o1, torch = self.o1, self.torch
        rows = q.shape[0]
        out = torch.empty((rows, self.g.nh, self.g.dv), dtype=torch.float32, device=self.dev)
        qd, kd, vd = self.up(q), self.up(k), self.up(v)
        gd = self.up(gate) if gate is not None else None
        o1.check(o1.o1_chunk_attend(self.state, self.g, self.scratch, qd, kd, vd, gd, rows, out), "chunk")
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def tokens(self, q, k, v, gate=None):
        """Row by row through o1_token_attend."""
        o1, torch = self.o1, self.torch
        rows = q.shape[0]
        out = torch.empty((rows, self.g.nh, self.g.dv), dtype=torch.float32, device=self.dev)
        qd, kd, vd = self.up(q), self.up(k), self.up(v)
        gd = self.up(gate) if gate is not None else None
        for r in range(rows):
            o1.check(o1.o1_token_attend(self.state, self.g, self.scratch, qd[r], kd[r], vd[r],
                                        None if gd is None else gd[r], out[r]), "token")
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def read(self):
        arrs = self.o1.empty_state_arrays(self.g)
        self.o1.check(self.o1.o1_state_read(self.state, self.g, arrs), "read")
        return arrs


def flip_rows(diag):
    """Row-heads whose far mass cancels to within FLIP_MARGIN of its terms."""
    have, D, Dabs = diag[:3]
    return (Dabs > 0) & (np.abs(D) <= FLIP_MARGIN * Dabs)


def assert_outputs(got, want, diag=None, what=""):
    """The strict tolerance on every row-head but the flip-adjacent ones;
    prints the call's figures (max error over tolerance, flip-adjacent
    rows) and the worst rows before failing."""
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rows = want.shape[:2]
    skip = np.zeros(rows, dtype=bool) if diag is None else flip_rows(diag)
    err = np.abs(got - want)
    tol = ATOL + RTOL * np.abs(want)
    ratio = np.where(skip[..., None], 0.0, err / tol)
    row_ratio = ratio.max(axis=-1)
    bad = row_ratio > 1.0
    worst = float(row_ratio.max()) if row_ratio.size else 0.0
    print(f"PARITY {what}: max err/tol {worst:.4f}; row-heads above the tolerance {int(bad.sum())}; "
          f"flip-adjacent (|D| <= {FLIP_MARGIN} A) {int(skip.sum())} of {skip.size}", flush=True)
    if bad.any():
        order = np.argsort(-row_ratio, axis=None)[:5]
        info = []
        for wi in order:
            r_, h_ = np.unravel_index(wi, rows)
            dd = (f" have {int(diag[0][r_, h_])} D/A {diag[1][r_, h_] / max(diag[2][r_, h_], 1e-300):.3g}"
                  if diag is not None else "")
            info.append(f"(row {r_}, head {h_}): err/tol {row_ratio[r_, h_]:.3g} max|o| "
                        f"{np.abs(want[r_, h_]).max():.3g}{dd}")
        raise AssertionError(f"{what}: {int(bad.sum())} row-heads out of tolerance; worst " + "; ".join(info))
    keep = ~skip
    return {"max_abs": float(err[keep].max()) if keep.any() else 0.0,
            "max_rel_to_tol": worst, "flip_rows": int(skip.sum()),
            "have_frac": float(diag[0].mean()) if diag is not None else None}


def assert_state(gpu: dict, orc: oracle.OracleLayer, what=""):
    """Meta and position bit-exact, ring values bit-exact, rotated ring keys and
    the far field within tolerance (the far field compared as Z e^M, T e^M
    against the oracle's own max)."""
    np.testing.assert_array_equal(gpu["meta"].astype(np.int64), orc.meta.astype(np.int64), err_msg=what + " meta")
    assert int(gpu["pos"][0]) == int(orc.pos[0]), what + " pos"
    G = orc.meta.shape[0]
    for gi in range(G):
        ln, wg = int(orc.meta[gi, 0]), int(orc.meta[gi, 3])
        # slots holding keys: all of them once the ring has filled, else the first len
        used = np.arange(wg) if ln == wg else np.arange(ln)
        np.testing.assert_array_equal(gpu["ring_v"][gi, used], orc.ring_v[gi, used].astype(np.float32),
                                      err_msg=what + " ring_v")
        rk = gpu["ring_k"][gi, used].astype(np.float64)
        ok = np.abs(rk - orc.ring_k[gi, used]) <= 1e-5 + 1e-5 * np.abs(orc.ring_k[gi, used])
        assert ok.all(), what + f" ring_k group {gi}"
    M = gpu["far_max"].astype(np.float64)
    empty = np.isneginf(orc.M)
    assert (np.isneginf(M) == empty).all(), what + " far field emptiness"
    assert (gpu["far_mass"][empty] == 0).all() and (gpu["far_val"][empty] == 0).all(), what + " empty far field"
    live = ~empty
    if live.any():
        assert np.abs(M[live] - orc.M[live]).max() <= 1e-4, what + " far max"
        f = np.exp(M - np.where(live, orc.M, 0.0))
        Zg = gpu["far_mass"].astype(np.float64) * np.where(live, f, 0.0)
        np.testing.assert_allclose(Zg[live], orc.Z[live], rtol=1e-4, atol=1e-6, err_msg=what + " far mass")
        Tg = gpu["far_val"].astype(np.float64) * np.where(live, f, 0.0)[..., None]
        tol = 2e-4 * (1.0 + orc.Z[..., None]) + 1e-4 * np.abs(orc.T)
        bad = (np.abs(Tg - orc.T) > tol) & live[..., None]
        assert not bad.any(), what + f" far value sum: {bad.sum()} out of tolerance"

"""Pins of the serial oracle against what the method and mathematics fix.

None of these re-runs the oracle's own formulas: each compares it with a
different computation of the same quantity (textbook softmax attention, a
brute-force far sum with no running max and no ring, a closed form, a
recomputation from the evicted keys, the meta closed form, rotation worked
values and invariants, forced branches). The method is the one of
"cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs" (module doc; o1b_far_e,
o1b_attend, o1b_far_commit, o1b_ring_commit, o1b_meta) with the rotation of
"cortiq-engine 0.8.77 src/gpu_wgpu/dory.rs" (dory_prep, table in `run`).
"""
import math

import numpy as np
import pytest

import oracle
from sliding_window_landmark_gb300 import synth


# ---------------------------------------------------------------- helpers

def _layer(shape, seed, mu_abs=False, rect=False, scale=None, consts=None, lib=None):
    c = consts or synth.layer_constants(shape, seed, mu_abs=mu_abs)
    g = oracle.Geom(shape.groups, shape.heads_per_group, shape.d, shape.dv, shape.sinks,
                    shape.window, shape.landmarks, scale=scale, rope_base=shape.rope_base,
                    rect_far_mass=rect)
    lay = oracle.OracleLayer(g, c.sink_k, c.sink_v, c.k_tilde, c.q_tilde, c.mu,
                             group_windows=shape.group_windows, lib=lib)
    return lay, c, g


def _rot_table(d, p, base):
    """Textbook half-split rotary angles with the table rounded to f32 as the
    pages store it (dory.rs `run`: cos/sin in f64, kept as f32)."""
    half = d // 2
    j = np.arange(half)
    inv = np.array([np.float32(base ** (-2.0 * jj / d)) for jj in j], dtype=np.float64)
    ang = float(p) * inv
    return np.cos(ang).astype(np.float32).astype(np.float64), np.sin(ang).astype(np.float32).astype(np.float64)


def _rot(x, p, base):
    x = np.asarray(x, dtype=np.float64)
    if base == 0:
        return x.copy()
    d = x.shape[-1]
    c, s = _rot_table(d, p, base)
    a, b = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-np.asarray(x, dtype=np.float64)))


def _brute(shape, consts, q, k, v, gate, scale, rect=False, pos0=0):
    """Far algebra by brute force: for every row, the near set (sinks + the
    last min(wg, r+1) keys) with plain exponentials, and the far part as an
    explicit sum over every key evicted so far of
    K(q, k_e) = sum_b u_b(q) exp(scale qt_b . k_e), u_b = sum_a exp(scale q.kt_a) mu[a][b].
    No running max, no ring, no prefix state."""
    G, hpg, nh = shape.groups, shape.heads_per_group, shape.nh
    rows = q.shape[0]
    wins = shape.group_windows or (shape.window,) * G
    out = np.zeros((rows, nh, shape.dv))
    have = np.zeros((rows, nh), dtype=np.int8)
    marg = np.full((rows, nh), np.inf)
    kr = np.stack([_rot(k[r], pos0 + r, shape.rope_base) for r in range(rows)])  # [rows][G][d]
    for r in range(rows):
        for gi in range(G):
            wg = wins[gi]
            lo = max(0, r + 1 - wg)
            near_k = np.concatenate([consts.sink_k[gi].astype(np.float64), kr[lo:r + 1, gi]], 0)
            near_v = np.concatenate([consts.sink_v[gi].astype(np.float64), v[lo:r + 1, gi].astype(np.float64)], 0)
            ev = r + 1 - wg  # keys 0 .. ev-1 have been evicted
            for h in range(hpg):
                gh = gi * hpg + h
                qr = _rot(q[r, gh], pos0 + r, shape.rope_base)
                e_near = np.exp(scale * near_k @ qr)
                num = e_near @ near_v
                den = e_near.sum()
                if ev > 0:
                    f = scale * consts.k_tilde[gi].astype(np.float64) @ qr
                    u = np.exp(f) @ consts.mu[gh].astype(np.float64)
                    if rect:
                        u = np.maximum(u, 0.0)
                    ke = kr[:ev, gi]
                    kern = np.exp(scale * consts.q_tilde[gi, h].astype(np.float64) @ ke.T)  # [m][ev]
                    kq = u @ kern  # [ev]
                    D = kq.sum()
                    marg[r, gh] = abs(D) / max(np.abs(u[:, None] * kern).sum(), 1e-300)
                    if D >= 0:
                        have[r, gh] = 1
                        num = num + kq @ v[:ev, gi].astype(np.float64)
                        den = den + D
                o = num / den
                if gate is not None:
                    o = o * _sigmoid(gate[r, gh])
                out[r, gh] = o
    return out, have, marg


# ------------------------------------------------------------------ pins

def test_rope_worked_values(lib=None):
    """Half-split rotation (dory.rs dory_prep: element j with j + d/2) at
    position 1, base 1e6, d = 4: angles 1 and 1e-3 (f32)."""
    x = np.array([1.0, 2.0, 3.0, 4.0], dtype=np.float32)
    got = oracle.rope(x, 1, 1e6, lib=lib)
    c1, s1 = float(np.float32(math.cos(1.0))), float(np.float32(math.sin(1.0)))
    t = float(np.float32(1e-3))
    c2, s2 = float(np.float32(math.cos(t))), float(np.float32(math.sin(t)))
    want = [1 * c1 - 3 * s1, 2 * c2 - 4 * s2, 3 * c1 + 1 * s1, 4 * c2 + 2 * s2]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_rope_invariants(lib=None):
    rng = np.random.default_rng(0)
    d = 64
    x = rng.standard_normal(d).astype(np.float32)
    y = rng.standard_normal(d).astype(np.float32)
    # p = 0 is the identity
    np.testing.assert_array_equal(oracle.rope(x, 0, 1e6, lib=lib), x.astype(np.float64))
    for p in (1, 17, 1000, 123456):
        rx = oracle.rope(x, p, 1e6, lib=lib)
        # pair norms are preserved (f32 cos/sin: |c^2+s^2-1| <= ~1e-7)
        pn = rx[: d // 2] ** 2 + rx[d // 2:] ** 2
        pn0 = x[: d // 2].astype(np.float64) ** 2 + x[d // 2:].astype(np.float64) ** 2
        np.testing.assert_allclose(pn, pn0, rtol=3e-7)
    # the score depends only on the position difference
    s1 = oracle.rope(x, 100, 1e6, lib=lib) @ oracle.rope(y, 90, 1e6, lib=lib)
    s2 = oracle.rope(x, 5010, 1e6, lib=lib) @ oracle.rope(y, 5000, 1e6, lib=lib)
    assert abs(s1 - s2) < 1e-4 * (np.abs(x).sum() * np.abs(y).sum()) ** 0.5
    # base 0 turns rotation off
    np.testing.assert_array_equal(oracle.rope(x, 77, 0.0, lib=lib), x.astype(np.float64))


@pytest.mark.parametrize("rope_base", [1e6, 0.0])
def test_no_eviction_is_exact_softmax(rope_base, lib=None):
    """While no key has been evicted, the output is exact softmax attention
    over the sinks plus every key so far, times the sigmoid gate."""
    sh = synth.Shape(groups=2, heads_per_group=3, d=16, dv=8, sinks=3, window=24, landmarks=4,
                     rope_base=rope_base)
    lay, c, g = _layer(sh, seed=11, lib=lib)
    rows = 24
    q, k, v, gate = synth.layer_rows(sh, 11, 0, rows)
    got = np.concatenate([lay.rows(q[:7], k[:7], v[:7], gate[:7]),
                          lay.rows(q[7:], k[7:], v[7:], gate[7:])])
    scale = g.scale_f32()
    for r in range(rows):
        for gi in range(sh.groups):
            keys = np.concatenate([c.sink_k[gi].astype(np.float64),
                                   np.stack([_rot(k[j, gi], j, rope_base) for j in range(r + 1)])])
            vals = np.concatenate([c.sink_v[gi].astype(np.float64), v[: r + 1, gi].astype(np.float64)])
            for h in range(sh.heads_per_group):
                gh = gi * sh.heads_per_group + h
                s = scale * keys @ _rot(q[r, gh], r, rope_base)
                p = np.exp(s - s.max())
                want = (p @ vals) / p.sum() * _sigmoid(gate[r, gh])
                np.testing.assert_allclose(got[r, gh], want, rtol=1e-12, atol=1e-12)
    assert (lay.meta[:, 2] == 0).all()


BRUTE_CASES = [
    # (G, hpg, d, dv, ns, window, group windows, m, rows, rope, rect, mu_abs, splits)
    (2, 2, 8, 6, 2, 5, (3, 5), 3, 40, 0.0, False, False, (40,)),
    (2, 2, 8, 6, 2, 5, (5, 4), 3, 37, 1e6, False, False, (9, 1, 27)),
    (1, 3, 4, 4, 0, 4, None, 2, 30, 1e4, False, True, (30,)),
    (2, 1, 6, 5, 1, 5, (2, 5), 3, 33, 1e6, True, False, (33,)),
    (1, 2, 8, 8, 3, 3, None, 1, 25, 0.0, False, True, (5, 20)),
]


@pytest.mark.parametrize("case", BRUTE_CASES)
def test_brute_force_far_algebra(case, lib=None):
    """The whole far algebra against a brute-force sum on tiny shapes."""
    G, hpg, d, dv, ns, w, gw, m, rows, rope_base, rect, mu_abs, splits = case
    sh = synth.Shape(groups=G, heads_per_group=hpg, d=d, dv=dv, sinks=ns, window=w, landmarks=m,
                     rope_base=rope_base, group_windows=gw)
    lay, c, g = _layer(sh, seed=5 + rows, mu_abs=mu_abs, rect=rect, lib=lib)
    q, k, v, gate = synth.layer_rows(sh, 5 + rows, 0, rows)
    outs, haves = [], []
    r0 = 0
    for n in splits:
        o, (hv, _, _, _) = lay.rows(q[r0:r0 + n], k[r0:r0 + n], v[r0:r0 + n], gate[r0:r0 + n], diag=True)
        outs.append(o)
        haves.append(hv)
        r0 += n
    got = np.concatenate(outs)
    have = np.concatenate(haves)
    want, bh, marg = _brute(sh, c, q, k, v, gate, g.scale_f32(), rect=rect)
    ok = marg > 1e-7  # decision not within rounding of zero
    assert ok.mean() > 0.9
    np.testing.assert_array_equal(have[ok], bh[ok])
    np.testing.assert_allclose(got[ok], want[ok], rtol=1e-9, atol=1e-11)
    # the far part is really exercised
    assert have.sum() > 10


def test_unit_kernel_closed_form(lib=None):
    """qt = 0, kt = 0, mu = 1/m^2 (exact in f32 for m = 4) make every far weight 1:
    out = (sum_near e^s v + sum_evicted v) / (sum_near e^s + |evicted|)."""
    sh = synth.Shape(groups=1, heads_per_group=2, d=32, dv=16, sinks=2, window=8, landmarks=4,
                     rope_base=1e6)
    c = synth.layer_constants(sh, 3)
    c.q_tilde[:] = 0
    c.k_tilde[:] = 0
    c.mu[:] = 1.0 / sh.landmarks ** 2
    lay, _, g = _layer(sh, 3, consts=c, lib=lib)
    rows = 30
    q, k, v, _ = synth.layer_rows(sh, 3, 0, rows, gate=False)
    got = lay.rows(q, k, v)
    scale = g.scale_f32()
    for r in range(rows):
        lo = max(0, r + 1 - sh.window)
        keys = np.concatenate([c.sink_k[0].astype(np.float64),
                               np.stack([_rot(k[j, 0], j, 1e6) for j in range(lo, r + 1)])])
        vals = np.concatenate([c.sink_v[0].astype(np.float64), v[lo:r + 1, 0].astype(np.float64)])
        for h in range(2):
            e = np.exp(scale * keys @ _rot(q[r, h], r, 1e6))
            want = (e @ vals + v[:lo, 0].astype(np.float64).sum(0)) / (e.sum() + lo)
            np.testing.assert_allclose(got[r, h], want, rtol=1e-11, atol=1e-12)


def test_far_state_recomputation_and_monotone_max(lib=None):
    """M_b = max over evicted keys of l_be, Z_b e^M_b = sum e^l, T_b e^M_b =
    sum e^l v; M never decreases; farl == 0 iff the far field is empty."""
    sh = synth.Shape(groups=2, heads_per_group=2, d=16, dv=8, sinks=2, window=6, landmarks=3,
                     rope_base=1e6, group_windows=(4, 6))
    lay, c, g = _layer(sh, 21, lib=lib)
    rows = 40
    q, k, v, gate = synth.layer_rows(sh, 21, 0, rows)
    scale = g.scale_f32()
    prevM = lay.M.copy()
    for r in range(rows):
        lay.rows(q[r:r + 1], k[r:r + 1], v[r:r + 1], gate[r:r + 1])
        assert (lay.M >= prevM).all()
        prevM = lay.M.copy()
        for gi, wg in enumerate(sh.group_windows):
            ev = r + 1 - wg
            for h in range(2):
                gh = gi * 2 + h
                if ev <= 0:
                    assert lay.meta[gi, 2] == 0
                    assert np.isneginf(lay.M[gh]).all() and (lay.Z[gh] == 0).all() and (lay.T[gh] == 0).all()
                    continue
                assert lay.meta[gi, 2] == ev
                ke = np.stack([_rot(k[j, gi], j, 1e6) for j in range(ev)])
                l = scale * c.q_tilde[gi, h].astype(np.float64) @ ke.T  # [m][ev]
                np.testing.assert_allclose(lay.M[gh], l.max(1), rtol=1e-13, atol=1e-13)
                np.testing.assert_allclose(lay.Z[gh] * np.exp(lay.M[gh]), np.exp(l).sum(1), rtol=1e-11)
                np.testing.assert_allclose(lay.T[gh] * np.exp(lay.M[gh])[:, None],
                                           np.exp(l) @ v[:ev, gi].astype(np.float64), rtol=1e-10, atol=1e-12)


def test_meta_closed_form_and_ring_slots(lib=None):
    """After n pushes: len = min(wg, n), ev = max(0, n - wg), head = ev mod wg,
    farl = ev; slot (len0 + head0 + j) mod wg holds row j for the last wg rows."""
    sh = synth.Shape(groups=3, heads_per_group=1, d=8, dv=4, sinks=1, window=7, landmarks=2,
                     rope_base=0.0, group_windows=(7, 3, 5))
    lay, c, g = _layer(sh, 4, lib=lib)
    q, k, v, _ = synth.layer_rows(sh, 4, 0, 50, gate=False)
    n = 0
    for chunk in (1, 2, 6, 1, 13, 27):
        lay.rows(q[n:n + chunk], k[n:n + chunk], v[n:n + chunk])
        n += chunk
        for gi, wg in enumerate(sh.group_windows):
            ev = max(0, n - wg)
            assert tuple(lay.meta[gi]) == (min(wg, n), ev % wg, ev, wg)
            for j in range(max(0, n - wg), n):
                slot = j % wg  # head0 = len0 = 0 at the start
                np.testing.assert_array_equal(lay.ring_k[gi, slot], k[j, gi].astype(np.float64))
                np.testing.assert_array_equal(lay.ring_v[gi, slot], v[j, gi].astype(np.float64))
    assert int(lay.pos[0]) == n


def test_position_shift_invariance(lib=None):
    """With no sinks and nothing evicted, outputs depend on position
    differences only: shifting the start position leaves them unchanged."""
    sh = synth.Shape(groups=1, heads_per_group=2, d=32, dv=8, sinks=0, window=16, landmarks=2,
                     rope_base=1e4)
    c = synth.layer_constants(sh, 8)
    q, k, v, gate = synth.layer_rows(sh, 8, 0, 16)
    outs = []
    for pos0 in (0, 1000):
        g = oracle.Geom(1, 2, 32, 8, 0, 16, 2, rope_base=1e4)
        lay = oracle.OracleLayer(g, c.sink_k, c.sink_v, c.k_tilde, c.q_tilde, c.mu, pos0=pos0, lib=lib)
        outs.append(lay.rows(q, k, v, gate))
    np.testing.assert_allclose(outs[0], outs[1], rtol=0, atol=2e-5)


def test_forced_far_branches(lib=None):
    """m = 1 with mu = -1 makes the far mass negative: the far part is dropped
    and the output is near-only softmax. With the rectifier, mu = -1 gives
    u = 0: the far part is kept but adds nothing."""
    for rect in (False, True):
        sh = synth.Shape(groups=1, heads_per_group=2, d=16, dv=8, sinks=2, window=5, landmarks=1,
                         rope_base=1e6)
        c = synth.layer_constants(sh, 9)
        c.mu[:] = -1.0
        lay, _, g = _layer(sh, 9, rect=rect, consts=c, lib=lib)
        rows = 20
        q, k, v, gate = synth.layer_rows(sh, 9, 0, rows)
        got, (have, D, _, _) = lay.rows(q, k, v, gate, diag=True)
        scale = g.scale_f32()
        for r in range(rows):
            lo = max(0, r + 1 - 5)
            keys = np.concatenate([c.sink_k[0].astype(np.float64),
                                   np.stack([_rot(k[j, 0], j, 1e6) for j in range(lo, r + 1)])])
            vals = np.concatenate([c.sink_v[0].astype(np.float64), v[lo:r + 1, 0].astype(np.float64)])
            for h in range(2):
                s = scale * keys @ _rot(q[r, h], r, 1e6)
                p = np.exp(s - s.max())
                want = p @ vals / p.sum() * _sigmoid(gate[r, h])
                np.testing.assert_allclose(got[r, h], want, rtol=1e-12, atol=1e-13)
                if r >= 5:
                    assert have[r, h] == (1 if rect else 0)
                    assert (D[r, h] == 0.0) if rect else (D[r, h] < 0.0)


def _floor_layer(mu_value, lib=None):
    """One group, one head, one landmark, window 2, rotation off. Every key
    is e0 and the landmark query is 400 e0, so an evicted key's far logit is
    l = scale * 400 (about 141) while every near score stays below 1: once a
    key is evicted the far max F + M dominates the row's exponent c by more
    than 100, every near weight e^{s - c} is below e^-140, and the
    denominator meets the 1e-30 floor unless the far mass carries it.
    The landmark key is zero (F = 0) and mu = mu_value."""
    sh = synth.Shape(groups=1, heads_per_group=1, d=8, dv=4, sinks=1, window=2, landmarks=1, rope_base=0.0)
    c = synth.layer_constants(sh, 17)
    c.sink_k[:] = 0.0
    c.k_tilde[:] = 0.0
    c.q_tilde[:] = 0.0
    c.q_tilde[0, 0, 0, 0] = 400.0
    c.mu[:] = np.float32(mu_value)
    lay, _, g = _layer(sh, 17, consts=c, lib=lib)
    rows = 5
    q, _, v, _ = synth.layer_rows(sh, 17, 0, rows, gate=False)
    q = (0.1 * q).astype(np.float32)
    k = np.zeros((rows, 1, 8), dtype=np.float32)
    k[:, 0, 0] = 1.0
    return sh, c, g, lay, q, k, v


FLOOR_CASES = [3e-31, 4e-30, -1.0]


@pytest.mark.parametrize("mu_value", FLOOR_CASES)
def test_denominator_floor(mu_value, lib=None):
    """The 1e-30 floor on the denominator (o1_batch.rs o1b_attend; dory.rs
    dory_osoft), taken in the units where the row's largest exponent is 0.
    With the far max dominating (see _floor_layer), after n evictions the far
    field holds M = l, Z = n, T = v_0 + ... + v_{n-1} exactly (every logit is
    equal), the gain is mu, and the near terms are below e^-140:
      mu > 0: out = mu T / max(mu Z, 1e-30): the evicted values' sum scaled
              by mu / 1e-30 while mu Z < 1e-30 (3e-31: a floored
              denominator), their mean once mu Z > 1e-30 (4e-30);
      mu < 0: the far part is dropped but its max still sets the exponent,
              so out = sum_x e^{s_x - l} v_x / 1e-30, about 1e-31 |v|."""
    sh, c, g, lay, q, k, v = _floor_layer(mu_value, lib=lib)
    got = lay.rows(q, k, v, None)
    scale = g.scale_f32()
    l = scale * 400.0
    mu = float(np.float32(mu_value))
    for r in range(2, 5):
        n = r - 1   # keys 0 .. r - 2 evicted
        if mu > 0:
            T = v[:n, 0].astype(np.float64).sum(axis=0)
            want = mu * T / max(mu * n, 1e-30)
            np.testing.assert_allclose(got[r, 0], want, rtol=1e-9, atol=0)
        else:
            keys = np.concatenate([c.sink_k[0].astype(np.float64), k[r - 1:r + 1, 0].astype(np.float64)])
            vals = np.concatenate([c.sink_v[0].astype(np.float64), v[r - 1:r + 1, 0].astype(np.float64)])
            s = scale * keys @ q[r, 0].astype(np.float64)
            want = np.exp(s - l) @ vals / 1e-30
            np.testing.assert_allclose(got[r, 0], want, rtol=1e-9, atol=0)
            assert 0 < np.abs(want).max() < 1e-29


def test_threads_do_not_change_results(lib=None):
    sh = synth.Shape(groups=3, heads_per_group=2, d=16, dv=8, sinks=2, window=6, landmarks=3,
                     group_windows=(6, 4, 5))
    q, k, v, gate = synth.layer_rows(sh, 2, 0, 30)
    res = []
    for th in (1, 3):
        lay, _, _ = _layer(sh, 2, lib=lib)
        res.append((lay.rows(q, k, v, gate, threads=th), lay.snapshot()))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    for key in ("meta", "ring_k", "M", "Z", "T"):
        np.testing.assert_array_equal(res[0][1][key], res[1][1][key])


def test_meta_rewind_closed_form(lib=None):
    """Rewinding pushes (dory.rs dory_o1_back, applied once per row): on a ring
    not yet full, k rewinds after n pushes leave len = n - k (head, farl
    unchanged); on a full ring after n pushes (ev = n - wg evictions), k <= ev
    rewinds leave len = wg, farl = ev - k, head = (ev - k) mod wg; the position
    moves back by k; ring contents and the far field are untouched; a rewind
    some group cannot take is refused with nothing changed."""
    sh = synth.Shape(groups=3, heads_per_group=1, d=8, dv=4, sinks=1, window=7, landmarks=2,
                     rope_base=0.0, group_windows=(7, 3, 5))
    lay, c, g = _layer(sh, 6, lib=lib)
    q, k, v, _ = synth.layer_rows(sh, 6, 0, 40, gate=False)
    lay.rows(q[:2], k[:2], v[:2])
    # group windows 7, 3, 5 after 2 pushes: none full
    snap = lay.snapshot()
    assert lay.back(2)
    for gi, wg in enumerate(sh.group_windows):
        assert tuple(lay.meta[gi]) == (0, 0, 0, wg)
    assert int(lay.pos[0]) == 0
    for key in ("ring_k", "ring_v", "M", "Z", "T"):
        np.testing.assert_array_equal(lay.snapshot()[key], snap[key])
    # refused: a ring with fewer entries than the rewind
    assert not lay.back(1)
    assert int(lay.pos[0]) == 0
    n = 23
    lay.rows(q[:n], k[:n], v[:n])
    for kk in (1, 3, 9):
        before = lay.snapshot()
        assert lay.back(kk)
        for gi, wg in enumerate(sh.group_windows):
            ev = n - wg
            assert tuple(lay.meta[gi]) == (wg, (ev - kk) % wg, ev - kk, wg)
        assert int(lay.pos[0]) == n - kk
        for key in ("ring_k", "ring_v", "M", "Z", "T"):
            np.testing.assert_array_equal(lay.snapshot()[key], before[key])
        lay.rows(q[n - kk:n], k[n - kk:n], v[n - kk:n])   # push the same rows again
    # more evictions to rewind than group 0 (window 7, 16 evictions) has
    assert not lay.back(17)
    for gi, wg in enumerate(sh.group_windows):
        assert tuple(lay.meta[gi]) == (wg, (n - wg) % wg, n - wg, wg)


def test_rewind_then_repush_reproduces_rows(lib=None):
    """On a ring that never fills, nothing reaches the far field, so rewinding
    n rows and pushing the same n rows again gives the same outputs and the
    same state, exactly."""
    sh = synth.Shape(groups=2, heads_per_group=2, d=16, dv=8, sinks=2, window=32, landmarks=3)
    lay, c, g = _layer(sh, 8, lib=lib)
    q, k, v, gt = synth.layer_rows(sh, 8, 0, 20)
    lay.rows(q[:10], k[:10], v[:10], gt[:10])
    first = lay.rows(q[10:], k[10:], v[10:], gt[10:])
    snap = lay.snapshot()
    assert lay.back(10)
    again = lay.rows(q[10:], k[10:], v[10:], gt[10:])
    np.testing.assert_array_equal(first, again)
    for key, val in lay.snapshot().items():
        np.testing.assert_array_equal(val, snap[key], err_msg=key)

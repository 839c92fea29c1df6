"""The seeded input generator both sides draw from: SplitMix64 against its
published output sequence, the Box-Muller draws against N(0, 1) statistics,
and the counter property (any slice of any tensor is reproducible on its
own), which lets a parity test ask for rows r0 .. r0 + n of a prompt without
generating the rows before them."""
import math

import numpy as np

from sliding_window_landmark_gb300 import synth


def test_splitmix64_published_sequence():
    """SplitMix64 from state 0 (Steele, Lea and Flood, OOPSLA 2014; the
    reference implementation advances the state by the golden gamma and
    mixes): its first three outputs."""
    gamma = int(synth._GAMMA)
    states = np.array([0, gamma, (2 * gamma) % 2 ** 64], dtype=np.uint64)
    got = [int(x) for x in synth._mix(states)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_normal_draws_have_standard_normal_statistics():
    n = 1 << 20
    x = synth.normal(7, 0, synth.Q, (n,)).astype(np.float64)
    se = 1.0 / math.sqrt(n)
    assert abs(x.mean()) < 5 * se
    assert abs(x.var() - 1.0) < 5 * math.sqrt(2.0) * se
    p1 = 0.6826894921370859   # P(|X| < 1) for X ~ N(0, 1)
    assert abs(np.mean(np.abs(x) < 1.0) - p1) < 5 * math.sqrt(p1 * (1 - p1)) * se
    kurt = np.mean(x ** 4) / x.var() ** 2
    assert abs(kurt - 3.0) < 5 * math.sqrt(96.0) * se
    a = synth.normal(7, 0, synth.MU, (n,), absolute=True)
    assert (a >= 0).all() and abs(a.mean() - math.sqrt(2 / math.pi)) < 5 * se


def test_streams_are_independent():
    n = 1 << 18
    base = synth.normal(3, 2, synth.K, (n,)).astype(np.float64)
    for other in (synth.normal(3, 2, synth.V, (n,)), synth.normal(3, 3, synth.K, (n,)),
                  synth.normal(4, 2, synth.K, (n,))):
        assert abs(np.corrcoef(base, other.astype(np.float64))[0, 1]) < 5 / math.sqrt(n)


def test_any_slice_is_reproducible_alone():
    full = synth.normal(11, 1, synth.GATE, (5000,))
    np.testing.assert_array_equal(synth.normal(11, 1, synth.GATE, (1234,), offset=3000), full[3000:4234])
    sh = synth.Shape(groups=2, heads_per_group=3, d=16, dv=8, sinks=2, window=32, landmarks=4)
    whole = synth.layer_rows(sh, 5, 0, 90)
    part = synth.layer_rows(sh, 5, 37, 40)
    for w, p in zip(whole, part):
        np.testing.assert_array_equal(w[37:77], p)

"""The precision argument of the tensor-core window path, emulated on the
CPU with numpy's IEEE half precision.

Each fp32 operand x is split into x_hi = fp16(x) and x_lo = fp16(x - x_hi)
(the subtraction is exact in fp32), and a product is taken as
hi.hi + hi.lo + lo.hi with fp32 accumulation: the error-compensated split of
Markidis et al. (2018) and Ootomo & Yokota (2022), here with fp16 halves.
The dropped lo.lo term is about 2^-22 of |x y|. So a dot product of d terms
should land within a few times 2^-22 of the exact one, relative to the sum
of |x_i y_i|, plus fp32 accumulation. A single fp16 pass is off by about
2^-11, which is why the path does not use one.
"""
import numpy as np


def _split(x):
    hi = x.astype(np.float16)
    lo = (x - hi.astype(np.float32)).astype(np.float16)
    return hi.astype(np.float32), lo.astype(np.float32)


def _dot_fp32(a, b):
    acc = np.zeros(a.shape[0], dtype=np.float32)
    for i in range(a.shape[1]):
        acc = acc + a[:, i] * b[:, i]   # one fp32 product and add per term, in order
    return acc


def test_three_term_split_dot_products():
    rng = np.random.default_rng(5)
    d, n = 256, 2000
    q = rng.standard_normal((n, d)).astype(np.float32)
    k = rng.standard_normal((n, d)).astype(np.float32)
    exact = np.sum(q.astype(np.float64) * k.astype(np.float64), axis=1)
    scale = np.sum(np.abs(q.astype(np.float64) * k.astype(np.float64)), axis=1)
    qh, ql = _split(q)
    kh, kl = _split(k)
    three = _dot_fp32(qh, kh) + _dot_fp32(qh, kl) + _dot_fp32(ql, kh)
    one = _dot_fp32(qh, kh)
    rel3 = np.abs(three.astype(np.float64) - exact) / scale
    rel1 = np.abs(one.astype(np.float64) - exact) / scale
    # the split: a few times 2^-22 per term, plus fp32 accumulation over d terms
    assert rel3.max() < 4 * 2.0 ** -22 + 2 * 2.0 ** -24 * np.sqrt(d)
    # one fp16 pass: about a thousand times worse (2e-5 median, 1e-4 at worst
    # here), which the 1e-4 relative tolerance on outputs cannot absorb
    assert np.median(rel1) > 300 * np.median(rel3) and rel1.max() > 5e-5


def test_split_of_short_mantissas_is_exact_and_range_is_bounded():
    """Values with at most 22 significant bits split into hi + lo exactly;
    values beyond fp16's largest finite (65504) do not fit, which is why the
    path raises O1_FLAG_FP16_RANGE for them."""
    x = np.array([1.0, -2.5, 0.099975586, 1024.0, 3.0517578e-05], dtype=np.float32)
    hi, lo = _split(x)
    np.testing.assert_array_equal(hi + lo, x)
    with np.errstate(over="ignore"):
        assert not np.isfinite(np.array([70000.0], dtype=np.float32).astype(np.float16)).all()

"""The float32 layer's tensor-core arithmetic, emulated on the CPU.

The float32 expert GEMMs split every operand v into hi = v with its low 13 mantissa bits
cleared (a tf32 value) and lo = v - hi, and add three tf32 products per step:
hi_a*hi_b + hi_a*lo_b + lo_a*hi_b.  The tensor core reads lo as tf32 too (its low 13 bits
dropped).  These tests pin the claim that this keeps float32 accuracy: every product is
within 3 * 2^-20 of exact, and dot products stay within the float32 layer's tolerance
(1e-3), where plain tf32 operands would not.
"""

import numpy as np


def tf32_trunc(v):
    """v (float32) with its low 13 mantissa bits cleared."""
    return (np.asarray(v, np.float32).view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)


def split(v):
    v = np.asarray(v, np.float32)
    hi = tf32_trunc(v)
    lo = (v - hi).astype(np.float32)  # exact: the cleared bits
    return hi, lo


def three_product(a, b):
    """hi_a*hi_b + hi_a*lo_b + lo_a*hi_b with each operand read as tf32, in float64."""
    ah, al = split(a)
    bh, bl = split(b)
    ah, al, bh, bl = (tf32_trunc(t).astype(np.float64) for t in (ah, al, bh, bl))
    return ah * bh + ah * bl + al * bh


def test_split_is_exact():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(100_000) * np.exp(rng.uniform(-20, 20, 100_000))).astype(np.float32)
    hi, lo = split(v)
    assert np.array_equal(hi.astype(np.float64) + lo.astype(np.float64), v.astype(np.float64))
    assert np.array_equal(tf32_trunc(hi), hi)  # hi is a tf32 value
    assert (np.abs(lo) < np.abs(v) * 2.0 ** -10 + 1e-45).all()


def test_product_error_bound():
    rng = np.random.default_rng(1)
    a = rng.standard_normal(200_000).astype(np.float32)
    b = rng.standard_normal(200_000).astype(np.float32)
    exact = a.astype(np.float64) * b.astype(np.float64)
    err = np.abs(three_product(a, b) - exact)
    assert (err <= 3 * 2.0 ** -20 * np.abs(exact) + 1e-300).all()
    # plain tf32 operands are three orders of magnitude worse
    plain = tf32_trunc(a).astype(np.float64) * tf32_trunc(b).astype(np.float64)
    assert np.abs(plain - exact).max() > 100 * err.max()


def test_dot_products_meet_the_float32_tolerance():
    # the toy layer's shapes: H = 512 inputs, weights ~ N(0, 0.02)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    w = (rng.standard_normal((256, 512)) * 0.02).astype(np.float32)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    xh, xl = split(x)
    wh, wl = split(w)
    f = lambda t: tf32_trunc(t).astype(np.float64)
    three = f(xh) @ f(wh).T + f(xh) @ f(wl).T + f(xl) @ f(wh).T
    plain = f(x) @ f(w).T
    rel = lambda y: np.linalg.norm(y - exact) / np.linalg.norm(exact)
    assert rel(three) < 1e-5 and np.abs(three - exact).max() < 1e-5
    assert rel(plain) > 1e-4  # tf32 alone gives up about three decimal digits

"""exp2 with a polynomial fractional core -- replay oracle.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

"Fast Polynomial Transcendentals for LLMs" (arXiv 2610.00049), Appendix B.1:
x = n + f, n = floor(x), f in [0, 1), 2^x = 2^n 2^f (eq. 16); only 2^f is
approximated, 2^n is rebuilt from the exponent bits.  Fractional cores:

  D1    p(f) = 1 + f                                    (endpoint constrained)
  PWL2  p(f) = 1 + a f + 2 (1 - a) max(f - 1/2, 0)        (eq. 17)
  D2    p(f) = 1 + a f + (1 - a) f^2                    (eq. 18)
  D3    FA4's p(f) = 1 + 0.6951461434 f + 0.2275643945 f^2 + 0.0771190897 f^3 (eq. 19)

Parameters: "sampled minimax" minimises the maximum relative error on a
1,000,001-point grid of [0, 1]; "least squares" minimises the sum of squared
absolute errors on the same grid (the reading that reproduces the printed
a = 0.7852775264 and 0.6563658611).

Deployed evaluator (this build's definition; the paper's FA4 core is FP16
PWL2 in inline PTX): FP32 in, FP32 out.
  xc = min(max(x, -126), 128);  n = floor(xc);  f = xc - n (FP32, one rounding)
  h  = f rounded to FP16
  core in packed FP16, one rounding per operation, coefficients rounded to
  FP16 (PWL2 uses RN(a) and RN(2 (1 - a)), D2 uses RN(a) and 1 - RN(a)):
    D1    p = fma(h, 1, 1)
    PWL2  p = fma(h, a, 1);  m = max(fma(h, 1, -1/2), 0);  p = fma(m, b, p)
    D2    v = fma(b, h, a);  p = fma(v, h, 1)
    D3    v = fma(c3, h, c2);  v = fma(v, h, c1);  p = fma(v, h, 1)
  y  = FP32 bits of p (exact) + (n << 23)       (exponent reconstruction)
  NaN in -> 0x7FFFFFFF.
"""
from __future__ import annotations

import numpy as np
from scipy.optimize import minimize_scalar

from . import tformat as tf

A_PWL2_MINIMAX = 0.7980513010
A_D2_MINIMAX = 0.6602339719
A_PWL2_LS = 0.7852775264
A_D2_LS = 0.6563658611
FA4_D3 = (1.0, 0.6951461434, 0.2275643945, 0.0771190897)
VARIANTS = ("D1", "PWL2", "D2", "D3")
GRID = 1_000_001


def grid():
    return np.linspace(0.0, 1.0, GRID)


def pwl2(a, f):
    return 1.0 + a * f + 2.0 * (1.0 - a) * np.maximum(f - 0.5, 0.0)


def d2(a, f):
    return 1.0 + a * f + (1.0 - a) * f * f


def d3(f, c=FA4_D3):
    return c[0] + f * (c[1] + f * (c[2] + f * c[3]))


def rel_stats(p, f):
    """(max, rms) relative error of p against 2^f."""
    r = p / np.exp2(f) - 1.0
    return float(np.max(np.abs(r))), float(np.sqrt(np.mean(r * r)))


def fit_minimax(family):
    """a minimising the sampled maximum relative error (bounded 1-D search)."""
    f = grid()
    t = np.exp2(f)
    res = minimize_scalar(lambda a: np.max(np.abs(family(a, f) / t - 1.0)),
                          bounds=(0.5, 1.0), method="bounded", options={"xatol": 1e-12})
    return float(res.x)


def fit_least_squares(family):
    """a minimising the sum of squared absolute errors; p is affine in a."""
    f = grid()
    base = family(0.0, f)
    g = family(1.0, f) - base
    return float(np.sum(g * (np.exp2(f) - base)) / np.sum(g * g))


def f16_coefficients(variant):
    """Target-format constants of each core, as FP16 bit patterns."""
    r = lambda v: int(tf.from_f64(v, "f16"))
    if variant == "D1":
        return (r(1.0),)
    if variant == "PWL2":
        return r(A_PWL2_MINIMAX), r(2.0 * (1.0 - A_PWL2_MINIMAX))
    if variant == "D2":
        a = r(A_D2_MINIMAX)
        return a, r(1.0 - float(tf.decode(np.uint16(a), "f16")))
    return tuple(r(c) for c in FA4_D3[1:])


def core_f16(variant, h):
    """The fractional core on FP16 bit patterns h (one rounding per op)."""
    F = "f16"
    one, mhalf, zero = np.uint16(0x3C00), np.uint16(0xB800), np.uint16(0)
    c = [np.uint16(v) for v in f16_coefficients(variant)]
    if variant == "D1":
        return tf.fma(h, one, one, F)
    if variant == "PWL2":
        p = tf.fma(h, c[0], one, F)
        d = tf.fma(h, one, mhalf, F)
        m = np.where(tf.greater(d, zero, F), d, zero).astype(np.uint16)   # max(d, +0)
        return tf.fma(m, c[1], p, F)
    if variant == "D2":
        v = tf.fma(c[1], h, c[0], F)
        return tf.fma(v, h, one, F)
    v = tf.fma(c[2], h, c[1], F)
    v = tf.fma(v, h, c[0], F)
    return tf.fma(v, h, one, F)


def exp2_replay(variant, x):
    """Deployed evaluator on FP32 inputs x (float32 array) -> uint32 bits."""
    x = np.asarray(x, dtype=np.float32)
    nan = np.isnan(x)
    xc = np.minimum(np.maximum(np.where(nan, np.float32(0), x), np.float32(-126.0)),
                    np.float32(128.0))
    n = np.floor(xc)
    f = (xc - n).astype(np.float32)                 # IEEE single subtraction
    h = f.astype(np.float16).view(np.uint16)        # round to nearest even
    p = core_f16(variant, h).view(np.float16).astype(np.float32)
    y = p.view(np.uint32).astype(np.int64) + (n.astype(np.int64) << 23)
    y = (y & 0xFFFFFFFF).astype(np.uint32)
    return np.where(nan, np.uint32(0x7FFFFFFF), y).astype(np.uint32)

"""Exact FP16 / BF16 fused multiply-add in scaled integers, vectorised.

A second exact model next to ``exact_t`` (Python fractions, one element at a
time), fast enough for tens of millions of triples.  Written independently of
``oracle/tformat.py`` (which rounds an FP64 product and a TwoSum error term):
here every finite value is ``(-1)^s M 2^E`` with an integer significand M, the
product's significand is the integer ``Ma * Mb``, and the exact sum of the
product and the addend is an int64 on the grid of the lower of their two
exponents.  Rounding to the format is done on that integer with shifts (round
to nearest, ties to even, subnormals kept, overflow to infinity); a NaN
result is the canonical 0x7FFF.

Far-apart terms: if the exponents differ by more than GAP, the smaller term
is below 2^(Eb - 17) where 2^Eb is the lowest bit of the larger term, while
every rounding boundary near the larger term (representable numbers and the
midpoints between them) lies on the grid 2^(Eb - fb - 2) with fb <= 10.  So
the smaller term only decides the side of the larger term, and it is
replaced by a single unit of its own sign at 2^(Eb - GAP - 1), which keeps
the int64 below 2^61.
"""
from __future__ import annotations

import numpy as np

FORMATS = {"f16": (5, 10, 15), "bf16": (8, 7, 127)}   # exponent bits, fraction bits, bias
NAN = 0x7FFF
GAP = 38


def _fields(x, fmt):
    eb, fb, bias = FORMATS[fmt]
    emax = (1 << eb) - 1
    x = np.asarray(x, dtype=np.uint16).astype(np.int64)
    s = x >> 15
    e = (x >> fb) & emax
    f = x & ((1 << fb) - 1)
    nan = (e == emax) & (f != 0)
    inf = (e == emax) & (f == 0)
    M = np.where(e > 0, f | (1 << fb), f)
    E = np.maximum(e, 1) - bias - fb
    return s, M, E, nan, inf


def _bitlen(a):
    """floor(log2 a) + 1 for int64 a > 0 (a < 2^62)."""
    af = a.astype(np.float64)
    n = np.floor(np.log2(np.maximum(af, 1.0))).astype(np.int64) + 1
    # float64 may round a up to the next power of two: correct by one
    n = np.where((a >> np.clip(n - 1, 0, 62)) == 0, n - 1, n)
    n = np.where((a >> np.clip(n, 0, 62)) != 0, n + 1, n)
    return n


def _round(V, emin, zsign, fmt):
    """Round V * 2^emin (int64, exact) to the format; zsign = sign of a zero
    result when V == 0."""
    eb, fb, bias = FORMATS[fmt]
    emax = (1 << eb) - 1
    neg = V < 0
    A = np.abs(V)
    nz = A != 0
    L = np.where(nz, _bitlen(np.where(nz, A, 1)), 1)
    k = emin + L - 1                                   # exponent of the top bit
    qe = np.maximum(k, 1 - bias) - fb                  # exponent of the quantum
    sh = qe - emin
    left = np.clip(-sh, 0, 62)
    right = np.clip(sh, 0, 63)
    q_exact = A << left
    q_trunc = np.where(sh >= 63, 0, A >> right)
    rem = np.where(sh >= 63, A, A - (q_trunc << right))
    half = np.where(sh >= 1, np.int64(1) << np.clip(sh - 1, 0, 62), 0)
    half = np.where(sh > 63, np.int64(1) << 62, half)  # A < 2^61 stays below it
    up = (rem > half) | ((rem == half) & ((q_trunc & 1) == 1))
    q = np.where(sh <= 0, q_exact, q_trunc + np.where((sh > 0) & up, 1, 0))
    carry = q >= (1 << (fb + 1))
    q = np.where(carry, q >> 1, q)
    qe = qe + carry
    sign = np.where(nz, neg.astype(np.int64), zsign)
    e = qe + fb + bias
    normal = q >= (1 << fb)
    bits = np.where(normal, (e << fb) | (q - (1 << fb)), q)
    bits = np.where(normal & (e >= emax), emax << fb, bits)
    return ((sign << 15) | bits).astype(np.uint16)


def fma(a, b, c, fmt):
    """Correctly rounded a * b + c, element-wise on bit patterns."""
    eb, fb, bias = FORMATS[fmt]
    inf_bits = ((1 << eb) - 1) << fb
    a, b, c = np.broadcast_arrays(np.asarray(a, np.uint16), np.asarray(b, np.uint16),
                                  np.asarray(c, np.uint16))
    sa, Ma, Ea, na, ia = _fields(a, fmt)
    sb, Mb, Eb, nb, ib = _fields(b, fmt)
    sc, Mc, Ec, nc, ic = _fields(c, fmt)
    sp = sa ^ sb
    Mp = Ma * Mb
    Ep = Ea + Eb
    # finite part (specials overwritten below)
    Mp0 = np.where(ia | ib | na | nb, 0, Mp)
    Mc0 = np.where(ic | nc, 0, Mc)
    Ep0 = np.where(Mp0 == 0, Ec, Ep)                  # a zero term takes the other's exponent
    Ec0 = np.where(Mc0 == 0, Ep0, Ec)
    P = np.where(sp == 1, -Mp0, Mp0)
    C = np.where(sc == 1, -Mc0, Mc0)
    d = Ep0 - Ec0
    near = np.abs(d) <= GAP
    emin = np.minimum(Ep0, Ec0)
    dn = np.clip(d, -GAP, GAP)
    V_near = (P << np.clip(dn, 0, GAP)) + (C << np.clip(-dn, 0, GAP))
    # far apart: the larger-exponent term at 2^(GAP+1), the other as one unit
    p_big = d > 0
    big = np.where(p_big, P, C)
    small = np.where(p_big, C, P)
    V_far = (big << (GAP + 1)) + np.sign(small)
    e_far = np.where(p_big, Ep0, Ec0) - (GAP + 1)
    V = np.where(near, V_near, V_far)
    em = np.where(near, emin, e_far)
    zsign = ((Mp0 == 0) & (Mc0 == 0) & (sp == 1) & (sc == 1)).astype(np.int64)
    out = _round(V, em, zsign, fmt)
    # specials: NaN in; inf * 0; inf - inf; inf results
    zero_a = (Ma == 0) & ~ia & ~na
    zero_b = (Mb == 0) & ~ib & ~nb
    pinf = ia | ib
    nan = na | nb | nc | (ia & zero_b) | (ib & zero_a) | (pinf & ic & (sp != sc))
    out = np.where(pinf, ((sp << 15) | inf_bits).astype(np.uint16), out)
    out = np.where(~pinf & ic, ((sc << 15) | inf_bits).astype(np.uint16), out)
    return np.where(nan, np.uint16(NAN), out).astype(np.uint16)


def mul(a, b, fmt):
    """a * b rounded once (= a * b + (-0))."""
    return fma(a, b, np.uint16(0x8000), fmt)


def add(a, b, fmt):
    """a + b rounded once (= a * 1 + b)."""
    return fma(a, np.uint16(0x3C00 if fmt == "f16" else 0x3F80), b, fmt)

"""Exact rational model of FP16 / BF16, used to pin the oracle's arithmetic.

Written independently of ``oracle/tformat.py``: values are Python
``fractions.Fraction`` built from the bit fields, every operation is computed
exactly, and the rounding to the format is done on the exact rational with
integer arithmetic (round to nearest, ties to even, subnormals kept, overflow
to infinity).  Slow -- one element at a time -- and obviously correct.
"""
from __future__ import annotations

from fractions import Fraction

# name: (exponent bits, fraction bits, bias)
FORMATS = {"f16": (5, 10, 15), "bf16": (8, 7, 127)}
NAN = 0x7FFF


def fields(fmt):
    eb, fb, bias = FORMATS[fmt]
    return eb, fb, bias, (1 << eb) - 1


def decode(bits: int, fmt: str):
    """-> ('nan', None) | ('inf', sign) | ('num', Fraction, signbit)."""
    eb, fb, bias, emax = fields(fmt)
    s = bits >> 15
    e = (bits >> fb) & emax
    f = bits & ((1 << fb) - 1)
    if e == emax:
        return ("nan", None) if f else ("inf", s)
    if e == 0:
        v = Fraction(f, 1 << fb) * Fraction(2) ** (1 - bias)
    else:
        v = (1 + Fraction(f, 1 << fb)) * Fraction(2) ** (e - bias)
    return ("num", -v if s else v, s)


def encode(v: Fraction, signbit: int, fmt: str) -> int:
    """Round the exact rational ``v`` to the format (``signbit`` gives the
    sign of a zero result)."""
    eb, fb, bias, emax = fields(fmt)
    if v == 0:
        return signbit << 15
    s = 1 if v < 0 else 0
    a = -v if s else v
    # exponent k with 2^k <= a < 2^(k+1)
    k = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** k > a:
        k -= 1
    elif Fraction(2) ** (k + 1) <= a:
        k += 1
    k = max(k, 1 - bias)                       # subnormal range: fixed quantum
    quantum = Fraction(2) ** (k - fb)
    m = a / quantum
    q, r = divmod(m.numerator, m.denominator)
    twice = 2 * r
    if twice > m.denominator or (twice == m.denominator and q % 2 == 1):
        q += 1
    # q * quantum is the rounded magnitude
    if q == 0:
        return s << 15
    if q >= (1 << (fb + 1)):                   # carried into the next binade
        q >>= 1
        k += 1
    if q < (1 << fb):                          # subnormal
        return (s << 15) | q
    e = k + bias
    if e >= emax:
        return (s << 15) | (emax << fb)
    return (s << 15) | (e << fb) | (q - (1 << fb))


def fma(a: int, b: int, c: int, fmt: str) -> int:
    A, B, C = decode(a, fmt), decode(b, fmt), decode(c, fmt)
    if "nan" in (A[0], B[0], C[0]):
        return NAN
    if A[0] == "inf" or B[0] == "inf":
        other = B if A[0] == "inf" else A
        if other[0] == "num" and other[1] == 0:
            return NAN                         # inf * 0
        ps = (A[2] if A[0] == "num" else A[1]) ^ (B[2] if B[0] == "num" else B[1])
        if C[0] == "inf" and C[1] != ps:
            return NAN
        return (ps << 15) | (0x7C00 if fmt == "f16" else 0x7F80)
    if C[0] == "inf":
        return (C[1] << 15) | (0x7C00 if fmt == "f16" else 0x7F80)
    p = A[1] * B[1]
    psign = A[2] ^ B[2]
    v = p + C[1]
    if v == 0:
        # exact zero: -0 only if both addends are -0 (round to nearest)
        zsign = 1 if (p == 0 and C[1] == 0 and psign == 1 and C[2] == 1) else 0
        return encode(v, zsign, fmt)
    return encode(v, 0, fmt)


def mul(a: int, b: int, fmt: str) -> int:
    # a*b rounded once == a*b + (-0) rounded once
    return fma(a, b, 0x8000, fmt)


def add(a: int, b: int, fmt: str) -> int:
    one = 0x3C00 if fmt == "f16" else 0x3F80
    return fma(a, one, b, fmt)


def from_fraction(v: Fraction, fmt: str) -> int:
    return encode(v, 0, fmt)

"""Target-format (FP16 / BF16) arithmetic for the replay oracle.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py`` for who may import it.

Values travel as ``uint16`` bit patterns.  Each operation decodes its operands
to FP64 (exact for both formats), forms the exact result as an unevaluated
FP64 pair ``s + e`` (``s`` = the FP64 rounding of the exact result, ``e`` its
exact error), and rounds that pair once to the target format, to nearest with
ties to even, keeping subnormals and overflowing to infinity.  This is the
"one rounding per multiply-add" semantics of the packed FMA the paper deploys
("Fast Polynomial Transcendentals for LLMs", §3.2 and Fig. 2c; §3.4 names the
``__hfma2`` / ``fma.rn.bf16x2`` instructions).

Why the pair is enough: a product of two FP16 (11-bit) or BF16 (8-bit)
significands has at most 22 significant bits, so it is exact in FP64; the
TwoSum of that product and an addend gives ``s + e`` exactly.  Every midpoint
between two adjacent target-format values is itself an FP64 number, and
rounding to FP64 is monotone, so ``s`` lies on the same side of any midpoint
as the exact result, or on the midpoint itself -- and only then does the sign
of ``e`` decide.

NaN results are the canonical quiet NaN ``0x7FFF`` in both formats.
"""
from __future__ import annotations

import numpy as np

F16 = "f16"
BF16 = "bf16"

# (precision p incl. hidden bit, minimum normal exponent, largest finite value)
_FMT = {
    F16: (11, -14, 65504.0),
    BF16: (8, -126, float.fromhex("0x1.fep127")),
}

CANONICAL_NAN = np.uint16(0x7FFF)
SIGN = np.uint16(0x8000)
MAG = np.uint16(0x7FFF)


def _u16(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16)


def decode(bits, fmt: str) -> np.ndarray:
    """Target-format bit patterns -> exact FP64 values."""
    b = _u16(bits)
    with np.errstate(invalid="ignore"):        # signalling-NaN payloads
        if fmt == F16:
            return b.view(np.float16).astype(np.float64)
        if fmt == BF16:
            return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(fmt)


def is_nan(bits, fmt: str) -> np.ndarray:
    b = _u16(bits) & MAG
    return b > (np.uint16(0x7C00) if fmt == F16 else np.uint16(0x7F80))


def _encode_exact(mag: np.ndarray, fmt: str) -> np.ndarray:
    """Non-negative FP64 values that are exactly representable -> bits."""
    if fmt == F16:
        return mag.astype(np.float16).view(np.uint16)
    return (mag.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _two_sum(a: np.ndarray, b: np.ndarray):
    """Knuth's TwoSum: s = fl(a + b) and e with s + e == a + b exactly."""
    s = a + b
    bp = s - a
    ap = s - bp
    e = (a - ap) + (b - bp)
    return s, e


def round_pair(s, e, fmt: str) -> np.ndarray:
    """Round the exact value ``s + e`` (``s`` = its FP64 rounding) to ``fmt``.

    Round to nearest, ties to even; subnormals kept; magnitudes that round
    above the largest finite value become infinity; NaN becomes 0x7FFF.
    """
    p, emin, maxfin = _FMT[fmt]
    s = np.asarray(s, dtype=np.float64)
    e = np.asarray(e, dtype=np.float64)
    s, e = np.broadcast_arrays(s, e)
    out = np.zeros(s.shape, dtype=np.uint16)
    neg = np.signbit(s)
    nan = np.isnan(s)
    inf = np.isinf(s)
    fin = ~(nan | inf)

    a = np.where(fin, np.abs(s), 0.0)
    # error measured in the direction of growing magnitude
    e_mag = np.where(neg, -e, e)
    e_mag = np.where(fin, e_mag, 0.0)
    _, ex = np.frexp(a)                       # a = m * 2**ex, m in [0.5, 1)
    ulp_exp = np.maximum(ex - 1, emin) - (p - 1)
    q = np.ldexp(1.0, ulp_exp)                # spacing of the format at a
    k = a / q                                 # exact: power-of-two scaling
    kf = np.floor(k)
    frac = k - kf
    up = (frac > 0.5) | ((frac == 0.5) & (e_mag > 0)) | (
        (frac == 0.5) & (e_mag == 0) & (np.fmod(kf, 2.0) == 1.0))
    r = (kf + up) * q
    over = r > maxfin
    r = np.where(over, 0.0, r)
    mag_bits = _encode_exact(r, fmt)
    inf_bits = np.uint16(0x7C00) if fmt == F16 else np.uint16(0x7F80)
    mag_bits = np.where(over | inf, inf_bits, mag_bits)
    out = np.where(neg, mag_bits | SIGN, mag_bits).astype(np.uint16)
    out = np.where(nan, CANONICAL_NAN, out).astype(np.uint16)
    return out


def from_f64(x, fmt: str) -> np.ndarray:
    """Round FP64 values to the target format (RNE)."""
    x = np.asarray(x, dtype=np.float64)
    return round_pair(x, np.zeros_like(x), fmt)


def fma(a, b, c, fmt: str) -> np.ndarray:
    """a*b + c with a single rounding (the packed FMA)."""
    A, B, C = decode(a, fmt), decode(b, fmt), decode(c, fmt)
    with np.errstate(invalid="ignore", over="ignore"):
        p = A * B                              # exact for finite operands
        s, e = _two_sum(p, C)
    return round_pair(s, np.where(np.isfinite(s), e, 0.0), fmt)


def mul(a, b, fmt: str) -> np.ndarray:
    """a*b with a single rounding."""
    A, B = decode(a, fmt), decode(b, fmt)
    with np.errstate(invalid="ignore", over="ignore"):
        p = A * B
    return round_pair(p, np.zeros_like(p), fmt)


def add(a, b, fmt: str) -> np.ndarray:
    """a+b with a single rounding."""
    A, B = decode(a, fmt), decode(b, fmt)
    with np.errstate(invalid="ignore", over="ignore"):
        s, e = _two_sum(A, B)
    return round_pair(s, np.where(np.isfinite(s), e, 0.0), fmt)


def min_nan(a, b, fmt: str) -> np.ndarray:
    """Minimum that propagates NaN (canonical NaN out if either is NaN).

    Operands of opposite-signed zero never meet in the programs (the first
    operand is an absolute value and the second a positive clamp).
    """
    A, B = decode(a, fmt), decode(b, fmt)
    r = np.where(B < A, _u16(b), _u16(a))
    return np.where(is_nan(a, fmt) | is_nan(b, fmt), CANONICAL_NAN, r).astype(np.uint16)


def absval(a) -> np.ndarray:
    """Clear the sign bit (a bitwise operation; NaN payloads pass through)."""
    return (_u16(a) & MAG).astype(np.uint16)


def xorsign(v, x) -> np.ndarray:
    """Flip the sign of ``v`` where ``x`` is negative (sign-bit transfer)."""
    return (_u16(v) ^ (_u16(x) & SIGN)).astype(np.uint16)


def greater(a, b, fmt: str) -> np.ndarray:
    """Ordered a > b (False if either is NaN)."""
    return decode(a, fmt) > decode(b, fmt)


def all_patterns() -> np.ndarray:
    """Every 16-bit pattern in ascending order."""
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


def finite_mask(bits, fmt: str) -> np.ndarray:
    exp_all = np.uint16(0x7C00) if fmt == F16 else np.uint16(0x7F80)
    return (_u16(bits) & exp_all) != exp_all

"""Pins of the oracle's target-format arithmetic (oracle/tformat.py).

Against: (1) an independent exact-rational model (tests/exact_t.py) on
structured exhaustive domains and on random triples with every special value
mixed in; (2) a second exact model in scaled integers (tests/exact_int.py,
itself pinned to the rational one here), which is fast enough to check ten
million random triples per format and exhaustive rows of mul and add;
(3) library routines that are correctly rounded in special cases: numpy's
float64 -> float16 conversion, and float32 -> bfloat16 conversion of torch, on
products that are exact in the wider type.
"""
import numpy as np
import pytest
import torch

import exact_int as ei
import exact_t as ex
from oracle import tformat as tf

FMTS = ["f16", "bf16"]

SPECIALS = {
    "f16": [0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x0400, 0x7BFF, 0xFBFF,
            0x7C00, 0xFC00, 0x7E00, 0x7C01, 0xFFFF, 0x3C00, 0xBC00, 0x3800,
            0x3BFF, 0x3C01, 0x5BFF],
    "bf16": [0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x7F7F, 0xFF7F,
             0x7F80, 0xFF80, 0x7FC0, 0x7F81, 0xFFFF, 0x3F80, 0xBF80, 0x3F00,
             0x3F7F, 0x3F81, 0x5F7F],
}


def _rand_bits(rng, n, fmt):
    """Mix of uniform bit patterns, moderate values and special values."""
    b = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    # a third: values of moderate magnitude (exponent field near the bias)
    k = n // 3
    if fmt == "f16":
        mid = (rng.integers(0x2000, 0x5800, k)).astype(np.uint16)
    else:
        mid = (rng.integers(0x3800, 0x4300, k)).astype(np.uint16)
    mid |= (rng.integers(0, 2, k).astype(np.uint16) << 15)
    b[:k] = mid
    sp = np.array(SPECIALS[fmt], dtype=np.uint16)
    idx = rng.random(n) < 0.05
    b[idx] = sp[rng.integers(0, len(sp), idx.sum())]
    return b


def _same(a, b):
    return np.array_equal(np.asarray(a, np.uint16), np.asarray(b, np.uint16))


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_encode_roundtrip_exhaustive(fmt):
    x = tf.all_patterns()
    fin = tf.finite_mask(x, fmt)
    y = tf.from_f64(tf.decode(x, fmt), fmt)
    assert _same(y[fin], x[fin])
    assert _same(y[tf.is_nan(x, fmt)], np.full(int(tf.is_nan(x, fmt).sum()), 0x7FFF))


@pytest.mark.parametrize("fmt", FMTS)
def test_decode_matches_exact_fields(fmt):
    rng = np.random.default_rng(7)
    for b in rng.integers(0, 65536, 3000):
        d = ex.decode(int(b), fmt)
        v = float(tf.decode(np.uint16(b), fmt))
        if d[0] == "num":
            assert v == float(d[1]) and np.signbit(v) == bool(d[2])
        elif d[0] == "inf":
            assert np.isinf(v) and np.signbit(v) == bool(d[1])
        else:
            assert np.isnan(v)


@pytest.mark.parametrize("fmt", FMTS)
def test_fma_random_triples_vs_exact(fmt):
    rng = np.random.default_rng(11 if fmt == "f16" else 12)
    n = 60000
    a, b, c = (_rand_bits(rng, n, fmt) for _ in range(3))
    got = tf.fma(a, b, c, fmt)
    for i in range(n):
        want = ex.fma(int(a[i]), int(b[i]), int(c[i]), fmt)
        assert int(got[i]) == want, (hex(a[i]), hex(b[i]), hex(c[i]), hex(got[i]), hex(want))


@pytest.mark.parametrize("fmt", FMTS)
def test_fma_cancellation_and_far_addends(fmt):
    """Near-cancellation (result far below the operands) and addends far
    below the product's last bit -- the cases where a sticky bit decides."""
    rng = np.random.default_rng(5)
    rows = []
    for _ in range(20000):
        a = int(rng.integers(0, 65536)) & 0x7FFF
        b = int(rng.integers(0, 65536)) & 0x7FFF
        if not (tf.finite_mask(np.uint16(a), fmt) and tf.finite_mask(np.uint16(b), fmt)):
            continue
        p = float(tf.decode(np.uint16(a), fmt)) * float(tf.decode(np.uint16(b), fmt))
        c = int(tf.from_f64(-p, fmt))                      # cancels the product
        c2 = int(tf.from_f64(p * 2.0 ** -30, fmt))         # far below its last bit
        c3 = int(tf.from_f64(-p * 2.0 ** -12, fmt))
        rows += [(a, b, c), (a, b, c2), (a, b, c3)]
    a, b, c = (np.array(col, dtype=np.uint16) for col in zip(*rows))
    got = tf.fma(a, b, c, fmt)
    for i in range(len(rows)):
        assert int(got[i]) == ex.fma(int(a[i]), int(b[i]), int(c[i]), fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_mul_add_exhaustive_against_specials(fmt):
    """Every pattern times / plus every special value."""
    x = tf.all_patterns()[::7]
    for s in SPECIALS[fmt]:
        got_m = tf.mul(x, np.uint16(s), fmt)
        got_a = tf.add(x, np.uint16(s), fmt)
        for i in range(0, len(x), 13):
            assert int(got_m[i]) == ex.mul(int(x[i]), s, fmt)
            assert int(got_a[i]) == ex.add(int(x[i]), s, fmt)


def test_f16_mul_matches_numpy_conversion():
    """The product of two FP16 values is exact in FP64, and numpy's FP64 ->
    FP16 conversion is correctly rounded: a library pin for FP16 mul."""
    rng = np.random.default_rng(3)
    a = rng.integers(0, 65536, 1_000_000, dtype=np.uint32).astype(np.uint16)
    b = rng.integers(0, 65536, 1_000_000, dtype=np.uint32).astype(np.uint16)
    got = tf.mul(a, b, "f16")
    with np.errstate(all="ignore"):
        want = (a.view(np.float16).astype(np.float64) * b.view(np.float16).astype(np.float64)
                ).astype(np.float16).view(np.uint16)
    nan = np.isnan(want.view(np.float16))
    assert _same(got[~nan], want[~nan])
    assert np.all(got[nan] == 0x7FFF)


def test_bf16_mul_matches_torch_conversion():
    """BF16 products with exponents well inside the FP32 range are exact in
    FP32; torch's FP32 -> BF16 cast rounds to nearest-even."""
    rng = np.random.default_rng(4)
    n = 1_000_000
    e = rng.integers(0x30, 0x50, (2, n)).astype(np.uint16)
    m = rng.integers(0, 128, (2, n)).astype(np.uint16)
    s = rng.integers(0, 2, (2, n)).astype(np.uint16)
    bits = (s << 15) | (e << 7) | m
    a, b = bits[0], bits[1]
    got = tf.mul(a, b, "bf16")
    fa = torch.from_numpy((a.astype(np.uint32) << 16).view(np.float32))
    fb = torch.from_numpy((b.astype(np.uint32) << 16).view(np.float32))
    want = (fa * fb).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert _same(got, want)


@pytest.mark.parametrize("fmt", FMTS)
def test_ties_round_to_even(fmt):
    """Exact midpoints between neighbours round to the even neighbour."""
    one = tf.from_f64(1.0, fmt)
    p = 11 if fmt == "f16" else 8
    half_ulp = tf.from_f64(2.0 ** -p, fmt)               # 1 + half ulp(1) is a tie
    assert int(tf.add(one, half_ulp, fmt)) == int(one)   # 1.0 is even
    nxt = np.uint16(int(one) + 1)                        # 1 + ulp (odd)
    up = tf.add(nxt, half_ulp, fmt)
    assert int(up) == int(one) + 2                       # ties away from odd
    assert int(up) == ex.add(int(nxt), int(half_ulp), fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_min_nan(fmt):
    x = tf.all_patterns()
    lc = tf.from_f64(4.75, fmt)
    a = tf.absval(x)
    got = tf.min_nan(a, lc, fmt)
    nan = tf.is_nan(x, fmt)
    assert np.all(got[nan] == 0x7FFF)
    va = tf.decode(a[~nan], fmt)
    want = np.where(va < 4.75, a[~nan], lc)
    assert _same(got[~nan], want)


@pytest.mark.parametrize("fmt", FMTS)
def test_from_f64_vs_exact(fmt):
    from fractions import Fraction
    rng = np.random.default_rng(9)
    vals = np.concatenate([rng.normal(0, 3, 4000), rng.uniform(-1e5, 1e5, 1000),
                           rng.normal(0, 1e-6, 1000), rng.normal(0, 1e-40, 500),
                           np.array([65519.99, 65520.0, 65536.0, 3.3e38, 3.4e38, 1e39])])
    got = tf.from_f64(vals, fmt)
    for v, g in zip(vals, got):
        assert int(g) == ex.from_fraction(Fraction(float(v)), fmt), v


# ------------------------------------------------ the scaled-integer model

def _cancelling(rng, n, fmt):
    """Triples whose addend is within a few ulps of -a*b (heavy cancellation),
    with a and b of moderate magnitude."""
    lo, hi = (0x2000, 0x5800) if fmt == "f16" else (0x3800, 0x4300)
    a = rng.integers(lo, hi, n).astype(np.uint16) | (rng.integers(0, 2, n).astype(np.uint16) << 15)
    b = rng.integers(lo, hi, n).astype(np.uint16) | (rng.integers(0, 2, n).astype(np.uint16) << 15)
    p = ei.mul(a, b, fmt) ^ np.uint16(0x8000)
    c = (p.astype(np.int64) + rng.integers(-3, 4, n)).astype(np.uint16)
    return a, b, c


@pytest.mark.parametrize("fmt", FMTS)
def test_integer_model_matches_rationals(fmt):
    """The scaled-integer model agrees with the exact-rational model on mixed
    random triples (specials included) and on cancelling triples."""
    rng = np.random.default_rng(21 if fmt == "f16" else 22)
    n = 15000
    a, b, c = (_rand_bits(rng, n, fmt) for _ in range(3))
    a2, b2, c2 = _cancelling(rng, 5000, fmt)
    a, b, c = np.concatenate([a, a2]), np.concatenate([b, b2]), np.concatenate([c, c2])
    got = ei.fma(a, b, c, fmt)
    for i in range(a.size):
        assert int(got[i]) == ex.fma(int(a[i]), int(b[i]), int(c[i]), fmt), (
            hex(a[i]), hex(b[i]), hex(c[i]))


@pytest.mark.slow
@pytest.mark.parametrize("fmt", FMTS)
def test_fma_ten_million_triples(fmt):
    """10^7 triples per format: oracle fma, mul and add equal the exact
    integer model bit for bit.  Each block of 10^6 mixes uniform patterns,
    moderate magnitudes and specials (_rand_bits) or holds cancelling triples."""
    rng = np.random.default_rng(31 if fmt == "f16" else 32)
    block = 1_000_000
    for k in range(10):
        if k % 3 == 2:
            a, b, c = _cancelling(rng, block, fmt)
        else:
            a, b, c = (_rand_bits(rng, block, fmt) for _ in range(3))
        want = ei.fma(a, b, c, fmt)
        got = tf.fma(a, b, c, fmt)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, [(hex(a[i]), hex(b[i]), hex(c[i]), hex(got[i]), hex(want[i]))
                               for i in bad[:5]]
        if k < 4:
            assert _same(tf.mul(a, b, fmt), ei.mul(a, b, fmt))
            assert _same(tf.add(a, c, fmt), ei.add(a, c, fmt))


@pytest.mark.parametrize("fmt", FMTS)
def test_mul_add_exhaustive_rows(fmt):
    """Every pattern as the first operand against 48 second operands (the
    specials and random patterns): mul and add equal the integer model."""
    x = tf.all_patterns()
    rng = np.random.default_rng(41)
    ys = list(SPECIALS[fmt]) + [int(v) for v in rng.integers(0, 65536, 48 - len(SPECIALS[fmt]))]
    for y in ys:
        yy = np.uint16(y)
        assert _same(tf.mul(x, yy, fmt), ei.mul(x, yy, fmt)), hex(y)
        assert _same(tf.add(x, yy, fmt), ei.add(x, yy, fmt)), hex(y)


def test_integer_model_catches_double_rounding():
    """Must-fail control: an fma that rounds a*b + c in FP64 and then again to
    BF16 (a plausible oracle mistake) disagrees with the integer model on
    random BF16 triples, whose exponent range lets the FP64 sum be inexact.
    (For FP16 the same shortcut gives the correctly rounded result: with its
    narrow exponent range, whatever the FP64 sum drops lies far from every
    FP16 rounding boundary unless the result overflows.)"""
    rng = np.random.default_rng(51)
    a, b, c = (_rand_bits(rng, 200_000, "bf16") for _ in range(3))
    with np.errstate(all="ignore"):
        naive = tf.from_f64(tf.decode(a, "bf16") * tf.decode(b, "bf16") + tf.decode(c, "bf16"),
                            "bf16")
    assert np.count_nonzero(naive != ei.fma(a, b, c, "bf16")) > 0

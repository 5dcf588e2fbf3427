"""Pins of the exp2 fractional-core oracle (oracle/exp2.py) against the
printed parameters and Table 8 of Appendix B.1 (tests/golden/table8_exp2.txt),
exact endpoints, and FP64 2^x."""
import os

import numpy as np
import pytest

from oracle import exp2 as e2
from oracle import tformat as tf

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "table8_exp2.txt")


def rows():
    out = []
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            fam, obj, a, mx, rms = line.split()
            out.append((fam, obj, None if a == "-" else float(a), float(mx), float(rms)))
    return out


def _p(fam, obj, a):
    f = e2.grid()
    if fam == "D1":
        return 1.0 + f
    if fam == "D3":
        return e2.d3(f)
    return (e2.pwl2 if fam == "PWL2" else e2.d2)(a, f)


@pytest.mark.parametrize("row", rows())
def test_table8_errors(row):
    fam, obj, a, mx, rms = row
    got_mx, got_rms = e2.rel_stats(_p(fam, obj, a), e2.grid())
    assert abs(got_mx - mx) <= 0.0006 * mx and abs(got_rms - rms) <= 0.0006 * rms


@pytest.mark.parametrize("fam,obj,printed", [
    ("PWL2", "ls", e2.A_PWL2_LS), ("D2", "ls", e2.A_D2_LS),
    ("PWL2", "mm", e2.A_PWL2_MINIMAX), ("D2", "mm", e2.A_D2_MINIMAX)])
def test_parameters_reproduce(fam, obj, printed):
    family = e2.pwl2 if fam == "PWL2" else e2.d2
    a = e2.fit_least_squares(family) if obj == "ls" else e2.fit_minimax(family)
    # least squares has a closed form; the minimax optimum is flat to ~1e-9
    assert abs(a - printed) <= (5e-11 if obj == "ls" else 2e-8)


def test_fa4_d3_endpoint_printed():
    assert round(sum(e2.FA4_D3), 5) == 1.99983


def test_fp16_pwl2_coefficients_and_error():
    a, b = e2.f16_coefficients("PWL2")
    assert float(tf.decode(np.uint16(a), "f16")) == 0.7978515625
    assert float(tf.decode(np.uint16(b), "f16")) == 0.40380859375
    # endpoints exact after target-precision rounding
    h = tf.from_f64(np.array([0.0, 1.0]), "f16")
    p = tf.decode(e2.core_f16("PWL2", h), "f16")
    assert p[0] == 1.0 and p[1] == 2.0
    # the printed maximum relative error of the rounded FP16 core, 1.132e-2
    hh = np.arange(0x0000, 0x3C01, dtype=np.uint16)           # every FP16 in [0, 1]
    fv = tf.decode(hh, "f16")
    mx, _ = e2.rel_stats(tf.decode(e2.core_f16("PWL2", hh), "f16"), fv)
    assert abs(mx - 1.132e-2) <= 0.02 * 1.132e-2


@pytest.mark.parametrize("variant", e2.VARIANTS)
def test_endpoints_and_reconstruction(variant):
    """p(0) = 1 exactly; 2^n for integer x exactly; 2^x within the core's
    error plus the FP16 rounding of f; specials."""
    n = np.arange(-126, 128, dtype=np.float32)
    y = e2.exp2_replay(variant, n).view(np.float32)
    assert np.array_equal(y, np.exp2(n.astype(np.float64)).astype(np.float32))
    rng = np.random.default_rng(3)
    x = rng.uniform(-120, 120, 200_000).astype(np.float32)
    y = e2.exp2_replay(variant, x).view(np.float32).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1)
    core = {"D1": 6.2e-2, "PWL2": 1.2e-2, "D2": 3.5e-3, "D3": 1.5e-3}[variant]
    assert rel.max() <= core
    sp = np.array([np.nan, np.inf, -np.inf, 200.0, -200.0, 0.0, -0.0], dtype=np.float32)
    y = e2.exp2_replay(variant, sp)
    assert y[0] == 0x7FFFFFFF and y[1] == 0x7F800000 and y[3] == 0x7F800000
    assert y[2] == y[4] == np.float32(2.0 ** -126).view(np.uint32)
    assert y[5] == y[6] == 0x3F800000

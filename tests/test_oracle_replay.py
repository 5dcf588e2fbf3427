"""Pins of the oracle's program replay (oracle/replay.py).

Against: the exact symmetry of each reduction (§3.1, Fig. 1: odd, even,
centred-odd, x/2 + even), the endpoint values the reductions fix exactly
(P(0) = f(0), eq. 3 and eq. 7), the clamp of eq. 2, the exact tail, the
error against the FP64 functions (a dropped sign, a wrong index or a swapped
operand sends it far past the stated bound), an element-by-element replay in
exact rational arithmetic, and library polynomial evaluation for the
real-arithmetic metric.  Two must-fail controls show the checks can fail.
"""
import zlib
from fractions import Fraction

import numpy as np
import pytest
from numpy.polynomial import polynomial as npoly

import exact_t as ex
import golden_programs as gp
from oracle import reference as ref
from oracle import tformat as tf
from oracle.replay import backward, evaluate, evaluate_real, forward, swiglu_backward, swiglu_forward

PROGS = gp.load()
KEYS = sorted(PROGS)
X = tf.all_patterns()


def _neg(x):
    return (x ^ np.uint16(0x8000)).astype(np.uint16)


@pytest.mark.parametrize("k", KEYS)
def test_symmetry_exact(k):
    p = PROGS[k]
    y, yn = forward(p, X), forward(p, _neg(X))
    nan = tf.is_nan(X, p.fmt)
    if p.form == "E":
        assert np.array_equal(y, yn)
    elif p.form == "O":
        assert np.array_equal(y[~nan], yn[~nan] ^ np.uint16(0x8000))
    elif p.form == "CO":
        # y(x) + y(-x) = 1 up to the two final roundings (one ulp of 1/2..1)
        s = tf.decode(y[~nan], p.fmt) + tf.decode(yn[~nan], p.fmt)
        ulp1 = 2.0 ** (-10 if p.fmt == "f16" else -7)
        assert np.max(np.abs(s - 1.0)) <= ulp1
    else:  # HX: s(x) - s(-x) = x (eq. 4) up to roundings, inside the clamp
        fin = tf.finite_mask(X, p.fmt)
        xv = tf.decode(X, p.fmt)
        inside = fin & (np.abs(xv) <= p.lc)
        d = tf.decode(y[inside], p.fmt) - tf.decode(yn[inside], p.fmt) - xv[inside]
        assert np.max(np.abs(d)) <= 2 * p.info["stated_max_abs_err"] + 2.0 ** -8 * p.lc


@pytest.mark.parametrize("k", KEYS)
def test_endpoints_and_specials(k):
    p = PROGS[k]
    fmt = p.fmt
    half = int(tf.from_f64(0.5, fmt))
    pz, nz = np.uint16(0), np.uint16(0x8000)
    inf = np.uint16(0x7C00 if fmt == "f16" else 0x7F80)
    y0, yn0 = int(forward(p, pz)), int(forward(p, nz))
    if p.form == "CO":
        assert y0 == half and yn0 == half
    elif p.form == "O":
        assert y0 == 0 and yn0 == 0x8000                 # tanh(+-0) = +-0
    elif p.form == "E":
        assert y0 == yn0 == p.coef[0] == int(tf.from_f64(ref.residual_at_zero(p.fn, p.direction), fmt))
    else:
        assert float(tf.decode(y0, fmt)) == 0.0 and float(tf.decode(yn0, fmt)) == 0.0
    # NaN in -> canonical NaN out
    nans = X[tf.is_nan(X, fmt)]
    assert np.all(forward(p, nans) == 0x7FFF)
    # clamp (eq. 2): for |x| >= Lc the clamp forms see t = Lc
    xv = tf.decode(X, fmt)
    big = (np.abs(xv) >= p.lc) & ~tf.is_nan(X, fmt)
    if p.form in ("CO", "O", "E"):
        lcx = np.where(np.signbit(xv[big]), p.lc_bits | 0x8000, p.lc_bits).astype(np.uint16)
        assert np.array_equal(forward(p, X[big]), forward(p, lcx))
    else:  # exact tail: max(x, +0) beyond the clamp, +-inf included
        tail = (np.abs(xv) > p.lc) & ~tf.is_nan(X, fmt)
        yt = forward(p, X[tail])
        want = np.where(xv[tail] > 0, X[tail], np.uint16(0))
        assert np.array_equal(yt, want)
        assert int(forward(p, inf)) == int(inf) and int(forward(p, inf | 0x8000)) == 0


@pytest.mark.parametrize("k", KEYS)
def test_error_within_stated_bound(k):
    p = PROGS[k]
    fin = tf.finite_mask(X, p.fmt)
    x = X[fin]
    y = tf.decode(forward(p, x), p.fmt)
    err = np.abs(y - ref.function(p.fn, p.direction)(tf.decode(x, p.fmt)))
    assert np.all(np.isfinite(y))
    assert err.max() == pytest.approx(p.info["stated_max_abs_err"], rel=0, abs=0)
    assert err.max() < 0.05     # a sign, index or operand mistake lands near 0.5 or worse


def _exact_program(p, xbits):
    """Element-by-element replay in exact rational arithmetic (tests/exact_t),
    written from the reductions of §3.1 / §3.3."""
    fmt = p.fmt
    out = []
    half = ex.from_fraction(Fraction(1, 2), fmt)
    for xb in xbits:
        xb = int(xb)
        a = xb & 0x7FFF
        da, dl = ex.decode(a, fmt), ex.decode(p.lc_bits, fmt)
        if da[0] == "nan":
            out.append(0x7FFF)
            continue
        t = p.lc_bits if (da[0] == "inf" or da[1] > dl[1]) else a
        last = 0 if p.form == "E" else 1
        v = p.coef[p.degree]
        for j in range(p.degree - 1, last - 1, -1):
            v = ex.fma(v, t, p.coef[j], fmt)
        sgn = xb & 0x8000
        if p.form == "E":
            y = v
        elif p.form == "CO":
            y = ex.fma(v ^ sgn, t, half, fmt)
        elif p.form == "O":
            y = ex.mul(v ^ sgn, t, fmt)
        else:
            y = ex.fma(v, t, ex.mul(xb, half, fmt), fmt)
            dx = ex.decode(xb, fmt)
            mag = da[1] if da[0] == "num" else None
            if da[0] == "inf" or mag > dl[1]:
                positive = (dx[0] == "inf" and dx[1] == 0) or (dx[0] == "num" and dx[1] > 0)
                y = xb if positive else 0
        out.append(y)
    return np.array(out, dtype=np.uint16)


@pytest.mark.parametrize("k", KEYS)
def test_replay_vs_exact_rationals(k):
    p = PROGS[k]
    rng = np.random.default_rng(zlib.crc32(k.encode()))
    xs = np.concatenate([rng.integers(0, 65536, 400, dtype=np.uint32).astype(np.uint16),
                         tf.from_f64(rng.normal(0, 3, 400), p.fmt),
                         np.array([0, 0x8000, 0x7FFF, 0xFFFF], dtype=np.uint16),
                         np.array([p.lc_bits, p.lc_bits | 0x8000, p.lc_bits + 1, p.lc_bits - 1],
                                  dtype=np.uint16)])
    assert np.array_equal(forward(p, xs), _exact_program(p, xs))


@pytest.mark.parametrize("k", KEYS)
def test_backward_and_swiglu_products(k):
    p = PROGS[k]
    rng = np.random.default_rng(1)
    x = tf.from_f64(rng.normal(0, 3, 3000), p.fmt)
    dy = tf.from_f64(rng.normal(0, 1, 3000), p.fmt)
    y = forward(p, x)
    dx = backward(p, x, dy)
    for i in range(0, 3000, 7):
        assert int(dx[i]) == ex.mul(int(dy[i]), int(y[i]), p.fmt)
    if p.fn == ref.SILU and p.direction == ref.FWD:
        d = PROGS[gp.key(ref.SILU, ref.BWD, p.fmt, 4)]
        u = tf.from_f64(rng.normal(0, 2, 3000), p.fmt)
        yy = swiglu_forward(p, x, u)
        dg, du = swiglu_backward(p, d, x, u, dy)
        sp = forward(d, x)
        for i in range(0, 3000, 7):
            assert int(yy[i]) == ex.mul(int(y[i]), int(u[i]), p.fmt)
            assert int(du[i]) == ex.mul(int(dy[i]), int(y[i]), p.fmt)
            assert int(dg[i]) == ex.mul(ex.mul(int(dy[i]), int(u[i]), p.fmt), int(sp[i]), p.fmt)


@pytest.mark.parametrize("k", KEYS)
def test_real_replay_matches_numpy_polyval(k):
    p = PROGS[k]
    c = p.coef_values()
    x = np.linspace(-p.lc, p.lc, 2001)
    t = np.abs(x)
    poly = npoly.polyval(t, c)
    want = {"E": poly, "CO": 0.5 + np.sign(x) * poly, "O": np.sign(x) * poly,
            "HX": 0.5 * x + poly}[p.form]
    got = evaluate_real(p.form, c, p.lc, x)
    assert np.max(np.abs(got - want)) <= 1e-13


def test_must_fail_perturbed_coefficient():
    """A program with one coefficient moved by one ulp must not replay equal
    to the original: the parity comparison can fail."""
    p = PROGS["sigmoid.fwd.bf16.D3"]
    bad = list(p.coef)
    bad[2] += 1
    y = forward(p, X)
    yb = evaluate(p.form, tuple(bad), p.lc_bits, X, p.fmt)
    assert not np.array_equal(y, yb)


def test_must_fail_coarsened_program():
    """Coefficients coarsened to 16 levels must break the stated bound."""
    p = PROGS["sigmoid.fwd.bf16.D3"]
    c = p.coef_values()
    coarse = tf.from_f64(np.round(c * 16) / 16, p.fmt)
    fin = tf.finite_mask(X, p.fmt)
    y = tf.decode(evaluate(p.form, tuple(coarse), p.lc_bits, X[fin], p.fmt), p.fmt)
    err = np.max(np.abs(y - ref.sigmoid(tf.decode(X[fin], p.fmt))))
    assert err > p.info["stated_max_abs_err"]


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_swiglu_sigmoid_rule_vs_exact_and_fp64(fmt):
    """The deployed B1/B4 rule (s = g p, s' = p + g p (1 - p)) element by
    element in exact rationals, and its error against the FP64 SiLU and SiLU'
    within the bound the sigmoid program's own error implies."""
    from oracle.replay import swiglu_sigmoid_backward, swiglu_sigmoid_forward
    sig = PROGS[gp.key(ref.SIGMOID, ref.FWD, fmt, 3)]
    rng = np.random.default_rng(17)
    g = tf.from_f64(rng.normal(0, 3, 4000), fmt)
    u = tf.from_f64(rng.normal(0, 1, 4000), fmt)
    dy = tf.from_f64(rng.normal(0, 1, 4000), fmt)
    one = int(tf.from_f64(1.0, fmt))
    y = swiglu_sigmoid_forward(sig, g, u)
    dg, du = swiglu_sigmoid_backward(sig, g, u, dy)
    p = forward(sig, g)
    for i in range(0, 4000, 9):
        pi, gi = int(p[i]), int(g[i])
        s = ex.mul(gi, pi, fmt)
        assert int(y[i]) == ex.mul(s, int(u[i]), fmt)
        q = ex.fma(pi ^ 0x8000, pi, pi, fmt)
        sd = ex.fma(gi, q, pi, fmt)
        assert int(du[i]) == ex.mul(int(dy[i]), s, fmt)
        assert int(dg[i]) == ex.mul(ex.mul(int(dy[i]), int(u[i]), fmt), sd, fmt)
    # error of s = g p and s' against FP64, with u = dy = 1
    x = X[tf.finite_mask(X, fmt)]
    xv = tf.decode(x, fmt)
    x, xv = x[np.abs(xv) < 64], xv[np.abs(xv) < 64]
    ones = np.full(x.size, one, np.uint16)
    s = tf.decode(swiglu_sigmoid_forward(sig, x, ones), fmt)
    sd = tf.decode(swiglu_sigmoid_backward(sig, x, ones, ones)[0], fmt)
    e_p = sig.info["stated_max_abs_err"]
    ulp = 2.0 ** (-10 if fmt == "f16" else -7)
    assert np.all(np.abs(s - ref.silu(xv)) <= np.abs(xv) * (e_p + ulp) + ulp)
    # s' = p + x p (1 - p): |d s'| <= e_p (1 + |x| |1 - 2p|) + rounding
    bound = e_p * (1 + np.abs(xv)) + 4 * ulp * (1 + np.abs(xv))
    assert np.all(np.abs(sd - ref.dsilu(xv)) <= bound)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("fn", [ref.TANH, ref.SIGMOID])
def test_derived_program_is_the_polynomial_derivative(fmt, fn):
    """The differentiated program's coefficients are the derivative of the
    forward polynomial (numpy polyder) rounded once; multiples by powers of
    two are exact; in real arithmetic the two agree to the coefficient
    rounding."""
    from oracle.replay import derive
    D = 4 if fn == ref.TANH else 3
    p = PROGS[gp.key(fn, ref.FWD, fmt, D)]
    d = derive(p)
    assert d.form == "E" and d.degree == D - 1 and d.lc_bits == p.lc_bits
    c = p.coef_values()
    e = d.coef_values()
    want = npoly.polyder(c)                        # c_1 + 2 c_2 t + ... (c_0 = 0)
    assert e[0] == want[0] and e[1] == want[1]     # 1 x c_1 and 2 x c_2: exact
    if D >= 4:
        assert e[3] == want[3]                     # 4 x c_4: exact
    ulp = 2.0 ** (-10 if fmt == "f16" else -7)
    assert np.all(np.abs(e - want) <= np.abs(want) * ulp / 2 + 1e-30)
    t = np.linspace(0, p.lc, 501)
    assert np.max(np.abs(npoly.polyval(t, e) - npoly.polyval(t, want))) <= \
        np.sum(np.abs(want) * ulp / 2 * p.lc ** np.arange(D))
    # it approximates the true derivative, but worse than the direct
    # derivative fit: "backward has its own error profile" (Appendix D,
    # item 2; §5.1 on the backward sweeps)
    f = ref.function(fn, ref.BWD)
    x = X[tf.finite_mask(X, fmt)]
    y = tf.decode(forward(d, x), fmt)
    err = np.max(np.abs(y - f(tf.decode(x, fmt))))
    direct = PROGS[gp.key(fn, ref.BWD, fmt, 4)]
    assert direct.info["stated_max_abs_err"] < err < 0.15


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_softcap_alpha_one_is_the_tanh_program(fmt):
    from oracle.replay import softcap_forward
    p = PROGS[gp.key(ref.TANH, ref.FWD, fmt, 4)]
    assert np.array_equal(softcap_forward(p, 1.0, X), forward(p, X))


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("alpha", [30.0, 50.0, 2.5])
def test_softcap_symmetry_error_and_products(fmt, alpha):
    """softcap is odd and its derivative even, bit for bit; the error against
    FP64 alpha tanh(x / alpha) stays within alpha times the tanh program's
    bound plus the two scalings' roundings; each product rounds once."""
    from oracle.replay import softcap_backward, softcap_consts, softcap_forward
    p = PROGS[gp.key(ref.TANH, ref.FWD, fmt, 4)]
    dp = PROGS[gp.key(ref.TANH, ref.BWD, fmt, 4)]
    y, yn = softcap_forward(p, alpha, X), softcap_forward(p, alpha, _neg(X))
    nan = tf.is_nan(X, fmt)
    assert np.array_equal(y[~nan], yn[~nan] ^ np.uint16(0x8000))
    ones = np.full(X.size, int(tf.from_f64(1.0, fmt)), np.uint16)
    d, dn = softcap_backward(dp, alpha, X, ones), softcap_backward(dp, alpha, _neg(X), ones)
    assert np.array_equal(d, dn)
    a, ia = softcap_consts(alpha, fmt)
    av, iav = float(tf.decode(np.uint16(a), fmt)), float(tf.decode(np.uint16(ia), fmt))
    fin = tf.finite_mask(X, fmt) & (np.abs(tf.decode(X, fmt)) < 1e4)
    xv = tf.decode(X[fin], fmt)
    z = tf.decode(tf.mul(X[fin], np.uint16(ia), fmt), fmt)
    yv = tf.decode(y[fin], fmt)
    ulp = 2.0 ** (-10 if fmt == "f16" else -7)
    bound = (av * p.info["stated_max_abs_err"] + av * np.abs(z - xv / alpha) + abs(av - alpha)
             + ulp * np.abs(yv))
    assert np.all(np.abs(yv - alpha * np.tanh(xv / alpha)) <= bound + 1e-12)
    rng = np.random.default_rng(23)
    xs = tf.from_f64(rng.normal(0, alpha, 500), fmt)
    dys = tf.from_f64(rng.normal(0, 1, 500), fmt)
    ys = softcap_forward(p, alpha, xs)
    ds = softcap_backward(dp, alpha, xs, dys)
    zs = tf.mul(xs, np.uint16(ia), fmt)
    th, dth = forward(p, zs), forward(dp, zs)
    for i in range(500):
        assert int(zs[i]) == ex.mul(int(xs[i]), ia, fmt)
        assert int(ys[i]) == ex.mul(a, int(th[i]), fmt)
        assert int(ds[i]) == ex.mul(int(dys[i]), int(dth[i]), fmt)

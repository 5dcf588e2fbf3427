"""Pins of the oracle's FP64 reference functions (oracle/reference.py).

Against mpmath at 50 digits (independent arbitrary-precision evaluation) and
against exact identities: sigma(-x) = 1 - sigma(x) and Phi(-x) = 1 - Phi(x)
(§3.1), s(x) - s(-x) = x (eq. 4), s'(x) + s'(-x) = 1 (eq. 9),
sigma' = sigma (1 - sigma) (eq. 10), tanh' = 1 - tanh^2 (eq. 11).
"""
import numpy as np
import pytest

from oracle import reference as ref

mp = pytest.importorskip("mpmath")
mp.mp.dps = 50

GRID = np.concatenate([np.linspace(-30, 30, 241), [1e-8, -1e-8, 1e-3, -2.5e-3, 0.0, 44.0, -44.0]])


def _mp_funcs():
    sig = lambda x: 1 / (1 + mp.exp(-x))
    Phi = lambda x: mp.ncdf(x)
    phi = lambda x: mp.npdf(x)
    return {
        (ref.SIGMOID, ref.FWD): sig,
        (ref.TANH, ref.FWD): mp.tanh,
        (ref.SILU, ref.FWD): lambda x: x * sig(x),
        (ref.GELU, ref.FWD): lambda x: x * Phi(x),
        (ref.SIGMOID, ref.BWD): lambda x: sig(x) * (1 - sig(x)),
        (ref.TANH, ref.BWD): lambda x: 1 - mp.tanh(x) ** 2,
        (ref.SILU, ref.BWD): lambda x: sig(x) + x * sig(x) * (1 - sig(x)),
        (ref.GELU, ref.BWD): lambda x: Phi(x) + x * phi(x),
    }


@pytest.mark.parametrize("key", list(_mp_funcs().keys()))
def test_functions_vs_mpmath(key):
    f = ref.function(*key)
    g = _mp_funcs()[key]
    got = f(GRID)
    for x, y in zip(GRID, got):
        want = float(g(mp.mpf(float(x))))
        # a few FP64 ulps relative, and an absolute floor (cancellation in s', GELU')
        # far below any FP16 / BF16 ulp of the outputs
        assert abs(y - want) <= 2e-15 * abs(want) + 1e-16, (key, x, y, want)


@pytest.mark.parametrize("fn", [ref.SIGMOID, ref.TANH, ref.SILU, ref.GELU])
@pytest.mark.parametrize("d", [ref.FWD, ref.BWD])
def test_residuals_vs_mpmath(fn, d):
    """The half-domain residual the fitter targets (§3.1, §3.3)."""
    g = _mp_funcs()[(fn, d)]
    form = ref.form_of(fn, d)
    r = ref.residual(fn, d)
    t = np.linspace(0, 12, 97)
    for ti, yi in zip(t, r(t)):
        x = mp.mpf(float(ti))
        full = g(x)
        want = {"CO": full - mp.mpf(1) / 2, "O": full, "E": full, "HX": full - x / 2}[form]
        assert abs(yi - float(want)) <= 1e-15 * max(1.0, abs(float(want)))
    assert float(r(np.array([0.0]))[0]) == ref.residual_at_zero(fn, d)


def test_identities():
    x = np.linspace(-20, 20, 4001)
    assert np.max(np.abs(ref.sigmoid(-x) - (1 - ref.sigmoid(x)))) <= 2.3e-16
    assert np.max(np.abs(ref.Phi(-x) - (1 - ref.Phi(x)))) <= 2.3e-16
    assert np.max(np.abs(ref.silu(x) - ref.silu(-x) - x)) <= 2 * np.spacing(20.0)
    assert np.max(np.abs(ref.gelu(x) - ref.gelu(-x) - x)) <= 2 * np.spacing(20.0)
    assert np.max(np.abs(ref.dsilu(x) + ref.dsilu(-x) - 1)) <= 1e-14
    assert np.max(np.abs(ref.dgelu(x) + ref.dgelu(-x) - 1)) <= 1e-14
    s = ref.sigmoid(x)
    assert np.max(np.abs(ref.dsigmoid(x) - s * (1 - s))) <= 2e-16
    assert np.max(np.abs(ref.dtanh(x) - (1 - np.tanh(x) ** 2))) <= 4e-16


def test_forms_follow_section_3():
    """Which reduction each (function, direction) uses (§3.1, §3.3)."""
    assert ref.form_of(ref.SIGMOID, ref.FWD) == "CO"
    assert ref.form_of(ref.TANH, ref.FWD) == "O"
    assert ref.form_of(ref.SILU, ref.FWD) == "HX"
    assert ref.form_of(ref.GELU, ref.FWD) == "HX"
    assert ref.form_of(ref.SIGMOID, ref.BWD) == "E"
    assert ref.form_of(ref.TANH, ref.BWD) == "E"
    assert ref.form_of(ref.SILU, ref.BWD) == "CO"
    assert ref.form_of(ref.GELU, ref.BWD) == "CO"

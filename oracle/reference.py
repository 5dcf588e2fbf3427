"""FP64 reference functions and the reduced residuals that the fitter targets.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

Citations are to "Fast Polynomial Transcendentals for LLMs" (arXiv 2610.00049).

Functions (all FP64, numerically stable for every finite input):

* sigmoid  sigma(x) = 1 / (1 + e^-x)
* tanh
* SiLU     s(x) = x sigma(x)
* GELU     x Phi(x), Phi the standard normal CDF ("exact GELU", §3.1)
* derivatives sigma' = sigma(x) sigma(-x) (eq. 10 rewritten without the
  cancellation of 1 - sigma), tanh' = 1 / cosh^2 (eq. 11),
  s'(x) = sigma(x) + x sigma'(x) (eq. 9), GELU'(x) = Phi(x) + x phi(x).

Reduced residuals on the half domain t >= 0 (§3.1 eq. 3-6, §3.3):

* centred-odd  ("CO"): sigma(t) - 1/2, s'(t) - 1/2, GELU'(t) - 1/2
* odd          ("O") : tanh t
* even         ("E") : sigma'(t), tanh'(t)
* x/2 + even   ("HX"): s(t) - t/2 = t (sigma(t) - 1/2), GELU(t) - t/2
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erfc

SIGMOID, TANH, SILU, GELU = 0, 1, 2, 3
FWD, BWD = 0, 1
FN_NAMES = {SIGMOID: "sigmoid", TANH: "tanh", SILU: "silu", GELU: "gelu"}

# Program forms (§3.1, §3.3)
CO, O, E, HX = "CO", "O", "E", "HX"


def form_of(fn: int, direction: int) -> str:
    """Reduction form for each (function, direction), §3.1 and §3.3."""
    if direction == FWD:
        return {SIGMOID: CO, TANH: O, SILU: HX, GELU: HX}[fn]
    return {SIGMOID: E, TANH: E, SILU: CO, GELU: CO}[fn]


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        z = np.exp(-np.abs(x))
        pos = 1.0 / (1.0 + z)
        return np.where(x >= 0, pos, z / (1.0 + z))


def tanh(x):
    return np.tanh(np.asarray(x, dtype=np.float64))


def Phi(x):
    """Standard normal CDF via the complementary error function."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * erfc(-x / math.sqrt(2.0))


def phi(x):
    x = np.asarray(x, dtype=np.float64)
    return np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def gelu(x):
    x = np.asarray(x, dtype=np.float64)
    return x * Phi(x)


def dsigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return sigmoid(x) * sigmoid(-x)


def dtanh(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        c = np.cosh(x)
        return 1.0 / (c * c)


def dsilu(x):
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        return sigmoid(x) + x * dsigmoid(x)


def dgelu(x):
    x = np.asarray(x, dtype=np.float64)
    return Phi(x) + x * phi(x)


def function(fn: int, direction: int):
    """The true function a program approximates (forward value or derivative)."""
    if direction == FWD:
        return {SIGMOID: sigmoid, TANH: tanh, SILU: silu, GELU: gelu}[fn]
    return {SIGMOID: dsigmoid, TANH: dtanh, SILU: dsilu, GELU: dgelu}[fn]


def residual(fn: int, direction: int):
    """The reduced half-domain target f(t), t >= 0, that the polynomial fits."""
    form = form_of(fn, direction)
    f = function(fn, direction)
    if form == CO:
        return lambda t: f(t) - 0.5
    if form == O or form == E:
        return f
    if fn == SILU:                    # HX: t (sigma(t) - 1/2), eq. 5
        return lambda t: np.asarray(t, dtype=np.float64) * (sigmoid(t) - 0.5)
    return lambda t: np.asarray(t, dtype=np.float64) * (Phi(t) - 0.5)


def residual_at_zero(fn: int, direction: int) -> float:
    """f(0) of the reduced target: 0 for CO/O/HX, 1/4 for sigma', 1 for tanh'."""
    form = form_of(fn, direction)
    if form != E:
        return 0.0
    return 0.25 if fn == SIGMOID else 1.0


def value_range(fn: int, direction: int):
    """Range [lo, hi] that the output of a program must respect, or None.

    The range gate (one of the "shape or boundary" checks of §3.2 step 6)
    applies where the true range has exactly representable bounds: sigmoid in
    [0, 1], tanh in [-1, 1], sigma' in [0, 1/4], tanh' in [0, 1].  SiLU, GELU
    and their derivatives have irrational extrema and get no range gate.
    """
    if direction == FWD:
        return {SIGMOID: (0.0, 1.0), TANH: (-1.0, 1.0)}.get(fn)
    return {SIGMOID: (0.0, 0.25), TANH: (0.0, 1.0)}.get(fn)


def monotone_on_half(fn: int, direction: int) -> int:
    """+1 / -1 if the true function is non-decreasing / non-increasing on
    [0, inf), 0 if it is neither (the monotonicity gate of §3.2 step 7 applies
    to the first two kinds only)."""
    if direction == FWD:
        return 1                      # sigmoid, tanh, SiLU, GELU all rise on t >= 0
    if fn in (SIGMOID, TANH):
        return -1                     # sigma', tanh' fall on t >= 0
    return 0                          # s', GELU' overshoot 1 and come back

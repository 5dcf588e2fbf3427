"""Replay of the polynomial programs, element by element, in three orders.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

Citations are to "Fast Polynomial Transcendentals for LLMs" (arXiv 2610.00049).

A program is the reduction form (§3.1, §3.3), the coefficients c_0..c_D rounded
to the target format T (§3.2 step 3), and the runtime clamp Lc (§3.2, eq. 2).
With t = min(|x|, Lc) (eq. 2) and the Horner value v of the polynomial in t:

  CO  centred-odd  y = 1/2 + sign(x) * t * (c_1 + c_2 t + ... + c_D t^(D-1))  (eq. 3)
  O   odd          y =       sign(x) * t * (c_1 + ...          + c_D t^(D-1))
  E   even         y = c_0 + c_1 t + ... + c_D t^D
  HX  x/2 + even   y = x/2 + t * (c_1 + ... + c_D t^(D-1))  for |x| <= Lc   (eq. 6)
                   y = max(x, +0)                           for |x| >  Lc

Deployed order ("fused"): every Horner stage is one packed FMA with one
rounding; the sign is transferred bitwise onto v; the final stage is one more
FMA that folds in 1/2 (CO) or x/2 (HX), or a multiply by t (O).  The fitter's
search emulator ("split", §3.2 step 4) rounds each multiply and each add
separately in the same order.  The Table 2 metric ("real") evaluates the
rounded coefficients without any intermediate rounding (§4.1).

The backward product of a derivative program is dx = dy * y rounded once; the
SwiGLU gate (eq. 15) is y = s(g) * u and its backward dg = (dy * u) * s'(g),
du = dy * s(g), each product rounded once.  The paper's deployed B1/B4 rule
instead recomputes the sigmoid program p and forms s = g p and
s' = p + g p (1 - p) (§3.3 "Forward and backward programs", §5.2.4).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import tformat as tf
from .reference import CO, E, HX, O, form_of


@dataclass
class Program:
    fn: int
    direction: int
    fmt: str
    degree: int
    li: float
    lc: float
    coef: tuple          # c_0 .. c_D as target-format bit patterns
    lc_bits: int
    info: dict = field(default_factory=dict)

    @property
    def form(self) -> str:
        return form_of(self.fn, self.direction)

    def coef_values(self) -> np.ndarray:
        return tf.decode(np.array(self.coef, dtype=np.uint16), self.fmt)


def _half(fmt):
    return tf.from_f64(0.5, fmt)


def _horner(coef, t, last, fmt, fused):
    """v = c_D; v = v*t + c_j for j = D-1 .. last."""
    D = len(coef) - 1
    v = np.broadcast_to(np.uint16(coef[D]), np.shape(t)).astype(np.uint16)
    for j in range(D - 1, last - 1, -1):
        cj = np.uint16(coef[j])
        if fused:
            v = tf.fma(v, t, cj, fmt)
        else:
            v = tf.add(tf.mul(v, t, fmt), cj, fmt)
    return v


def evaluate(form, coef, lc_bits, x, fmt, fused=True):
    """Replay a program on target-format inputs ``x`` (bit patterns).

    ``lc_bits`` may be an array that broadcasts against ``x`` (the fitter
    replays many clamps at once).
    """
    x = np.asarray(x, dtype=np.uint16)
    a = tf.absval(x)
    t = tf.min_nan(a, np.asarray(lc_bits, dtype=np.uint16), fmt)       # eq. 2
    x = np.broadcast_to(x, t.shape)
    if form == E:
        return _horner(coef, t, 0, fmt, fused)
    v = _horner(coef, t, 1, fmt, fused)
    half = _half(fmt)
    if form == CO:
        s = tf.xorsign(v, x)
        return tf.fma(s, t, half, fmt) if fused else tf.add(tf.mul(s, t, fmt), half, fmt)
    if form == O:
        return tf.mul(tf.xorsign(v, x), t, fmt)
    if form == HX:
        h = tf.mul(x, half, fmt)
        y = tf.fma(v, t, h, fmt) if fused else tf.add(tf.mul(v, t, fmt), h, fmt)
        tail = tf.greater(a, np.asarray(lc_bits, dtype=np.uint16), fmt)
        relu = np.where(tf.greater(x, np.uint16(0), fmt), x, np.uint16(0))
        return np.where(tail, relu, y).astype(np.uint16)
    raise ValueError(form)


def forward(prog: Program, x, fused=True):
    return evaluate(prog.form, prog.coef, prog.lc_bits, x, prog.fmt, fused)


def backward(prog: Program, x, dy):
    """dx = dy * y(x) for a derivative program (one rounding)."""
    return tf.mul(dy, forward(prog, x), prog.fmt)


def swiglu_forward(silu_prog: Program, g, u):
    """y = s(g) * u (§5.2.4 eq. 15), one rounding for the gate product."""
    return tf.mul(forward(silu_prog, g), u, silu_prog.fmt)


def swiglu_backward(silu_prog: Program, dsilu_prog: Program, g, u, dy):
    """(dg, du) = ((dy*u) * s'(g), dy * s(g)), each product rounded once."""
    fmt = silu_prog.fmt
    dg = tf.mul(tf.mul(dy, u, fmt), forward(dsilu_prog, g), fmt)
    du = tf.mul(dy, forward(silu_prog, g), fmt)
    return dg, du


def swiglu_sigmoid_forward(sig_prog: Program, g, u):
    """The deployed B1/B4 SwiGLU of §3.3 / §5.2.4: recompute the sigmoid
    program p(g), form SiLU as s = g * p, then y = s * u (each product
    rounded once)."""
    fmt = sig_prog.fmt
    p = forward(sig_prog, g)
    return tf.mul(tf.mul(g, p, fmt), u, fmt)


def swiglu_sigmoid_backward(sig_prog: Program, g, u, dy):
    """Backward of the deployed B1/B4 SwiGLU: s' = p + g p (1 - p) (§3.3),
    evaluated as q = fma(-p, p, p) = p - p^2 and s' = fma(g, q, p), each
    rounding once; dg = (dy * u) * s', du = dy * (g * p)."""
    fmt = sig_prog.fmt
    p = forward(sig_prog, g)
    q = tf.fma(tf.xorsign(p, np.uint16(0x8000)), p, p, fmt)
    sd = tf.fma(g, q, p, fmt)
    s = tf.mul(g, p, fmt)
    dg = tf.mul(tf.mul(dy, u, fmt), sd, fmt)
    du = tf.mul(dy, s, fmt)
    return dg, du


def derive(prog: Program) -> Program:
    """Differentiated-polynomial backward (§3.3: "B2 differentiates its D4
    tanh program and evaluates the resulting D3 program").  For an odd or
    centred-odd program y = [1/2 +] sign(x) (c_1 t + ... + c_D t^D), the
    derivative on |x| < Lc is the even polynomial c_1 + 2 c_2 t + ... +
    D c_D t^(D-1); each coefficient (j+1) c_(j+1) is rounded once to the
    target format.  The result is an even-form program of degree D - 1 with
    the same clamp (beyond Lc it keeps the value at Lc)."""
    assert prog.form in (CO, O)
    c = prog.coef_values()
    e = [(j + 1) * float(c[j + 1]) for j in range(prog.degree)]   # exact in FP64
    bits = tuple(int(b) for b in tf.from_f64(np.array(e), prog.fmt))
    from .reference import BWD
    return Program(fn=prog.fn, direction=BWD, fmt=prog.fmt, degree=prog.degree - 1,
                   li=prog.li, lc=prog.lc, coef=bits, lc_bits=prog.lc_bits,
                   info={"derived_from_degree": prog.degree})


def softcap_consts(alpha: float, fmt: str):
    """alpha and 1/alpha rounded once to the target format."""
    return int(tf.from_f64(alpha, fmt)), int(tf.from_f64(1.0 / alpha, fmt))


def softcap_forward(tanh_prog: Program, alpha: float, x):
    """softcap_alpha(x) = alpha tanh(x / alpha) (§2.3 eq. 1): z = x * (1/alpha),
    y = alpha * tanh_program(z), each product rounded once."""
    fmt = tanh_prog.fmt
    a, ia = softcap_consts(alpha, fmt)
    z = tf.mul(x, np.uint16(ia), fmt)
    return tf.mul(np.uint16(a), forward(tanh_prog, z), fmt)


def softcap_backward(dtanh_prog: Program, alpha: float, x, dy):
    """d/dx softcap = tanh'(x / alpha) (eq. 12: the scale cancels):
    dx = dy * dtanh_program(x * (1/alpha)), each product rounded once."""
    fmt = dtanh_prog.fmt
    _, ia = softcap_consts(alpha, fmt)
    z = tf.mul(x, np.uint16(ia), fmt)
    return tf.mul(dy, forward(dtanh_prog, z), fmt)


def evaluate_real(form, coef_values, lc, x):
    """Real-arithmetic replay (FP64, no intermediate rounding): the Table 2
    metric evaluates the rounded coefficients this way (§4.1)."""
    x = np.asarray(x, dtype=np.float64)
    t = np.minimum(np.abs(x), lc)
    D = len(coef_values) - 1
    last = 0 if form == E else 1
    v = np.full_like(t, coef_values[D])
    for j in range(D - 1, last - 1, -1):
        v = v * t + coef_values[j]
    if form == E:
        return v
    sv = np.where(np.signbit(x), -v, v)
    if form == CO:
        return 0.5 + sv * t
    if form == O:
        return sv * t
    y = 0.5 * x + v * t
    return np.where(np.abs(x) > lc, np.maximum(x, 0.0), y)

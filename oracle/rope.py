"""Paired sine/cosine from a Q0.32 turn phase, and fused RoPE -- replay oracle.

TEST INFRASTRUCTURE ONLY -- see ``oracle/__init__.py``.

"Fast Polynomial Transcendentals for LLMs" (arXiv 2610.00049), Appendix B.2:
the host stores each frequency's turn increment Delta_i = round(omega_i 2^32
/ 2 pi) as an unsigned Q0.32 word; at position p the kernel forms
(p Delta_i) mod 2^32, reduces it to a signed Q15 half-turn coordinate and
evaluates a packed FP16 D5 sine and D6 cosine that share the squared input.
The fused experiment reads FP16 Q [B, S, Hq, D] and K [B, S, Hkv, D], applies
the complex rotation and writes [B, Hq, S, D] and [B, Hkv, S, D].

Readings (the page prints no coefficients and no reduction details):
* omega_i = base^(-2 i / D), i = 0 .. D/2 - 1; rotation of interleaved pairs
  (x_2i, x_2i+1) as the complex number x_2i + i x_2i+1.
* Reduction: s = phi as a signed 32-bit turn (s / 2^31 half-turns in
  [-1, 1)); outside [-1/2, 1/2] half-turns fold by the symmetry
  sin(pi u) = sin(pi (+-1 - u)), cos(pi u) = -cos(pi (+-1 - u)); then
  q = s' >> 16 (arithmetic) is the signed Q15 half-turn coordinate
  (u = q / 2^15 in [-1/2, 1/2]).  A D5 odd sine over a full half-turn errs
  by 1.6e-2, over the folded quarter-turn by 1.6e-4.
* Programs: sin(pi u) ~ u (s1 + s3 w + s5 w^2), cos(pi u) ~ 1 + c2 w + c4 w^2
  + c6 w^3 with w = u^2, fitted like eq. 7-8: least squares on 2,000 Chebyshev
  nodes of [0, 1/2] with the end value exact (sin = 1, cos = 0 at u = 1/2),
  in FP64; coefficients rounded to FP16.
* Packed FP16 evaluation, one rounding per operation:
    u = FP16(q) * 2^-15;  w = u * u
    sin: v = fma(s5, w, s3); v = fma(v, w, s1); sin = v * u
    cos: v = fma(c6, w, c4); v = fma(v, w, c2); cos = fma(v, w, 1); negated if folded
* Rotation of (a, b) by (c, s): t = (b s, a s) -> (-(b s), a s);
  out = fma((a, b), (c, c), t) = (a c - b s, b c + a s).
  Backward rotates by -theta: the same with s negated.
"""
from __future__ import annotations

import math

import numpy as np

from . import tformat as tf

F = "f16"
N_NODES = 2000


def turn_increments(head_dim: int, base: float = 10000.0) -> np.ndarray:
    """Delta_i = round(omega_i 2^32 / 2 pi), omega_i = base^(-2i/D)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    omega = base ** (-2.0 * i / head_dim)
    return np.round(omega * 2.0 ** 32 / (2.0 * math.pi)).astype(np.uint64).astype(np.uint32)


def _constrained_ls(f_target, powers, fixed, end_value, x_end=0.5):
    """min ||sum_k a_k x^p_k + fixed(x) - f|| on Chebyshev nodes of [0, x_end]
    subject to the polynomial taking end_value at x_end: the last coefficient
    is eliminated through the constraint."""
    k = np.arange(N_NODES, dtype=np.float64)
    x = 0.5 * x_end * (1.0 + np.cos((2.0 * k + 1.0) * math.pi / (2.0 * N_NODES)))
    y = f_target(x) - fixed(x)
    r = end_value - fixed(np.array([x_end]))[0]        # sum_k a_k x_end^p_k = r
    pl = powers[-1]
    # a_last = (r - sum_{k<last} a_k x_end^p_k) / x_end^pl
    cols = [x ** p - x ** pl * (x_end ** p / x_end ** pl) for p in powers[:-1]]
    A = np.stack(cols, axis=1)
    rhs = y - x ** pl * (r / x_end ** pl)
    a, *_ = np.linalg.lstsq(A, rhs, rcond=None)
    last = (r - sum(a[j] * x_end ** powers[j] for j in range(len(a)))) / x_end ** pl
    return np.concatenate([a, [last]])


def fit_sincos():
    """FP64 coefficients (s1, s3, s5) and (c2, c4, c6)."""
    s = _constrained_ls(lambda u: np.sin(math.pi * u), [1, 3, 5], lambda u: 0.0 * u, 1.0)
    c = _constrained_ls(lambda u: np.cos(math.pi * u), [2, 4, 6], lambda u: 1.0 + 0.0 * u, 0.0)
    return s, c


def sincos_coefficients():
    """FP16 bit patterns (s1, s3, s5), (c2, c4, c6)."""
    s, c = fit_sincos()
    return tuple(int(b) for b in tf.from_f64(s, F)), tuple(int(b) for b in tf.from_f64(c, F))


def phase_q15(pos, delta):
    """(q, flip): the signed Q15 half-turn coordinate after folding, and
    whether the cosine changes sign.  pos, delta broadcast (uint32 math)."""
    phi = (np.asarray(pos, dtype=np.uint64) * np.asarray(delta, dtype=np.uint64)) & 0xFFFFFFFF
    s = phi.astype(np.int64)
    s = np.where(s >= 2 ** 31, s - 2 ** 32, s)                    # signed turn, Q31 half-turns
    hi, lo = s > 2 ** 30, s < -(2 ** 30)
    s2 = np.where(hi, 2 ** 31 - s, np.where(lo, -(2 ** 31) - s, s))
    q = s2 >> 16                                                   # arithmetic shift
    return q.astype(np.int64), hi | lo


def sincos_f16(q, flip):
    """Packed-FP16 cos and sin (bit patterns) of pi * q / 2^15."""
    (s1, s3, s5), (c2, c4, c6) = sincos_coefficients()
    uq = tf.from_f64(np.asarray(q, dtype=np.float64), F)          # int -> FP16, one rounding
    u = tf.mul(uq, np.uint16(0x0200), F)                           # * 2^-15 (exact)
    w = tf.mul(u, u, F)
    v = tf.fma(np.uint16(s5), w, np.uint16(s3), F)
    v = tf.fma(v, w, np.uint16(s1), F)
    sn = tf.mul(v, u, F)
    v = tf.fma(np.uint16(c6), w, np.uint16(c4), F)
    v = tf.fma(v, w, np.uint16(c2), F)
    cs = tf.fma(v, w, np.uint16(0x3C00), F)
    cs = np.where(flip, cs ^ np.uint16(0x8000), cs).astype(np.uint16)
    return cs, sn


def rotate(x, cs, sn, inverse=False):
    """Complex rotation of interleaved pairs: x [..., D] bit patterns,
    cs, sn [..., D/2].  out = fma((a, b), (c, c), (-(b s), a s))."""
    a, b = x[..., 0::2], x[..., 1::2]
    if inverse:
        sn = sn ^ np.uint16(0x8000)
    bs = tf.mul(b, sn, F)
    as_ = tf.mul(a, sn, F)
    re = tf.fma(a, cs, bs ^ np.uint16(0x8000), F)
    im = tf.fma(b, cs, as_, F)
    out = np.empty_like(x)
    out[..., 0::2], out[..., 1::2] = re, im
    return out


def tables(seq: int, delta, pos_offset: int = 0):
    """cos, sin bit patterns [S, D/2] for positions pos_offset .. + S - 1."""
    pos = (np.arange(seq, dtype=np.uint64) + np.uint64(pos_offset))[:, None]
    q, flip = phase_q15(pos, np.asarray(delta, dtype=np.uint64)[None, :])
    return sincos_f16(q, flip)


def rope_forward(q, k, delta, pos_offset: int = 0):
    """q [B, S, Hq, D], k [B, S, Hkv, D] -> [B, Hq, S, D], [B, Hkv, S, D]."""
    B, S = q.shape[0], q.shape[1]
    cs, sn = tables(S, delta, pos_offset)                          # [S, D/2]
    c4, s4 = cs[None, :, None, :], sn[None, :, None, :]
    qo = rotate(q, c4, s4).transpose(0, 2, 1, 3).copy()
    ko = rotate(k, c4, s4).transpose(0, 2, 1, 3).copy()
    return qo, ko


def rope_backward(dq, dk, delta, pos_offset: int = 0):
    """Gradients [B, Hq, S, D], [B, Hkv, S, D] -> [B, S, Hq, D], [B, S, Hkv, D]
    (rotation by -theta, transposed back)."""
    S = dq.shape[2]
    cs, sn = tables(S, delta, pos_offset)
    c4, s4 = cs[None, None, :, :], sn[None, None, :, :]
    gq = rotate(dq, c4, s4, inverse=True).transpose(0, 2, 1, 3).copy()
    gk = rotate(dk, c4, s4, inverse=True).transpose(0, 2, 1, 3).copy()
    return gq, gk

"""Pins of the RoPE oracle (oracle/rope.py): the Q0.32 turn increments, the
phase reduction and folding (against high-precision angles), the
endpoint-constrained sine/cosine fits, the packed-FP16 programs over every
Q15 coordinate, the rotation in exact rationals, identity at position 0 and
the FP64 complex-multiplication reference."""
import math

import numpy as np
import pytest

import exact_t as ex
from oracle import rope
from oracle import tformat as tf

mp = pytest.importorskip("mpmath")


def test_turn_increments():
    d = rope.turn_increments(128)
    mp.mp.dps = 40
    for i in (0, 1, 17, 63):
        omega = mp.mpf(10000) ** (mp.mpf(-2 * i) / 128)
        assert int(d[i]) == int(mp.nint(omega * 2 ** 32 / (2 * mp.pi)))
    assert int(d[0]) == 683565276


def test_phase_reduction_and_fold():
    """q / 2^15 half-turns, with the fold, gives the same sine and the
    negated cosine as the unreduced angle (checked in high precision)."""
    mp.mp.dps = 30
    rng = np.random.default_rng(1)
    pos = rng.integers(0, 1 << 20, 400)
    delta = rng.integers(1, 1 << 32, 400, dtype=np.uint64)
    q, flip = rope.phase_q15(pos, delta)
    for p, dl, qq, fl in zip(pos, delta, q, flip):
        phi = (int(p) * int(dl)) % (1 << 32)
        theta = 2 * mp.pi * mp.mpf(phi) / 2 ** 32
        u = mp.mpf(int(qq)) / 2 ** 15
        assert abs(u) <= 0.5
        # q truncates 16 bits: the folded angle differs from the true one by < 2^-15 half-turns
        assert abs(mp.sin(mp.pi * u) - mp.sin(theta)) <= mp.pi * 2.0 ** -15
        sgn = -1 if fl else 1
        assert abs(sgn * mp.cos(mp.pi * u) - mp.cos(theta)) <= mp.pi * 2.0 ** -15


def test_fits_meet_end_values_and_normal_equations():
    s, c = rope.fit_sincos()
    assert abs(s[0] / 2 + s[1] / 8 + s[2] / 32 - 1.0) <= 1e-14          # sin(pi/2) = 1
    assert abs(1.0 + c[0] / 4 + c[1] / 16 + c[2] / 64) <= 1e-14          # cos(pi/2) = 0
    assert abs(s[0] - math.pi) < 2e-3 and abs(c[0] + math.pi ** 2 / 2) < 1e-2   # Taylor leading terms
    u = 0.25 * (1 + np.cos((2 * np.arange(2000) + 1) * math.pi / 4000))
    r = np.sin(math.pi * u) - (s[0] * u + s[1] * u ** 3 + s[2] * u ** 5)
    # residual orthogonal to the free directions u^p - u^5 (p/2)^(5-p)... of the constrained space
    for p in (1, 3):
        col = u ** p - u ** 5 * (0.5 ** p / 0.5 ** 5)
        assert abs(col @ r) <= 1e-10 * np.linalg.norm(col) * np.linalg.norm(r)


def test_sincos_every_q15_coordinate():
    q = np.arange(-16384, 16385)
    for flip in (False, True):
        cs, sn = rope.sincos_f16(q, np.full(q.size, flip))
        u = q / 32768.0
        cref = np.cos(np.pi * u) * (-1 if flip else 1)
        assert np.max(np.abs(tf.decode(cs, "f16") - cref)) < 1.2e-3
        assert np.max(np.abs(tf.decode(sn, "f16") - np.sin(np.pi * u))) < 1.2e-3
    # odd sine, even cosine, bit for bit
    cs, sn = rope.sincos_f16(q, np.zeros(q.size, bool))
    assert np.array_equal(sn, sn[::-1] ^ np.uint16(0x8000)) or np.array_equal(
        sn[q != 0], (sn[::-1] ^ np.uint16(0x8000))[q != 0])
    assert np.array_equal(cs, cs[::-1])


def test_rotation_exact_rationals():
    rng = np.random.default_rng(2)
    x = tf.from_f64(rng.normal(0, 2, (50, 8)), "f16")
    cs = tf.from_f64(rng.uniform(-1, 1, (50, 4)), "f16")
    sn = tf.from_f64(rng.uniform(-1, 1, (50, 4)), "f16")
    for inv in (False, True):
        out = rope.rotate(x, cs, sn, inverse=inv)
        for r in range(50):
            for j in range(4):
                a, b, c, s = int(x[r, 2 * j]), int(x[r, 2 * j + 1]), int(cs[r, j]), int(sn[r, j])
                if inv:
                    s ^= 0x8000
                bs, as_ = ex.mul(b, s, "f16"), ex.mul(a, s, "f16")
                assert int(out[r, 2 * j]) == ex.fma(a, c, bs ^ 0x8000, "f16")
                assert int(out[r, 2 * j + 1]) == ex.fma(b, c, as_, "f16")


def test_rope_forward_against_fp64_and_identity_at_position_zero():
    rng = np.random.default_rng(3)
    B, S, Hq, Hkv, D = 2, 33, 4, 2, 16
    q = tf.from_f64(rng.normal(0, 1, (B, S, Hq, D)), "f16")
    k = tf.from_f64(rng.normal(0, 1, (B, S, Hkv, D)), "f16")
    delta = rope.turn_increments(D)
    qo, ko = rope.rope_forward(q, k, delta)
    assert qo.shape == (B, Hq, S, D) and ko.shape == (B, Hkv, S, D)
    # position 0: cos = 1, sin = 0 exactly -> the input, transposed (up to -0 -> +0)
    assert np.array_equal(tf.decode(qo[:, :, 0, :], "f16"), tf.decode(q[:, 0, :, :], "f16"))
    # FP64 complex rotation with the true angles p * omega
    qv = tf.decode(q, "f16")
    z = qv[..., 0::2] + 1j * qv[..., 1::2]
    omega = 10000.0 ** (-2.0 * np.arange(D // 2) / D)
    ang = np.arange(S)[None, :, None, None] * omega[None, None, None, :]
    zr = z * np.exp(1j * ang)
    want = np.empty_like(qv)
    want[..., 0::2], want[..., 1::2] = zr.real, zr.imag
    got = tf.decode(qo, "f16").transpose(0, 2, 1, 3)
    bound = 1.3e-3 * (np.abs(qv[..., 0::2]) + np.abs(qv[..., 1::2])).repeat(2, axis=-1) \
        + 2.0 ** -10 * np.abs(want)
    assert np.all(np.abs(got - want) <= bound + 1e-6)
    # backward after forward returns the input up to the two rotations' error
    gq, gk = rope.rope_backward(qo, ko, delta)
    assert gq.shape == q.shape and gk.shape == k.shape
    assert np.max(np.abs(tf.decode(gq, "f16") - qv)) < 1e-2 * (np.abs(qv).max() + 1)

"""GPU parity: every kernel of libpolyact, called through the C ABI, against
the CPU replay oracle, bit for bit.

Cases: the raw packed instructions against the oracle's arithmetic; every
program over all 65,536 input patterns (±0, subnormals, ±inf, NaN); sizes
1..67 at element offsets 0..7 with guard bands; in-place calls; the
L2-resident (4,194,304) and HBM-resident (268,435,456) FP16 sweeps at full
size (every element: the program through the oracle's exhaustive table,
products rounded once -- a product of two 16-bit values is exact in FP32 --
plus oracle replay of sampled elements); dense SwiGLU [8192 x 14336] BF16 and
ragged routed-expert SwiGLU with Zipf segments, every element the same way
(plus untouched rows past the last offset and the offset-validation status);
small contiguous and strided cases replayed element by element.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import DEV, FMT, TDT, from_dev, guards_intact, oracle_program, sentinel_buffer, to_dev
from oracle import reference as ref
from oracle import tformat as tf
from oracle.replay import backward, forward, swiglu_backward, swiglu_forward
from polynomial_activation_gb300 import binding as B

pytestmark = pytest.mark.gpu

DTS = [B.POLY_BF16, B.POLY_F16]
FNS = [B.POLY_SIGMOID, B.POLY_TANH, B.POLY_SILU, B.POLY_GELU]
PROGRAMS = [(fn, d) for fn in FNS for d in (B.POLY_FWD, B.POLY_BWD)]
X_ALL = tf.all_patterns()


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available()
    torch.cuda.set_device(DEV)
    B.poly_reset_programs()
    yield
    torch.cuda.synchronize()


def _rand_bits(rng, n, fmt):
    b = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    k = n // 2
    b[:k] = tf.from_f64(rng.normal(0, 4, k), fmt)
    return b


# ---------------------------------------------------------------- arithmetic

@pytest.mark.parametrize("dt", DTS)
def test_silicon_matches_oracle_arithmetic(dt):
    """fma.rn / mul.rn / min.NaN / max / set.gt on random and special operands
    equal the oracle's one-rounding model (the programs rely on nothing else)."""
    fmt = FMT[dt]
    rng = np.random.default_rng(100 + dt)
    n = 1 << 20
    a, b, c = (_rand_bits(rng, n, fmt) for _ in range(3))
    sp = np.array([0, 0x8000, 1, 0x8001, 0x7FFF, 0xFFFF, 0x7C00 if dt == 0 else 0x7F80,
                   0xFC00 if dt == 0 else 0xFF80, 0x3C00 if dt == 0 else 0x3F80], dtype=np.uint16)
    for arr in (a, b, c):
        idx = rng.random(n) < 0.03
        arr[idx] = sp[rng.integers(0, len(sp), int(idx.sum()))]
    da, db, dc = to_dev(a, dt), to_dev(b, dt), to_dev(c, dt)
    out = torch.empty_like(da)

    def run(op):
        B.poly_diag_packed(op, dt, da, db, dc, out)
        return from_dev(out)

    assert np.array_equal(run(B.POLY_DIAG_FMA), tf.fma(a, b, c, fmt))
    assert np.array_equal(run(B.POLY_DIAG_MUL), tf.mul(a, b, fmt))
    # the clamp only ever sees min(|x|, Lc) with Lc > 0
    da2 = to_dev(tf.absval(a), dt)
    lc = np.full(n, int(tf.from_f64(4.75, fmt)), dtype=np.uint16)
    B.poly_diag_packed(B.POLY_DIAG_MIN_NAN, dt, da2, to_dev(lc, dt), dc, out)
    assert np.array_equal(from_dev(out), tf.min_nan(tf.absval(a), lc, fmt))
    gt = run(B.POLY_DIAG_GT)
    want_gt = np.where(tf.greater(a, b, fmt), np.uint16(0xFFFF), np.uint16(0))
    assert np.array_equal(gt, want_gt)
    # max(x, +0) as used by the exact tail: x away from zero and not NaN
    zero = np.zeros(n, dtype=np.uint16)
    ok = ~tf.is_nan(a, fmt) & (tf.decode(a, fmt) != 0)
    B.poly_diag_packed(B.POLY_DIAG_MAX, dt, da, to_dev(zero, dt), dc, out)
    mx = from_dev(out)
    want = np.where(tf.decode(a, fmt) > 0, a, np.uint16(0))
    assert np.array_equal(mx[ok], want[ok])


# ------------------------------------------------------------- exhaustive

@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("fn,d", PROGRAMS)
def test_exhaustive_patterns(fn, d, dt):
    """All 65,536 input patterns through every program, forward and backward."""
    op = oracle_program(fn, d, dt)
    x = X_ALL
    xd = to_dev(x, dt)
    out = torch.empty_like(xd)
    if d == B.POLY_FWD:
        B.poly_act_fwd(fn, dt, xd, out)
        want = forward(op, x)
    else:
        dy = _rand_bits(np.random.default_rng(5), x.size, FMT[dt])
        B.poly_act_bwd(fn, dt, xd, to_dev(dy, dt), out)
        want = backward(op, x, dy)
    got = from_dev(out)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(x[i]), hex(got[i]), hex(want[i])) for i in bad[:8]]


# ------------------------------------------------------- sizes and offsets

@pytest.mark.parametrize("dt", DTS)
def test_small_sizes_offsets_and_guards(dt):
    """n = 1..67 at element offsets 0..7 (scalar head, vector body, scalar
    tail, unaligned fallback); nothing outside [0, n) is written."""
    fmt = FMT[dt]
    rng = np.random.default_rng(9)
    ops = {(fn, d): oracle_program(fn, d, dt) for fn, d in PROGRAMS}
    G = 64
    for n in list(range(1, 68)) + [255, 1031]:
        for off_x in range(8):
            off_y = off_x if n % 3 else (off_x + 3) % 8      # sometimes mismatched alignment
            fn, d = PROGRAMS[(n + off_x) % len(PROGRAMS)]
            x = _rand_bits(rng, n, fmt)
            dy = _rand_bits(rng, n, fmt)
            xb = to_dev(np.concatenate([np.zeros(off_x, np.uint16), x]), dt)[off_x:]
            dyb = to_dev(np.concatenate([np.zeros(off_x, np.uint16), dy]), dt)[off_x:]
            buf, y = sentinel_buffer(n, G, dt, off_y)
            if d == B.POLY_FWD:
                B.poly_act_fwd(fn, dt, xb, y, n)
                want = forward(ops[(fn, d)], x)
            else:
                B.poly_act_bwd(fn, dt, xb, dyb, y, n)
                want = backward(ops[(fn, d)], x, dy)
            assert np.array_equal(from_dev(y), want), (n, off_x, off_y, fn, d)
            assert guards_intact(buf, n, G, off_y), (n, off_x, off_y)


def _at(bits, off, dt):
    """bits on the device, starting `off` elements past an aligned address."""
    return to_dev(np.concatenate([np.zeros(off, np.uint16), bits]), dt)[off:]


@pytest.mark.parametrize("dt", DTS)
def test_guard_bands_other_kernel_families(dt):
    """Softcap, the MUFU controls and dense SwiGLU (polynomial and control)
    write into sentinel-filled buffers at every 16-byte misalignment, small
    and odd sizes: each result is checked (the oracle; for the controls, the
    same call on aligned buffers) and nothing outside the output changes."""
    from oracle.replay import softcap_backward, softcap_forward
    fmt = FMT[dt]
    rng = np.random.default_rng(97)
    G = 64
    tp = oracle_program(B.POLY_TANH, B.POLY_FWD, dt)
    tdp = oracle_program(B.POLY_TANH, B.POLY_BWD, dt)
    s_op, d_op = _swiglu_ops(dt)
    for n in (1, 2, 7, 8, 9, 15, 17, 33, 67, 1031):
        for off in range(8):
            oo = (off + 3 * (n % 2)) % 8                   # output misaligned differently at odd n
            x, dy = _rand_bits(rng, n, fmt), _rand_bits(rng, n, fmt)
            xd, dyd = _at(x, off, dt), _at(dy, off, dt)
            xa, dya = to_dev(x, dt), to_dev(dy, dt)
            buf, y = sentinel_buffer(n, G, dt, oo)
            B.poly_softcap_fwd(dt, 30.0, xd, y, n)
            assert np.array_equal(from_dev(y), softcap_forward(tp, 30.0, x)), (n, off)
            assert guards_intact(buf, n, G, oo)
            buf, y = sentinel_buffer(n, G, dt, oo)
            B.poly_softcap_bwd(dt, 30.0, xd, dyd, y, n)
            assert np.array_equal(from_dev(y), softcap_backward(tdp, 30.0, x, dy)), (n, off)
            assert guards_intact(buf, n, G, oo)
            for fn, d in ((B.POLY_SIGMOID, 0), (B.POLY_GELU, 0), (B.POLY_TANH, 1), (B.POLY_SILU, 1)):
                ref = torch.empty_like(xa)
                buf, y = sentinel_buffer(n, G, dt, oo)
                if d == 0:
                    B.poly_ctrl_act_fwd(fn, dt, xa, ref, n)
                    B.poly_ctrl_act_fwd(fn, dt, xd, y, n)
                else:
                    B.poly_ctrl_act_bwd(fn, dt, xa, dya, ref, n)
                    B.poly_ctrl_act_bwd(fn, dt, xd, dyd, y, n)
                assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), (fn, d, n, off)
                assert guards_intact(buf, n, G, oo)
    for rows, cols in ((1, 1), (3, 13), (2, 8), (5, 17), (4, 64)):
        m = rows * cols
        for off in range(8):
            oo = (off + 5) % 8
            g, u, dy = (_rand_bits(rng, m, fmt) for _ in range(3))
            gd, ud, dyd = (_at(a, off, dt).view(rows, cols) for a in (g, u, dy))
            gr, ur, dyr = g.reshape(rows, cols), u.reshape(rows, cols), dy.reshape(rows, cols)
            for ctrl in (False, True):
                bufs = [sentinel_buffer(m, G, dt, oo) for _ in range(3)]
                y, dg, du = (b[1].view(rows, cols) for b in bufs)
                if ctrl:
                    B.poly_ctrl_swiglu_fwd(dt, gd, ud, y)
                    B.poly_ctrl_swiglu_bwd(dt, gd, ud, dyd, dg, du)
                    ga, ua, dya = (to_dev(a, dt).view(rows, cols) for a in (g, u, dy))
                    ry, rdg, rdu = torch.empty_like(ga), torch.empty_like(ga), torch.empty_like(ga)
                    B.poly_ctrl_swiglu_fwd(dt, ga, ua, ry)
                    B.poly_ctrl_swiglu_bwd(dt, ga, ua, dya, rdg, rdu)
                    want = (from_dev(ry), from_dev(rdg), from_dev(rdu))
                else:
                    B.poly_swiglu_fwd(dt, gd, ud, y)
                    B.poly_swiglu_bwd(dt, gd, ud, dyd, dg, du)
                    want = (swiglu_forward(s_op, gr, ur),) + tuple(swiglu_backward(s_op, d_op, gr, ur, dyr))
                for (b, _), got, w in zip(bufs, (y, dg, du), want):
                    assert np.array_equal(from_dev(got).reshape(rows, cols), np.reshape(w, (rows, cols))), \
                        (rows, cols, off, ctrl)
                    assert guards_intact(b, m, G, oo)


def test_guard_bands_exp2_and_rope():
    """exp2 (FP32, every 4-byte offset within 16 bytes) and fused RoPE
    (outputs inside sentinel buffers) write exactly their outputs."""
    from oracle import exp2 as e2, rope
    rng = np.random.default_rng(98)
    G = 32
    for n in (1, 3, 4, 5, 31, 67, 1029):
        for off in range(4):
            oo = (off + 1) % 4
            x = rng.uniform(-60, 10, n).astype(np.float32)
            xd = torch.from_numpy(np.concatenate([np.zeros(off, np.float32), x])).to(DEV)[off:]
            buf = torch.full((2 * G + oo + n,), 0x5A5A5A5A, dtype=torch.int32, device=DEV)
            y = buf[G + oo: G + oo + n].view(torch.float32)
            B.poly_exp2(B.POLY_EXP2_D2, xd, y, n)
            assert np.array_equal(y.cpu().numpy().view(np.uint32), e2.exp2_replay("D2", x)), (n, off)
            assert bool((buf[:G + oo] == 0x5A5A5A5A).all() and (buf[G + oo + n:] == 0x5A5A5A5A).all())
    for b, s, hq, hkv, d in ((1, 5, 3, 1, 8), (2, 9, 2, 3, 16), (1, 1, 1, 0, 64)):
        q, k = _rope_case(rng, b, s, hq, hkv, d)
        delta = rope.turn_increments(d)
        dd = torch.from_numpy(delta.view(np.int32)).to(DEV)
        qd, kd = to_dev(q, 0), to_dev(k, 0)
        nq, nk = b * hq * s * d, b * hkv * s * d
        Gh = 8 * 16                                           # a 16-byte multiple of FP16 elements
        bq = torch.full((2 * Gh + nq,), 0x5A5A, dtype=torch.int16, device=DEV)
        bk = torch.full((2 * Gh + nk,), 0x5A5A, dtype=torch.int16, device=DEV)
        qo = bq[Gh:Gh + nq].view(torch.float16).view(b, hq, s, d)
        ko = bk[Gh:Gh + nk].view(torch.float16).view(b, hkv, s, d)
        B.poly_rope_fwd(B.POLY_ROPE_POLY, qd, kd if hkv else None, qo, ko if hkv else None, dd,
                        batch=b, seq=s, hq=hq, hkv=hkv, head_dim=d, pos_offset=11)
        wq, wk = rope.rope_forward(q, k, delta, 11)
        assert np.array_equal(from_dev(qo).reshape(wq.shape), wq)
        if hkv:
            assert np.array_equal(from_dev(ko).reshape(wk.shape), wk)
        for t, m in ((bq, nq), (bk, nk)):
            assert bool((t[:Gh] == 0x5A5A).all() and (t[Gh + m:] == 0x5A5A).all())
        if not hkv:
            assert bool((bk == 0x5A5A).all())


def test_binding_checks_tensor_extents_before_launch():
    """A tensor too short for the call, a dtype that disagrees with the
    call's, or pageable host memory is refused by the binding before the
    library sees the address; the output stays untouched."""
    dt = B.POLY_F16
    x = torch.zeros(1000, dtype=torch.float16, device=DEV)
    dy_short = torch.zeros(999, dtype=torch.float16, device=DEV)
    y = torch.full((1000,), 0x5A5A, dtype=torch.int16, device=DEV).view(torch.float16)
    with pytest.raises(ValueError, match="dy"):
        B.poly_act_bwd(B.POLY_SIGMOID, dt, x, dy_short, y)
    with pytest.raises(ValueError, match="y"):
        B.poly_act_fwd(B.POLY_SIGMOID, dt, x, y[1:])
    with pytest.raises(ValueError, match="dtype"):
        B.poly_act_fwd(B.POLY_SIGMOID, B.POLY_BF16, x, y)
    with pytest.raises(ValueError, match="pinned"):
        B.poly_act_fwd(B.POLY_SIGMOID, dt, x, torch.empty(1000, dtype=torch.float16))
    with pytest.raises(ValueError, match="x"):                        # owns 2 bytes, shows 1000
        B.poly_act_fwd(B.POLY_SIGMOID, dt, torch.zeros(1, dtype=torch.float16, device=DEV).expand(1000), y)
    qb = torch.zeros((1, 4, 2, 8), dtype=torch.bfloat16, device=DEV)
    dlt = torch.from_numpy(B.poly_rope_turn_increments(8).view(np.int32)).to(DEV)
    with pytest.raises(ValueError, match="dtype"):                    # RoPE is FP16 only
        B.poly_rope_fwd(B.POLY_ROPE_POLY, qb, None, torch.empty((1, 2, 4, 8), dtype=torch.bfloat16,
                        device=DEV), None, dlt, hkv=0)
    g = torch.zeros((8, 64), dtype=torch.bfloat16, device=DEV)
    u_short = torch.zeros((8, 32), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError, match="u"):
        B.poly_swiglu_fwd(B.POLY_BF16, g, u_short, torch.empty_like(g), cols=64, ldu=64)
    torch.cuda.synchronize()
    assert bool((y.view(torch.int16) == 0x5A5A).all())


def test_injected_launch_failures_leave_outputs_and_context_intact():
    """Two injected launch failures (poly_debug_fail_launches): the next two
    launching calls -- an activation and a SwiGLU -- raise POLY_ECUDA with the
    injected CUDA code and write nothing; the third call runs and is exact,
    and the CUDA context stays usable."""
    dt, fmt = B.POLY_BF16, "bf16"
    n, G = 4099, 64
    x = _rand_bits(np.random.default_rng(12), n, fmt)
    xb = to_dev(x, dt)
    buf, y = sentinel_buffer(n, G, dt, 0)
    before = from_dev(buf).copy()
    g, u = (to_dev(_rand_bits(np.random.default_rng(s), 8 * 64, fmt), dt).view(8, 64)
            for s in (13, 14))
    ys = torch.full((8, 64), 0x1234, dtype=torch.int16, device=DEV).view(TDT[dt])
    assert B.poly_debug_fail_launches(701, 2) == 0
    try:
        with pytest.raises(B.PolyError) as e1:
            B.poly_act_fwd(B.POLY_SIGMOID, dt, xb, y, n)
        assert e1.value.status == B.POLY_ECUDA and "cudaError 701" in str(e1.value)
        assert B.lib().poly_last_cuda_error() == 701
        with pytest.raises(B.PolyError) as e2:
            B.poly_swiglu_fwd(dt, g, u, ys)
        assert e2.value.status == B.POLY_ECUDA
    finally:
        assert B.poly_debug_fail_launches(701, 0) == 0        # both consumed
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(buf), before)
    assert np.array_equal(from_dev(ys), np.full(8 * 64, 0x1234, np.uint16).reshape(8, 64))
    B.poly_act_fwd(B.POLY_SIGMOID, dt, xb, y, n)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(y), forward(oracle_program(B.POLY_SIGMOID, B.POLY_FWD, dt), x))
    assert guards_intact(buf, n, G, 0)


@pytest.mark.parametrize("dt", DTS)
def test_in_place(dt):
    fmt = FMT[dt]
    x = _rand_bits(np.random.default_rng(3), 100_003, fmt)
    for fn in FNS:
        op = oracle_program(fn, B.POLY_FWD, dt)
        t = to_dev(x, dt)
        B.poly_act_fwd(fn, dt, t, t)
        assert np.array_equal(from_dev(t), forward(op, x))
        dop = oracle_program(fn, B.POLY_BWD, dt)
        t = to_dev(x, dt)
        dy = to_dev(x[::-1].copy(), dt)
        B.poly_act_bwd(fn, dt, t, dy, dy)                   # dx written over dy
        assert np.array_equal(from_dev(dy), backward(dop, x, x[::-1].copy()))


# ------------------------------------------------------------ full configs

SIX = [(B.POLY_SIGMOID, B.POLY_FWD), (B.POLY_TANH, B.POLY_FWD), (B.POLY_SILU, B.POLY_FWD),
       (B.POLY_GELU, B.POLY_FWD), (B.POLY_SIGMOID, B.POLY_BWD), (B.POLY_TANH, B.POLY_BWD)]


def test_l2_resident_sweep_every_element():
    """4,194,304 FP16 elements, x ~ N(0, 3^2), dy ~ N(0, 1): all six programs,
    every element compared."""
    dt = B.POLY_F16
    x, dy = workloads.isolated_l2("f16")
    xd, dyd = to_dev(x, dt), to_dev(dy, dt)
    out = torch.empty_like(xd)
    for fn, d in SIX:
        op = oracle_program(fn, d, dt)
        if d == B.POLY_FWD:
            B.poly_act_fwd(fn, dt, xd, out)
            want = forward(op, x)
        else:
            B.poly_act_bwd(fn, dt, xd, dyd, out)
            want = backward(op, x, dy)
        assert np.array_equal(from_dev(out), want), (fn, d)


def _lut(op):
    return torch.from_numpy(forward(op, X_ALL).view(np.int16)).to(DEV)


def _apply_lut(op, xd):
    """program(x) for every element, from the oracle's exhaustive table."""
    idx = (xd.view(torch.int16).to(torch.int32) & 0xFFFF).long()
    return _lut(op)[idx].view(xd.dtype)


def _rn_mul(a, b):
    """a * b rounded once to the 16-bit format: the product of two FP16 or
    BF16 values is exact in FP32, and torch rounds its FP32 result once."""
    return (a.float() * b.float()).to(a.dtype)


def _equal_bits(got, want):
    g, w = got.view(torch.int16), want.view(torch.int16)
    nan = torch.isnan(want.float())
    return bool(torch.equal(g[~nan], w[~nan])) and bool(torch.isnan(got.float()[nan]).all())


def test_chunk_shape_switch_sizes():
    """Sizes on both sides of the point where a one-input call changes from
    one 16-byte chunk per thread (releasing the next launch after its loads)
    to two (releasing after its stores) -- two two-chunk blocks per SM --
    with and without an n mod 8 tail: every element against the oracle's
    table."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    edge = 2 * sms * 256 * 2 * 8
    dt = B.POLY_BF16
    op = oracle_program(B.POLY_GELU, B.POLY_FWD, dt)
    rng = np.random.default_rng(81)
    big = _rand_bits(rng, edge + 8192, "bf16")
    xd = to_dev(big, dt)
    for n in (edge - 4096 - 3, edge - 8, edge - 1, edge, edge + 5, edge + 8, edge + 4096 + 7):
        y = torch.full((n + 16,), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
        B.poly_act_fwd(B.POLY_GELU, dt, xd[:n], y[:n], n)
        assert _equal_bits(y[:n], _apply_lut(op, xd[:n])), n
        assert bool((y[n:].view(torch.int16) == 0x5A5A).all()), n


def test_two_input_launch_shape_switch_sizes():
    """Two-input one-output calls change shape with size: one chunk per thread
    while that grid holds at most 8 blocks per SM (the next launch released
    after the loads), two chunks while the two-chunk grid holds at most 16
    blocks per SM, one above (both released after the stores).  Sizes on both
    sides of every switch, with and without a tail, for the σ′ and GELU′
    backward programs (FP16), the SwiGLU forward (FP16) and its sigmoid rule
    (BF16), flat and on the halves of a fused gate-up buffer (rows mode):
    every element against the oracle's tables."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    edges = [8 * sms * 256 * 8, 16 * sms * 256 * 2 * 8]
    dt, bf = B.POLY_F16, B.POLY_BF16
    op = oracle_program(B.POLY_SIGMOID, B.POLY_BWD, dt)
    gelu_op = oracle_program(B.POLY_GELU, B.POLY_BWD, dt)
    s_op = oracle_program(B.POLY_SILU, B.POLY_FWD, dt)
    sig_bf = oracle_program(B.POLY_SIGMOID, B.POLY_FWD, bf)
    top = edges[-1] + 8192
    rng = np.random.default_rng(83)
    xd = to_dev(_rand_bits(rng, top, "f16"), dt)
    dyd = to_dev(_rand_bits(rng, top, "f16"), dt)
    xb = to_dev(_rand_bits(rng, top, "bf16"), bf)
    ub = to_dev(_rand_bits(rng, top, "bf16"), bf)
    for edge in edges:
        for n in (edge - 4096 - 3, edge - 8, edge, edge + 5, edge + 8, edge + 4096):
            y = torch.full((n + 16,), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
            B.poly_act_bwd(B.POLY_SIGMOID, dt, xd[:n], dyd[:n], y[:n], n)
            assert _equal_bits(y[:n], _rn_mul(dyd[:n], _apply_lut(op, xd[:n]))), (edge, n)
            assert bool((y[n:].view(torch.int16) == 0x5A5A).all()), (edge, n)
            B.poly_act_bwd(B.POLY_GELU, dt, xd[:n], dyd[:n], y[:n], n)
            assert _equal_bits(y[:n], _rn_mul(dyd[:n], _apply_lut(gelu_op, xd[:n]))), (edge, n)
            assert bool((y[n:].view(torch.int16) == 0x5A5A).all()), (edge, n)
            if n % 8 == 0:
                zb = torch.full((n + 16,), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[bf])
                B.poly_swiglu_fwd_v(B.POLY_SWIGLU_SIGMOID, bf, xb[:n].view(n // 8, 8),
                                    ub[:n].view(n // 8, 8), zb[:n].view(n // 8, 8))
                want = _rn_mul(_rn_mul(xb[:n], _apply_lut(sig_bf, xb[:n])), ub[:n])
                assert _equal_bits(zb[:n], want), (edge, n)
                assert bool((zb[n:].view(torch.int16) == 0x5A5A).all()), (edge, n)
            if n % 8 == 0:
                z = torch.full((n + 16,), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
                B.poly_swiglu_fwd(dt, xd[:n].view(n // 8, 8), dyd[:n].view(n // 8, 8),
                                  z[:n].view(n // 8, 8))
                assert _equal_bits(z[:n], _rn_mul(_apply_lut(s_op, xd[:n]), dyd[:n])), (edge, n)
                assert bool((z[n:].view(torch.int16) == 0x5A5A).all()), (edge, n)
        cols = 1024
        for rows in (edge // cols - 3, edge // cols, edge // cols + 1, edge // cols + 4):
            n = rows * cols
            g, u = xd[:n].view(rows, cols), dyd[:n].view(rows, cols)
            gu = torch.cat([g, u], dim=1)
            zb = torch.full((rows, cols + 8), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
            B.poly_swiglu_fwd(dt, gu[:, :cols], gu[:, cols:], zb[:, :cols])
            want = _rn_mul(_apply_lut(s_op, xd[:n]), dyd[:n])
            assert _equal_bits(zb[:, :cols].reshape(-1), want), (edge, rows)
            assert bool((zb[:, cols:].view(torch.int16) == 0x5A5A).all()), (edge, rows)


@pytest.mark.parametrize("dt", DTS)
def test_realigned_inputs_every_offset_pair(dt):
    """Inputs at other addresses modulo 16 bytes than the output take the
    realigning kernel (two aligned 16-byte loads and a funnel shift per
    chunk; its first and last chunks and the head and tail scalar): every
    pair of input / output element offsets 0..7, the second input at yet
    another offset, sizes around the head, body and tail boundaries -- every
    element against the oracle's tables, guard bands intact."""
    fmt = FMT[dt]
    rng = np.random.default_rng(71)
    op_f = oracle_program(B.POLY_GELU, B.POLY_FWD, dt)
    op_b = oracle_program(B.POLY_TANH, B.POLY_BWD, dt)
    s_op = oracle_program(B.POLY_SILU, B.POLY_FWD, dt)
    top = 8192
    xs = to_dev(_rand_bits(rng, top, fmt), dt)
    ds = to_dev(_rand_bits(rng, top, fmt), dt)
    G = 32
    for n in (1, 7, 8, 9, 15, 16, 17, 23, 24, 25, 31, 32, 33, 40, 41, 1000, 4099):
        for ox in range(8):
            for oy in range(8):
                od = (ox + 3 + oy) % 8
                x, dy = xs[ox:ox + n], ds[od:od + n]
                for kind in ("fwd", "bwd", "swiglu"):
                    buf = torch.full((n + 2 * G + 8,), 0x5A5A, dtype=torch.int16, device=DEV)
                    buf = buf.view(TDT[dt])
                    y = buf[G + oy:G + oy + n]
                    if kind == "fwd":
                        B.poly_act_fwd(B.POLY_GELU, dt, x, y, n)
                        want = _apply_lut(op_f, x)
                    elif kind == "bwd":
                        B.poly_act_bwd(B.POLY_TANH, dt, x, dy, y, n)
                        want = _rn_mul(dy, _apply_lut(op_b, x))
                    else:
                        B.poly_swiglu_fwd_v(B.POLY_SWIGLU_DIRECT, dt, x, dy, y, 1, n, n, n, n)
                        want = _rn_mul(_apply_lut(s_op, x), dy)
                    assert _equal_bits(y, want), (kind, n, ox, oy, od)
                    g = buf.view(torch.int16)
                    assert bool((g[:G + oy] == 0x5A5A).all() and
                                (g[G + oy + n:] == 0x5A5A).all()), (kind, n, ox, oy, od)


def test_random_sizes_offsets_and_families():
    """Sixty random calls: sizes log-uniform over 1..2^24 elements (across
    every launch-shape and release switch), inputs and output at independent
    element offsets 0..7 (same or different alignment, so dense, head / tail
    and scalar paths all run), both formats, every program, the activation
    forward and backward and the flat SwiGLU forward and backward under both
    rules: every element against the oracle's exhaustive tables, guard
    bands around every output intact."""
    rng = np.random.default_rng(2024)
    G = 64
    top = (1 << 24) + 16
    pools = {}
    for dt in DTS:
        fmt = FMT[dt]
        pools[dt] = [to_dev(_rand_bits(rng, top, fmt), dt) for _ in range(3)]
    for case in range(60):
        dt = DTS[case % 2]
        n = int(np.exp(rng.uniform(0.0, np.log(1 << 24))))
        offs = [int(o) for o in rng.integers(0, 8, 4)]
        kind = ("fwd", "bwd", "swiglu_fwd", "swiglu_bwd")[int(rng.integers(0, 4))]
        a, b, c = (pools[dt][k][offs[k]:offs[k] + n] for k in range(3))
        outs = []

        def out_buf():
            buf = torch.full((n + 2 * G + 8,), 0x5A5A, dtype=torch.int16, device=DEV)
            buf = buf.view(TDT[dt])
            outs.append(buf)
            return buf[G + offs[3]:G + offs[3] + n]

        if kind in ("fwd", "bwd"):
            fn = int(rng.integers(0, 4))
            d = B.POLY_FWD if kind == "fwd" else B.POLY_BWD
            op = oracle_program(fn, d, dt)
            y = out_buf()
            if d == B.POLY_FWD:
                B.poly_act_fwd(fn, dt, a, y, n)
                want = _apply_lut(op, a)
            else:
                B.poly_act_bwd(fn, dt, a, b, y, n)
                want = _rn_mul(b, _apply_lut(op, a))
            assert _equal_bits(y, want), (case, kind, fn, dt, n, offs)
        else:
            rule = int(rng.integers(0, 2))
            if rule == B.POLY_SWIGLU_DIRECT:
                s_lut = lambda t: _apply_lut(oracle_program(B.POLY_SILU, B.POLY_FWD, dt), t)
                d_lut = lambda t: _apply_lut(oracle_program(B.POLY_SILU, B.POLY_BWD, dt), t)
            else:
                sig = oracle_program(B.POLY_SIGMOID, B.POLY_FWD, dt)
                s_lut = lambda t: _rn_mul(t, _apply_lut(sig, t))
                d_lut = None
            if kind == "swiglu_fwd":
                y = out_buf()
                B.poly_swiglu_fwd_v(rule, dt, a, b, y, 1, n, n, n, n)
                assert _equal_bits(y, _rn_mul(s_lut(a), b)), (case, kind, rule, dt, n, offs)
            else:
                dg, du = out_buf(), out_buf()
                B.poly_swiglu_bwd_v(rule, dt, a, b, c, dg, du, 1, n, n, n, n, n, n)
                if d_lut is not None:
                    assert _equal_bits(dg, _rn_mul(_rn_mul(c, b), d_lut(a))), (case, rule, n, offs)
                else:   # fused s' = fma(g, fma(-p, p, p), p): the oracle on a sample
                    from oracle.replay import swiglu_sigmoid_backward
                    k = torch.from_numpy(np.unique(rng.integers(0, n, min(n, 4096)))).to(DEV)
                    host = [from_dev(t[k]) for t in (a, b, c)]
                    wdg, _ = swiglu_sigmoid_backward(sig, *host)
                    assert np.array_equal(from_dev(dg[k]), wdg), (case, rule, n, offs)
                assert _equal_bits(du, _rn_mul(c, s_lut(a))), (case, rule, n, offs)
        for buf in outs:
            g = buf.view(torch.int16)
            assert bool((g[:G + offs[3]] == 0x5A5A).all()), (case, kind, n, offs)
            assert bool((g[G + offs[3] + n:] == 0x5A5A).all()), (case, kind, n, offs)


@pytest.mark.parametrize("n", [(1 << 31) - 3, (1 << 31) + 13])
def test_index_width_limits(n):
    """Just below 2^31 elements (the dense kernel's 32-bit indices at their
    limit) and just above (the general kernel's 64-bit path): x cycles
    through all 65,536 FP16 patterns, so every element must equal the
    oracle's exhaustive table at x mod 65,536 (checked in slices of 2^28)."""
    dt = B.POLY_F16
    op = oracle_program(B.POLY_SIGMOID, B.POLY_FWD, dt)
    lut = _lut(op)                                   # int16 [65536] on the device
    pat = torch.from_numpy(X_ALL.view(np.int16)).to(DEV)
    x = torch.empty(n, dtype=torch.int16, device=DEV)
    full = n // 65536
    x[:full * 65536].view(full, 65536).copy_(pat.expand(full, 65536))
    x[full * 65536:] = pat[:n - full * 65536]
    y = torch.empty_like(x)
    B.poly_act_fwd(B.POLY_SIGMOID, dt, x.view(torch.float16), y.view(torch.float16), n)
    torch.cuda.synchronize()
    rows = 1 << 12                                   # 2^12 x 65,536 = 2^28 elements per slice
    for r0 in range(0, full, rows):
        r1 = min(full, r0 + rows)
        got = y[r0 * 65536:r1 * 65536].view(r1 - r0, 65536)
        assert bool((got == lut[None, :]).all()), (n, r0)
    assert torch.equal(y[full * 65536:], lut[:n - full * 65536])
    del x, y


def test_swiglu_above_2_31_elements():
    """SwiGLU forward and backward, dense and ragged, over 2^31 + 2,048
    elements (1,048,577 rows of 2,048): the general kernel's 64-bit path for
    two- and three-input operations.  The gate cycles through all 65,536 BF16
    patterns (the up and dy streams through shifted copies), so every element
    is checked against the oracle's exhaustive tables, in slices of 2^28;
    ragged rows past the last offset stay untouched."""
    dt = B.POLY_BF16
    s_op, d_op = _swiglu_ops(dt)
    ls, ld = _lut(s_op), _lut(d_op)
    rows, cols = 1_048_577, 2048
    n = rows * cols
    assert n > 1 << 31
    cap = rows + 7
    pat = torch.from_numpy(X_ALL.view(np.int16)).to(DEV)

    def cyclic(shift):
        t = torch.empty(cap * cols, dtype=torch.int16, device=DEV)
        p = torch.roll(pat, shift)
        full = t.numel() // 65536
        t[:full * 65536].view(full, 65536).copy_(p.expand(full, 65536))
        t[full * 65536:] = p[:t.numel() - full * 65536]
        return t.view(torch.bfloat16)

    g, u, dy = cyclic(0), cyclic(12_345), cyclic(40_000)

    def check(y, dg, du):
        step = 1 << 28
        for lo in range(0, n, step):
            hi = min(n, lo + step)
            gi = (g[lo:hi].view(torch.int16).to(torch.int32) & 0xFFFF).long()
            sg, sdg = ls[gi].view(torch.bfloat16), ld[gi].view(torch.bfloat16)
            us, dys = u[lo:hi], dy[lo:hi]
            if y is not None:
                assert _equal_bits(y[lo:hi], _rn_mul(sg, us)), lo
            if dg is not None:
                assert _equal_bits(dg[lo:hi], _rn_mul(_rn_mul(dys, us), sdg)), lo
                assert _equal_bits(du[lo:hi], _rn_mul(dys, sg)), lo
            del gi, sg, sdg

    gv, uv, dyv = (t[:n].view(rows, cols) for t in (g, u, dy))
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=DEV)
    B.poly_swiglu_fwd(dt, gv, uv, y)
    check(y.view(-1), None, None)
    dg, du = torch.empty_like(y), torch.empty_like(y)
    B.poly_swiglu_bwd(dt, gv, uv, dyv, dg, du)
    check(None, dg.view(-1), du.view(-1))
    del y, dg, du
    seg = torch.tensor([0, 500_000, 500_000, rows], dtype=torch.int32, device=DEV)
    gc, uc, dyc = (t.view(cap, cols) for t in (g, u, dy))
    fill = lambda: torch.full((cap, cols), 0x5A5A, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    y = fill()
    B.poly_swiglu_fwd_ragged(dt, gc, uc, y, seg)
    check(y.view(-1), None, None)
    assert bool((y[rows:].view(torch.int16) == 0x5A5A).all())
    del y
    dg, du = fill(), fill()
    B.poly_swiglu_bwd_ragged(dt, gc, uc, dyc, dg, du, seg)
    check(None, dg.view(-1), du.view(-1))
    assert bool((dg[rows:].view(torch.int16) == 0x5A5A).all())
    assert bool((du[rows:].view(torch.int16) == 0x5A5A).all())
    del dg, du, g, u, dy
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dt", DTS)
def test_hbm_resident_sweep_full_size(dt):
    """268,435,456 elements (512 MiB per tensor), 1 % outliers in [-40, 40],
    FP16 (the bench's step) and BF16.  Forward: every element equals the
    oracle's exhaustive table at its input.  Backward: 2^21 sampled elements
    plus both ends through the oracle, and every element as dy times the
    tabulated program, one rounding."""
    x, dy = workloads.isolated_hbm(FMT[dt])
    n = x.size
    xd, dyd = to_dev(x, dt), to_dev(dy, dt)
    out = torch.empty_like(xd)
    idx_x = xd.view(torch.int16).to(torch.int32) & 0xFFFF
    rng = np.random.default_rng(77)
    sample = np.unique(np.concatenate([rng.integers(0, n, 1 << 21), np.arange(4096),
                                       np.arange(n - 4096, n)]))
    for fn, d in SIX:
        op = oracle_program(fn, d, dt)
        if d == B.POLY_FWD:
            B.poly_act_fwd(fn, dt, xd, out)
            want = _lut(op)[idx_x.long()]
            assert torch.equal(out.view(torch.int16), want), fn
        else:
            B.poly_act_bwd(fn, dt, xd, dyd, out)
            got = from_dev(out[torch.from_numpy(sample).to(DEV)])
            assert np.array_equal(got, backward(op, x[sample], dy[sample])), fn
            # every element: dy * program(x), one rounding
            assert _equal_bits(out, _rn_mul(dyd, _apply_lut(op, xd))), fn
    del idx_x
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ SwiGLU

def _swiglu_ops(dt):
    return (oracle_program(B.POLY_SILU, B.POLY_FWD, dt),
            oracle_program(B.POLY_SILU, B.POLY_BWD, dt))


@pytest.mark.parametrize("dt", DTS)
def test_swiglu_small_every_element(dt):
    fmt = FMT[dt]
    s_op, d_op = _swiglu_ops(dt)
    rng = np.random.default_rng(21)
    for rows, cols in [(1, 1), (3, 7), (17, 1000), (64, 2048), (5, 8)]:
        g = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
        u = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
        dy = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
        gd, ud, dyd = to_dev(g, dt), to_dev(u, dt), to_dev(dy, dt)
        y = torch.empty_like(gd)
        B.poly_swiglu_fwd(dt, gd, ud, y)
        assert np.array_equal(from_dev(y).reshape(rows, cols), swiglu_forward(s_op, g, u))
        dg, du = torch.empty_like(gd), torch.empty_like(gd)
        B.poly_swiglu_bwd(dt, gd, ud, dyd, dg, du)
        wdg, wdu = swiglu_backward(s_op, d_op, g, u, dy)
        assert np.array_equal(from_dev(dg).reshape(rows, cols), wdg)
        assert np.array_equal(from_dev(du).reshape(rows, cols), wdu)


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("cols,pad", [(2048, 8), (1000, 24), (1001, 3)])
def test_swiglu_strided_every_element(dt, cols, pad):
    """Gate and up as the two halves of one [rows, 2 cols + pad] buffer (a
    fused gate/up projection output), outputs with their own pitch."""
    fmt = FMT[dt]
    s_op, d_op = _swiglu_ops(dt)
    rows = 37
    rng = np.random.default_rng(cols)
    W = 2 * cols + pad
    gu = _rand_bits(rng, rows * W, fmt).reshape(rows, W)
    dy = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
    gud = to_dev(gu, dt)
    g, u = gud[:, :cols], gud[:, cols:2 * cols]
    yb = torch.full((rows, cols + pad), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
    y = yb[:, :cols]
    B.poly_swiglu_fwd(dt, g, u, y)
    gg, uu = gu[:, :cols], gu[:, cols:2 * cols]
    assert np.array_equal(from_dev(y).reshape(rows, cols), swiglu_forward(s_op, gg, uu))
    assert bool((yb.view(torch.int16)[:, cols:] == 0x5A5A).all())
    dgb = torch.full((rows, cols + pad), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
    du = torch.empty(rows, cols, dtype=TDT[dt], device=DEV)
    B.poly_swiglu_bwd(dt, g, u, to_dev(dy, dt), dgb[:, :cols], du)
    wdg, wdu = swiglu_backward(s_op, d_op, gg, uu, dy)
    assert np.array_equal(from_dev(dgb[:, :cols]).reshape(rows, cols), wdg)
    assert np.array_equal(from_dev(du).reshape(rows, cols), wdu)
    assert bool((dgb.view(torch.int16)[:, cols:] == 0x5A5A).all())


def test_dense_swiglu_full_size_sampled():
    """[8192 x 14336] BF16, gate and up ~ 2 N(0, 1), dy ~ N(0, 1)."""
    dt = B.POLY_BF16
    s_op, d_op = _swiglu_ops(dt)
    g, u, dy = workloads.dense_swiglu("bf16")
    gd, ud, dyd = to_dev(g, dt), to_dev(u, dt), to_dev(dy, dt)
    y = torch.empty_like(gd)
    dg, du = torch.empty_like(gd), torch.empty_like(gd)
    B.poly_swiglu_fwd(dt, gd, ud, y)
    B.poly_swiglu_bwd(dt, gd, ud, dyd, dg, du)
    n = g.size
    rng = np.random.default_rng(31)
    s = np.unique(np.concatenate([rng.integers(0, n, 1 << 20), np.arange(2048),
                                  np.arange(n - 2048, n)]))
    sd = torch.from_numpy(s).to(DEV)
    gf, uf, dyf = g.reshape(-1), u.reshape(-1), dy.reshape(-1)
    assert np.array_equal(from_dev(y.view(-1)[sd]), swiglu_forward(s_op, gf[s], uf[s]))
    wdg, wdu = swiglu_backward(s_op, d_op, gf[s], uf[s], dyf[s])
    assert np.array_equal(from_dev(dg.view(-1)[sd]), wdg)
    assert np.array_equal(from_dev(du.view(-1)[sd]), wdu)
    # every element through the oracle's exhaustive tables
    sg, sdg = _apply_lut(s_op, gd), _apply_lut(d_op, gd)
    assert _equal_bits(y, _rn_mul(sg, ud))
    assert _equal_bits(dg, _rn_mul(_rn_mul(dyd, ud), sdg))
    assert _equal_bits(du, _rn_mul(dyd, sg))


def test_component_workloads_every_element():
    """The bench's component shapes, in the launch configuration it times:
    the SiLU probe (58,720,256 BF16 values) forward and backward, and the
    expert SwiGLU activation (24,576 x 1,280 BF16) forward and backward,
    every element through the oracle's exhaustive tables, plus a sample
    through the oracle's replay."""
    dt, fmt = B.POLY_BF16, "bf16"
    s_op, d_op = _swiglu_ops(dt)
    rng = np.random.default_rng(51)
    n = 58_720_256
    x = workloads.normal(n, 51, 3.0, fmt)
    dy = workloads.normal(n, 52, 1.0, fmt)
    xd, dyd = to_dev(x, dt), to_dev(dy, dt)
    out = torch.empty_like(xd)
    B.poly_act_fwd(B.POLY_SILU, dt, xd, out, n)
    assert _equal_bits(out, _apply_lut(s_op, xd))
    B.poly_act_bwd(B.POLY_SILU, dt, xd, dyd, out, n)
    assert _equal_bits(out, _rn_mul(dyd, _apply_lut(d_op, xd)))
    smp = np.unique(np.concatenate([rng.integers(0, n, 1 << 18), np.arange(n - 64, n)]))
    assert np.array_equal(from_dev(out[torch.from_numpy(smp).to(DEV)]),
                          backward(d_op, x[smp], dy[smp]))
    del x, dy, xd, dyd, out
    rows, cols = 24_576, 1_280
    m = rows * cols
    g = workloads.normal(m, 53, 1.5, fmt)
    u = workloads.normal(m, 54, 1.5, fmt)
    dy = workloads.normal(m, 55, 1.0, fmt)
    gd, ud, dyd = (to_dev(a, dt).view(rows, cols) for a in (g, u, dy))
    y, dg, du = torch.empty_like(gd), torch.empty_like(gd), torch.empty_like(gd)
    B.poly_swiglu_fwd(dt, gd, ud, y)
    B.poly_swiglu_bwd(dt, gd, ud, dyd, dg, du)
    sg, sdg = _apply_lut(s_op, gd), _apply_lut(d_op, gd)
    assert _equal_bits(y, _rn_mul(sg, ud))
    assert _equal_bits(dg, _rn_mul(_rn_mul(dyd, ud), sdg))
    assert _equal_bits(du, _rn_mul(dyd, sg))
    smp = np.unique(np.concatenate([rng.integers(0, m, 1 << 18), np.arange(m - cols, m)]))
    sd = torch.from_numpy(smp).to(DEV)
    assert np.array_equal(from_dev(y.view(-1)[sd]), swiglu_forward(s_op, g[smp], u[smp]))
    wdg, wdu = swiglu_backward(s_op, d_op, g[smp], u[smp], dy[smp])
    assert np.array_equal(from_dev(dg.view(-1)[sd]), wdg)
    assert np.array_equal(from_dev(du.view(-1)[sd]), wdu)


def test_ragged_swiglu_full_size_sampled():
    """16,384 tokens x top-8 over 64 experts: Zipf(1.1) segments summing to
    131,072 rows of 2048; the offsets stay on the device.  Rows past the last
    offset (a larger capacity) must stay untouched."""
    dt = B.POLY_BF16
    s_op, d_op = _swiglu_ops(dt)
    g, u, dy, seg = workloads.ragged_swiglu("bf16")
    rows, cols = g.shape
    cap = rows + 3000
    pad = np.zeros((cap - rows, cols), np.uint16)
    gd = to_dev(np.concatenate([g, pad]), dt).view(cap, cols)
    ud = to_dev(np.concatenate([u, pad]), dt).view(cap, cols)
    dyd = to_dev(np.concatenate([dy, pad]), dt).view(cap, cols)
    segd = torch.from_numpy(seg).to(DEV)
    status = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    fill = lambda: torch.full((cap, cols), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
    y, dg, du = fill(), fill(), fill()
    B.poly_swiglu_fwd_ragged(dt, gd, ud, y, segd, status=status)
    assert int(status.item()) == 0
    B.poly_swiglu_bwd_ragged(dt, gd, ud, dyd, dg, du, segd, status=status)
    assert int(status.item()) == 0
    for t in (y, dg, du):
        assert bool((t.view(torch.int16)[rows:] == 0x5A5A).all())
    n = rows * cols
    rng = np.random.default_rng(41)
    # every segment boundary row, plus random elements
    bnd = np.concatenate([np.arange(max(0, b - 1) * cols, min(rows, b + 1) * cols) for b in seg[1:-1]])
    s = np.unique(np.concatenate([rng.integers(0, n, 1 << 20), bnd, np.arange(n - cols, n)]))
    sd = torch.from_numpy(s).to(DEV)
    gf, uf, dyf = g.reshape(-1), u.reshape(-1), dy.reshape(-1)
    assert np.array_equal(from_dev(y.view(-1)[sd]), swiglu_forward(s_op, gf[s], uf[s]))
    wdg, wdu = swiglu_backward(s_op, d_op, gf[s], uf[s], dyf[s])
    assert np.array_equal(from_dev(dg.view(-1)[sd]), wdg)
    assert np.array_equal(from_dev(du.view(-1)[sd]), wdu)
    # every row of every segment through the oracle's exhaustive tables
    gs, us, dys = gd[:rows], ud[:rows], dyd[:rows]
    sg, sdg = _apply_lut(s_op, gs), _apply_lut(d_op, gs)
    assert _equal_bits(y[:rows], _rn_mul(sg, us))
    assert _equal_bits(dg[:rows], _rn_mul(_rn_mul(dys, us), sdg))
    assert _equal_bits(du[:rows], _rn_mul(dys, sg))


def test_ragged_launch_shape_switch_sizes():
    """Ragged calls take the dense kernel's launch shapes by row capacity
    (one chunk per thread up to 8 blocks per SM, two up to 16, one above, for
    the two-input forward): capacities on both sides of each edge, segments
    covering all but the last rows; every row inside against the oracle's
    tables and the rows past the last offset untouched, forward under both
    SwiGLU rules and backward (BF16, 2048 columns)."""
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    cols = 2048
    dt = B.POLY_BF16
    s_op, d_op = _swiglu_ops(dt)
    sig = oracle_program(B.POLY_SIGMOID, B.POLY_FWD, dt)
    rng = np.random.default_rng(89)
    for edge in (8 * sms * 256 * 8, 16 * sms * 256 * 2 * 8):
        for cap in (edge // cols - 1, edge // cols, edge // cols + 1):
            rows = cap - 5
            segd = torch.from_numpy(np.linspace(0, rows, 9).astype(np.int32)).to(DEV)
            gd, ud, dyd = (to_dev(_rand_bits(rng, cap * cols, "bf16"), dt).view(cap, cols)
                           for _ in range(3))
            fill = lambda: torch.full((cap, cols), 0x5A5A, dtype=torch.int16,
                                      device=DEV).view(TDT[dt])
            gs, us, dys = gd[:rows], ud[:rows], dyd[:rows]
            sg = _apply_lut(s_op, gs)
            y = fill()
            B.poly_swiglu_fwd_ragged(dt, gd, ud, y, segd)
            assert _equal_bits(y[:rows], _rn_mul(sg, us)), (edge, cap)
            y2 = fill()
            B.poly_swiglu_fwd_ragged_v(B.POLY_SWIGLU_SIGMOID, dt, gd, ud, y2, segd)
            assert _equal_bits(y2[:rows], _rn_mul(_rn_mul(gs, _apply_lut(sig, gs)), us)), (edge, cap)
            dg, du = fill(), fill()
            B.poly_swiglu_bwd_ragged(dt, gd, ud, dyd, dg, du, segd)
            assert _equal_bits(dg[:rows], _rn_mul(_rn_mul(dys, us), _apply_lut(d_op, gs))), (edge, cap)
            assert _equal_bits(du[:rows], _rn_mul(dys, sg)), (edge, cap)
            for t in (y, y2, dg, du):
                assert bool((t.view(torch.int16)[rows:] == 0x5A5A).all()), (edge, cap)


@pytest.mark.parametrize("cols", [24, 21])
@pytest.mark.parametrize("dt", DTS)
def test_ragged_small_every_element_and_status(dt, cols):
    """cols = 24: the dense kernel's ragged mode (rows start on 16-byte
    boundaries); cols = 21: the general kernel (scalar head and tail)."""
    fmt = FMT[dt]
    s_op, d_op = _swiglu_ops(dt)
    rng = np.random.default_rng(51)
    cap = 50
    seg = np.array([0, 3, 3, 10, 31, 40], dtype=np.int32)
    g = _rand_bits(rng, cap * cols, fmt).reshape(cap, cols)
    u = _rand_bits(rng, cap * cols, fmt).reshape(cap, cols)
    gd, ud = to_dev(g, dt), to_dev(u, dt)
    y = torch.full((cap, cols), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.poly_swiglu_fwd_ragged(dt, gd, ud, y, torch.from_numpy(seg).to(DEV), status=status)
    got = from_dev(y).reshape(cap, cols)
    assert np.array_equal(got[:40], swiglu_forward(s_op, g[:40], u[:40]))
    assert np.all(got[40:] == 0x5A5A) and int(status.item()) == 0
    # non-monotone offsets (still inside the capacity): status 1
    bad = torch.from_numpy(np.array([0, 5, 2, 10, 31, 40], dtype=np.int32)).to(DEV)
    B.poly_swiglu_fwd_ragged(dt, gd, ud, y, bad, status=status)
    assert int(status.item()) == 1
    # last offset beyond the capacity: clamped to it, status 1
    over = torch.from_numpy(np.array([0, 3, 3, 10, 31, 60], dtype=np.int32)).to(DEV)
    y2 = torch.empty_like(y)
    B.poly_swiglu_fwd_ragged(dt, gd, ud, y2, over, status=status)
    assert int(status.item()) == 1
    assert np.array_equal(from_dev(y2).reshape(cap, cols), swiglu_forward(s_op, g, u))
    # first offset above 0: rows [2, 40) are processed, rows before and after untouched, status 1
    late = torch.from_numpy(np.array([2, 3, 3, 10, 31, 40], dtype=np.int32)).to(DEV)
    y3 = torch.full((cap, cols), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
    B.poly_swiglu_fwd_ragged(dt, gd, ud, y3, late, status=status)
    assert int(status.item()) == 1
    got3 = from_dev(y3).reshape(cap, cols)
    assert np.array_equal(got3[2:40], swiglu_forward(s_op, g[2:40], u[2:40]))
    assert np.all(got3[:2] == 0x5A5A) and np.all(got3[40:] == 0x5A5A)


# ---------------------------------------------------------------- controls

@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("fn,d", PROGRAMS)
def test_mufu_controls_accuracy(fn, d, dt):
    """The special-function-unit controls approximate the true function to
    within two target-format ulps (plus the FP32 approximation error)."""
    fmt = FMT[dt]
    x = _rand_bits(np.random.default_rng(2), 1 << 16, fmt)
    x = x[tf.finite_mask(x, fmt)]
    x = x[np.abs(tf.decode(x, fmt)) < 60]
    xd = to_dev(x, dt)
    out = torch.empty_like(xd)
    f = ref.function(fn, d)(tf.decode(x, fmt))
    if d == B.POLY_FWD:
        B.poly_ctrl_act_fwd(fn, dt, xd, out)
    else:
        ones = to_dev(tf.from_f64(np.ones(x.size), fmt), dt)
        B.poly_ctrl_act_bwd(fn, dt, xd, ones, out)
    y = tf.decode(from_dev(out), fmt)
    ulp = np.spacing(np.abs(f).astype(np.float16 if fmt == "f16" else np.float32))
    ulp = ulp.astype(np.float64) * (1 if fmt == "f16" else 2.0 ** 16)
    tol = 2 * ulp + 1e-3 * (1.0 + np.abs(f))
    assert np.all(np.abs(y - f) <= tol), (fn, d, np.max(np.abs(y - f)))


@pytest.mark.parametrize("dt", DTS)
def test_mufu_swiglu_controls(dt):
    fmt = FMT[dt]
    rng = np.random.default_rng(8)
    g = _rand_bits(rng, 64 * 256, fmt)
    g = np.where(tf.finite_mask(g, fmt) & (np.abs(tf.decode(g, fmt)) < 30), g, np.uint16(0)).reshape(64, 256)
    u = tf.from_f64(rng.normal(0, 1, g.size), fmt).reshape(64, 256)
    gd, ud = to_dev(g, dt), to_dev(u, dt)
    y = torch.empty_like(gd)
    B.poly_ctrl_swiglu_fwd(dt, gd, ud, y)
    gv, uv = tf.decode(g, fmt), tf.decode(u, fmt)
    want = ref.silu(gv) * uv
    got = tf.decode(from_dev(y).reshape(64, 256), fmt)
    assert np.max(np.abs(got - want) / np.maximum(np.abs(want), 1)) < 2e-2
    dg, du = torch.empty_like(gd), torch.empty_like(gd)
    B.poly_ctrl_swiglu_bwd(dt, gd, ud, ud, dg, du)
    wdg = uv * uv * ref.dsilu(gv)
    wdu = uv * ref.silu(gv)
    assert np.max(np.abs(tf.decode(from_dev(dg).reshape(64, 256), fmt) - wdg) / np.maximum(np.abs(wdg), 1)) < 2e-2
    assert np.max(np.abs(tf.decode(from_dev(du).reshape(64, 256), fmt) - wdu) / np.maximum(np.abs(wdu), 1)) < 2e-2


@pytest.mark.parametrize("dt", DTS)
def test_host_memory_operands(dt):
    """On GB300 the GPU reaches pinned host memory over NVLink-C2C: inputs
    and outputs may live there, with bit-identical results."""
    fmt = FMT[dt]
    x = _rand_bits(np.random.default_rng(13), 300_001, fmt)
    op = oracle_program(B.POLY_SILU, B.POLY_FWD, dt)
    xh = torch.from_numpy(x.view(np.int16)).pin_memory().view(TDT[dt])
    yh = torch.full((x.size,), 0x5A5A, dtype=torch.int16).pin_memory().view(TDT[dt])
    B.poly_act_fwd(B.POLY_SILU, dt, xh, yh, x.size)
    torch.cuda.synchronize()
    assert np.array_equal(yh.view(torch.int16).numpy().view(np.uint16), forward(op, x))
    xd = to_dev(x, dt)
    yh2 = torch.empty(x.size, dtype=torch.int16).pin_memory().view(TDT[dt])
    B.poly_act_fwd(B.POLY_SILU, dt, xd, yh2, x.size)
    torch.cuda.synchronize()
    assert np.array_equal(yh2.view(torch.int16).numpy().view(np.uint16), forward(op, x))


def _strided_view(buf, off, rows, cols, ld):
    return torch.as_strided(buf, (rows, cols), (ld, 1), storage_offset=off)


@pytest.mark.parametrize("H", [72, 21])
@pytest.mark.parametrize("dt", DTS)
def test_swiglu_fused_gate_up_halves(dt, H):
    """Gate and up as the two halves of one [T, 2H] projection output, and
    dg, du written into the two halves of one [T, 2H] gradient buffer
    (leading dimension 2H everywhere): every element against the oracle."""
    fmt = FMT[dt]
    s_op, d_op = _swiglu_ops(dt)
    rng = np.random.default_rng(91)
    T = 37
    gu = _rand_bits(rng, T * 2 * H, fmt).reshape(T, 2 * H)
    dy = _rand_bits(rng, T * H, fmt).reshape(T, H)
    gud = to_dev(gu, dt).view(T, 2 * H)
    y = torch.empty((T, H), dtype=TDT[dt], device=DEV)
    B.poly_swiglu_fwd(dt, gud[:, :H], gud[:, H:], y)
    assert np.array_equal(from_dev(y).reshape(T, H), swiglu_forward(s_op, gu[:, :H], gu[:, H:]))
    dgu = torch.full((T, 2 * H), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
    B.poly_swiglu_bwd(dt, gud[:, :H], gud[:, H:], to_dev(dy, dt).view(T, H), dgu[:, :H], dgu[:, H:])
    wdg, wdu = swiglu_backward(s_op, d_op, gu[:, :H], gu[:, H:], dy)
    got = from_dev(dgu).reshape(T, 2 * H)
    assert np.array_equal(got[:, :H], wdg) and np.array_equal(got[:, H:], wdu)


@pytest.mark.parametrize("T,H", [(2100, 2048), (8200, 8192)])
def test_swiglu_fused_halves_large_every_element(T, H):
    """Gate / up and dg / du as halves of [T, 2H] buffers on both sides of the
    size at which the backward leaves the dense rows mode for the strided
    kernel (2^23 chunks of 8: T = 2100, H = 2048 gives 537,600 chunks, below;
    T = 8200, H = 8192 gives 8,396,800, above), every element through the
    oracle's exhaustive tables, products rounded once."""
    dt = B.POLY_BF16
    s_op, d_op = _swiglu_ops(dt)
    rng = np.random.default_rng(97)
    gu = to_dev(_rand_bits(rng, T * 2 * H, "bf16"), dt).view(T, 2 * H)
    dyd = to_dev(_rand_bits(rng, T * H, "bf16"), dt).view(T, H)
    g, u = gu[:, :H], gu[:, H:]
    y = torch.empty((T, H), dtype=TDT[dt], device=DEV)
    B.poly_swiglu_fwd(dt, g, u, y)
    dgu = torch.empty_like(gu)
    B.poly_swiglu_bwd(dt, g, u, dyd, dgu[:, :H], dgu[:, H:])
    gc, uc = g.contiguous(), u.contiguous()
    sg, sdg = _apply_lut(s_op, gc), _apply_lut(d_op, gc)
    assert _equal_bits(y, _rn_mul(sg, uc))
    assert _equal_bits(dgu[:, :H].contiguous(), _rn_mul(_rn_mul(dyd, uc), sdg))
    assert _equal_bits(dgu[:, H:].contiguous(), _rn_mul(dyd, sg))


def test_swiglu_random_layouts_every_element():
    """48 seeded cases: rows 1-40, cols 1-70, a leading dimension and an
    element offset of its own for every stream (0-13 padding, 0-7 elements
    of misalignment), both formats, both SwiGLU rules, forward and backward;
    every element against the oracle, and nothing outside an output's view
    is written."""
    from oracle.replay import swiglu_sigmoid_backward, swiglu_sigmoid_forward
    rng = np.random.default_rng(71)
    for case in range(48):
        dt = DTS[case % 2]
        fmt = FMT[dt]
        sig_rule = (case // 2) % 2 == 1
        rows, cols = int(rng.integers(1, 41)), int(rng.integers(1, 71))
        lds = [cols + int(rng.integers(0, 14)) for _ in range(6)]       # g, u, y, dy, dg, du
        offs = [int(rng.integers(0, 8)) for _ in range(6)]
        bufs = [torch.full((o + rows * l + 8,), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
                for o, l in zip(offs, lds)]
        vals = [_rand_bits(rng, rows * cols, fmt).reshape(rows, cols) for _ in range(3)]
        views = [_strided_view(b, o, rows, cols, l) for b, o, l in zip(bufs, offs, lds)]
        for v, a in zip((views[0], views[1], views[3]), vals):
            v.copy_(to_dev(a, dt).view(rows, cols))
        g, u, dy = vals
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_SIGMOID if sig_rule else B.POLY_SWIGLU_DIRECT)
        try:
            B.poly_swiglu_fwd(dt, views[0], views[1], views[2])
            B.poly_swiglu_bwd(dt, views[0], views[1], views[3], views[4], views[5])
        finally:
            B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)
        if sig_rule:
            sig = oracle_program(B.POLY_SIGMOID, B.POLY_FWD, dt)
            wy = swiglu_sigmoid_forward(sig, g, u)
            wdg, wdu = swiglu_sigmoid_backward(sig, g, u, dy)
        else:
            s_op, d_op = _swiglu_ops(dt)
            wy = swiglu_forward(s_op, g, u)
            wdg, wdu = swiglu_backward(s_op, d_op, g, u, dy)
        where = (case, rows, cols, lds, offs)
        for k, want in ((2, wy), (4, wdg), (5, wdu)):
            assert np.array_equal(from_dev(views[k]).reshape(rows, cols), want), where
            full = from_dev(bufs[k]).copy()
            idx = offs[k] + np.arange(rows)[:, None] * lds[k] + np.arange(cols)[None, :]
            full[idx.reshape(-1)] = 0x5A5A
            assert np.all(full == 0x5A5A), where


@pytest.fixture
def sigmoid_swiglu():
    B.poly_set_swiglu_variant(B.POLY_SWIGLU_SIGMOID)
    try:
        yield
    finally:
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)


@pytest.mark.parametrize("dt", DTS)
def test_swiglu_sigmoid_rule_every_element(dt, sigmoid_swiglu):
    """The paper's deployed B1/B4 rule, dense, strided and ragged layouts."""
    from oracle.replay import swiglu_sigmoid_backward, swiglu_sigmoid_forward
    fmt = FMT[dt]
    sig = oracle_program(B.POLY_SIGMOID, B.POLY_FWD, dt)
    rng = np.random.default_rng(61)
    for rows, cols, pad in [(1, 1, 0), (13, 1003, 0), (64, 2048, 0), (37, 2048, 8), (9, 1001, 5)]:
        W = cols + pad
        g = _rand_bits(rng, rows * W, fmt).reshape(rows, W)
        u = _rand_bits(rng, rows * W, fmt).reshape(rows, W)
        dy = _rand_bits(rng, rows * W, fmt).reshape(rows, W)
        gd, ud, dyd = (to_dev(a, dt).view(rows, W)[:, :cols] for a in (g, u, dy))
        gg, uu, dd = g[:, :cols], u[:, :cols], dy[:, :cols]
        y = torch.empty(rows, cols, dtype=TDT[dt], device=DEV)
        B.poly_swiglu_fwd(dt, gd, ud, y)
        assert np.array_equal(from_dev(y).reshape(rows, cols), swiglu_sigmoid_forward(sig, gg, uu))
        dg = torch.empty_like(y)
        du = torch.empty_like(y)
        B.poly_swiglu_bwd(dt, gd, ud, dyd, dg, du)
        wdg, wdu = swiglu_sigmoid_backward(sig, gg, uu, dd)
        assert np.array_equal(from_dev(dg).reshape(rows, cols), wdg)
        assert np.array_equal(from_dev(du).reshape(rows, cols), wdu)
    cols, cap = 40, 30
    seg = torch.from_numpy(np.array([0, 7, 7, 21, 26], dtype=np.int32)).to(DEV)
    g = _rand_bits(rng, cap * cols, fmt).reshape(cap, cols)
    u = _rand_bits(rng, cap * cols, fmt).reshape(cap, cols)
    dy = _rand_bits(rng, cap * cols, fmt).reshape(cap, cols)
    dg = torch.full((cap, cols), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
    du = torch.full((cap, cols), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
    B.poly_swiglu_bwd_ragged(dt, to_dev(g, dt).view(cap, cols), to_dev(u, dt).view(cap, cols),
                             to_dev(dy, dt).view(cap, cols), dg, du, seg)
    wdg, wdu = swiglu_sigmoid_backward(sig, g[:26], u[:26], dy[:26])
    assert np.array_equal(from_dev(dg).reshape(cap, cols)[:26], wdg)
    assert np.array_equal(from_dev(du).reshape(cap, cols)[:26], wdu)
    assert np.all(from_dev(dg).reshape(cap, cols)[26:] == 0x5A5A)


def test_swiglu_sigmoid_rule_dense_full_size_sampled(sigmoid_swiglu):
    from oracle.replay import swiglu_sigmoid_backward, swiglu_sigmoid_forward
    dt = B.POLY_BF16
    sig = oracle_program(B.POLY_SIGMOID, B.POLY_FWD, dt)
    g, u, dy = workloads.dense_swiglu("bf16")
    rows, cols = g.shape
    gd, ud, dyd = (to_dev(a, dt).view(rows, cols) for a in (g, u, dy))
    y, dg, du = torch.empty_like(gd), torch.empty_like(gd), torch.empty_like(gd)
    B.poly_swiglu_fwd(dt, gd, ud, y)
    B.poly_swiglu_bwd(dt, gd, ud, dyd, dg, du)
    n = g.size
    s = np.unique(np.random.default_rng(71).integers(0, n, 1 << 20))
    sd = torch.from_numpy(s).to(DEV)
    gf, uf, dyf = g.reshape(-1), u.reshape(-1), dy.reshape(-1)
    assert np.array_equal(from_dev(y.view(-1)[sd]), swiglu_sigmoid_forward(sig, gf[s], uf[s]))
    wdg, wdu = swiglu_sigmoid_backward(sig, gf[s], uf[s], dyf[s])
    assert np.array_equal(from_dev(dg.view(-1)[sd]), wdg)
    assert np.array_equal(from_dev(du.view(-1)[sd]), wdu)


# ------------------------------------------------- softcap, derived programs

@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("alpha", [1.0, 30.0, 50.0])
def test_softcap_exhaustive(dt, alpha):
    """alpha tanh(x / alpha) forward and tanh'(x / alpha) backward over every
    input pattern, bit for bit."""
    from oracle.replay import softcap_backward, softcap_forward
    fmt = FMT[dt]
    tp = oracle_program(B.POLY_TANH, B.POLY_FWD, dt)
    dp = oracle_program(B.POLY_TANH, B.POLY_BWD, dt)
    x = X_ALL
    dy = _rand_bits(np.random.default_rng(29), x.size, fmt)
    xd, dyd = to_dev(x, dt), to_dev(dy, dt)
    out = torch.empty_like(xd)
    B.poly_softcap_fwd(dt, alpha, xd, out)
    assert np.array_equal(from_dev(out), softcap_forward(tp, alpha, x))
    B.poly_softcap_bwd(dt, alpha, xd, dyd, out)
    assert np.array_equal(from_dev(out), softcap_backward(dp, alpha, x, dy))


def test_softcap_full_size_every_element():
    """alpha = 30 on the bench's 268,435,456-element FP16 tensors: the forward
    through the oracle's exhaustive table of softcap(x); the backward as dy
    times the tabulated tanh'(x * (1/alpha)), each product rounded once (a
    product of two FP16 values is exact in FP32)."""
    from oracle.replay import softcap_backward, softcap_forward
    dt, alpha = B.POLY_F16, 30.0
    tp = oracle_program(B.POLY_TANH, B.POLY_FWD, dt)
    dp = oracle_program(B.POLY_TANH, B.POLY_BWD, dt)
    x, dy = workloads.isolated_hbm("f16")
    xd, dyd = to_dev(x, dt), to_dev(dy, dt)
    del x, dy
    out = torch.empty_like(xd)
    idx = (xd.view(torch.int16).to(torch.int32) & 0xFFFF).long()
    B.poly_softcap_fwd(dt, alpha, xd, out)
    lut_f = torch.from_numpy(softcap_forward(tp, alpha, X_ALL).view(np.int16)).to(DEV)
    assert _equal_bits(out, lut_f[idx].view(torch.float16))
    B.poly_softcap_bwd(dt, alpha, xd, dyd, out)
    ones = np.full(X_ALL.size, 0x3C00, dtype=np.uint16)          # dy = 1 tabulates the factor
    lut_d = torch.from_numpy(softcap_backward(dp, alpha, X_ALL, ones).view(np.int16)).to(DEV)
    assert _equal_bits(out, _rn_mul(dyd, lut_d[idx].view(torch.float16)))


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("fn,D", [(B.POLY_TANH, 4), (B.POLY_SIGMOID, 3)])
def test_derived_program_backward_exhaustive(dt, fn, D):
    """The differentiated forward program installed as the backward program
    (degree 3 for tanh, degree 2 for sigmoid), through poly_act_bwd and, for
    tanh, the softcap backward."""
    from oracle.replay import derive, softcap_backward
    fmt = FMT[dt]
    fwd = B.poly_get_program(fn, B.POLY_FWD, dt)
    assert fwd.degree == D
    d = B.poly_derive_program(fwd)
    od = derive(oracle_program(fn, B.POLY_FWD, dt))
    assert d.coefficients() == list(od.coef)
    B.poly_set_program(d)
    try:
        x = X_ALL
        dy = _rand_bits(np.random.default_rng(31), x.size, fmt)
        xd, dyd = to_dev(x, dt), to_dev(dy, dt)
        out = torch.empty_like(xd)
        B.poly_act_bwd(fn, dt, xd, dyd, out)
        assert np.array_equal(from_dev(out), backward(od, x, dy))
        if fn == B.POLY_TANH:
            B.poly_softcap_bwd(dt, 30.0, xd, dyd, out)
            assert np.array_equal(from_dev(out), softcap_backward(od, 30.0, x, dy))
    finally:
        B.poly_reset_programs()


def test_derived_programs_every_degree():
    """Forward programs of degree 3-6 (sigmoid centred-odd, tanh odd) in both
    formats, differentiated by the library and by the oracle into even
    programs of degree 2-5: equal coefficients, and the backward kernel
    equals the oracle over every input."""
    from oracle import fit
    from oracle.replay import derive
    rng = np.random.default_rng(33)
    try:
        for dt in DTS:
            fmt = FMT[dt]
            xd = to_dev(X_ALL, dt)
            dy = _rand_bits(rng, X_ALL.size, fmt)
            dyd = to_dev(dy, dt)
            out = torch.empty_like(xd)
            for fn in (B.POLY_SIGMOID, B.POLY_TANH):
                for D in (3, 4, 5, 6):
                    fwd = B.poly_fit(fn, B.POLY_FWD, dt, D)
                    d = B.poly_derive_program(fwd)
                    od = derive(fit.make_program(fn, B.POLY_FWD, fmt, D, fwd.li, fwd.lc,
                                                 fwd.coefficients()))
                    assert d.degree == D - 1 and d.coefficients() == list(od.coef), (fn, D)
                    B.poly_set_program(d)
                    B.poly_act_bwd(fn, dt, xd, dyd, out)
                    assert np.array_equal(from_dev(out), backward(od, X_ALL, dy)), (fn, fmt, D)
    finally:
        B.poly_reset_programs()


# ------------------------------------------------------------------- exp2

def _exp2_inputs():
    rng = np.random.default_rng(41)
    dense = rng.uniform(-130, 130, 1 << 22).astype(np.float32)
    with np.errstate(invalid="ignore"):                                     # NaN payloads
        halfs = tf.all_patterns().view(np.float16).astype(np.float32)       # every FP16 value
    grid = (np.arange(-260, 261) / 2).astype(np.float32)                    # integers, halves
    near = np.nextafter(grid, np.float32(np.inf)).astype(np.float32)
    near2 = np.nextafter(grid, np.float32(-np.inf)).astype(np.float32)
    sp = np.array([np.nan, np.inf, -np.inf, 0.0, -0.0, 1e-30, -1e-30, 127.999, 128.0, 1e30,
                   -1e30, -126.0, -126.5, -125.999], dtype=np.float32)
    return np.concatenate([dense, halfs, grid, near, near2, sp])


@pytest.mark.parametrize("core", [B.POLY_EXP2_D1, B.POLY_EXP2_PWL2, B.POLY_EXP2_D2,
                                  B.POLY_EXP2_D3])
def test_exp2_cores_bit_exact(core):
    from oracle import exp2 as e2
    x = _exp2_inputs()
    xd = torch.from_numpy(x).to(DEV)
    y = torch.empty_like(xd)
    B.poly_exp2(core, xd, y)
    got = y.cpu().numpy().view(np.uint32)
    want = e2.exp2_replay(e2.VARIANTS[core], x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[i]), hex(got[i]), hex(want[i])) for i in bad[:6]]
    # unaligned start and odd length: scalar head and tail
    y2 = torch.empty(x.size + 3, dtype=torch.float32, device=DEV)
    B.poly_exp2(core, xd[1:], y2[2:2 + x.size - 1], x.size - 1)
    assert np.array_equal(y2[2:2 + x.size - 1].cpu().numpy().view(np.uint32), want[1:])


@pytest.mark.parametrize("core", [B.POLY_EXP2_D1, B.POLY_EXP2_PWL2, B.POLY_EXP2_D2,
                                  B.POLY_EXP2_D3])
def test_exp2_full_size_sampled(core):
    """2^27 FP32 elements, x ~ U[-60, 10] (the bench's case, 512 MiB per
    tensor): 2^20 sampled outputs plus the first and last 4,096, element by
    element against the oracle."""
    from oracle import exp2 as e2
    n = 1 << 27
    x = np.random.default_rng(7).uniform(-60, 10, n).astype(np.float32)
    xd = torch.from_numpy(x).to(DEV)
    y = torch.empty_like(xd)
    B.poly_exp2(core, xd, y)
    torch.cuda.synchronize()
    idx = np.unique(np.concatenate([np.random.default_rng(8).integers(0, n, 1 << 20),
                                    np.arange(4096), np.arange(n - 4096, n)]))
    got = y[torch.from_numpy(idx).to(DEV)].cpu().numpy().view(np.uint32)
    want = e2.exp2_replay(e2.VARIANTS[core], x[idx])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(x[idx[i]]), hex(got[i]), hex(want[i])) for i in bad[:6]]


def test_exp2_above_2_31_elements():
    """2^31 + 4,099 FP32 elements cycling through 65,536 values of
    U[-60, 10]: every element equals the oracle's value for its input
    (checked in slices of 2^28), tail included."""
    from oracle import exp2 as e2
    n = (1 << 31) + 4099
    pat = np.random.default_rng(17).uniform(-60, 10, 65536).astype(np.float32)
    want = torch.from_numpy(e2.exp2_replay("D2", pat).view(np.int32)).to(DEV)
    pd = torch.from_numpy(pat).to(DEV)
    x = torch.empty(n, dtype=torch.float32, device=DEV)
    full = n // 65536
    x[:full * 65536].view(full, 65536).copy_(pd.expand(full, 65536))
    x[full * 65536:] = pd[:n - full * 65536]
    y = torch.empty_like(x)
    B.poly_exp2(B.POLY_EXP2_D2, x, y)
    yi = y.view(torch.int32)
    rows = 1 << 12
    for r0 in range(0, full, rows):
        r1 = min(full, r0 + rows)
        assert bool((yi[r0 * 65536:r1 * 65536].view(r1 - r0, 65536) == want[None, :]).all()), r0
    assert torch.equal(yi[full * 65536:], want[:n - full * 65536])
    del x, y, yi
    torch.cuda.empty_cache()


def test_exp2_mufu_control_accuracy():
    x = np.random.default_rng(43).uniform(-120, 120, 1 << 20).astype(np.float32)
    xd = torch.from_numpy(x).to(DEV)
    y = torch.empty_like(xd)
    B.poly_ctrl_exp2(xd, y)
    rel = np.abs(y.cpu().numpy().astype(np.float64) / np.exp2(x.astype(np.float64)) - 1)
    assert rel.max() < 2e-6


# --------------------------------------------------------------------- RoPE

def _rope_case(rng, b, s, hq, hkv, d):
    q = tf.from_f64(rng.normal(0, 1, (b, s, hq, d)), "f16")
    k = tf.from_f64(rng.normal(0, 1, (b, s, hkv, d)), "f16")
    return q, k


@pytest.mark.parametrize("shape,pos", [((2, 37, 4, 2, 16), 0), ((1, 300, 3, 1, 128), 0),
                                       ((3, 5, 2, 0, 8), 123456), ((1, 64, 0, 2, 64), (1 << 32) - 64),
                                       ((2, 129, 8, 8, 128), 7)])
def test_rope_poly_bit_exact(shape, pos):
    from oracle import rope
    b, s, hq, hkv, d = shape
    rng = np.random.default_rng(sum(shape))
    q, k = _rope_case(rng, b, s, hq, hkv, d)
    delta = rope.turn_increments(d)
    dd = torch.from_numpy(delta.view(np.int32)).to(DEV)
    qd, kd = to_dev(q, 0), to_dev(k, 0)
    qo = torch.empty((b, hq, s, d), dtype=torch.float16, device=DEV)
    ko = torch.empty((b, hkv, s, d), dtype=torch.float16, device=DEV)
    B.poly_rope_fwd(B.POLY_ROPE_POLY, qd, kd, qo, ko, dd, batch=b, seq=s, hq=hq, hkv=hkv,
                    head_dim=d, pos_offset=pos)
    wq, wk = rope.rope_forward(q, k, delta, pos)
    assert np.array_equal(from_dev(qo).reshape(wq.shape), wq)
    assert np.array_equal(from_dev(ko).reshape(wk.shape), wk)
    # backward: gradients in [B, H, S, D] -> [B, S, H, D], rotated by -theta
    gq = torch.empty((b, s, hq, d), dtype=torch.float16, device=DEV)
    gk = torch.empty((b, s, hkv, d), dtype=torch.float16, device=DEV)
    B.poly_rope_bwd(B.POLY_ROPE_POLY, qo, ko, gq, gk, dd, batch=b, seq=s, hq=hq, hkv=hkv,
                    head_dim=d, pos_offset=pos)
    bq, bk = rope.rope_backward(wq, wk, delta, pos)
    assert np.array_equal(from_dev(gq).reshape(bq.shape), bq)
    assert np.array_equal(from_dev(gk).reshape(bk.shape), bk)
    # the cached-table variant, given the oracle's tables, applies the same rotation
    cs, sn = rope.tables(s, delta, pos)
    ct = torch.from_numpy(cs.view(np.int16)).to(DEV)
    st = torch.from_numpy(sn.view(np.int16)).to(DEV)
    qo2, ko2 = torch.empty_like(qo), torch.empty_like(ko)
    B.poly_rope_fwd(B.POLY_ROPE_TABLE, qd, kd, qo2, ko2, None, ct, st, batch=b, seq=s, hq=hq,
                    hkv=hkv, head_dim=d, pos_offset=pos)
    assert torch.equal(qo2.view(torch.int16), qo.view(torch.int16))
    assert torch.equal(ko2.view(torch.int16), ko.view(torch.int16))


def test_rope_random_shapes():
    """24 seeded random shapes -- batch 1-3, sequence 1-70, Hq 0-19, Hkv 0-9
    (so eight-head chunks straddle the Q / K boundary), head dimension 8-256,
    random position offsets -- forward and backward bit for bit, and the
    table variant fed the oracle's tables."""
    from oracle import rope
    rng = np.random.default_rng(123)
    for case in range(24):
        b, s = int(rng.integers(1, 4)), int(rng.integers(1, 71))
        hq, hkv = int(rng.integers(0, 20)), int(rng.integers(0, 10))
        if hq + hkv == 0:
            hq = 1
        d = 8 * int(rng.integers(1, 33))
        pos = int(rng.integers(0, (1 << 32) - s))
        q, k = _rope_case(rng, b, s, hq, hkv, d)
        delta = rope.turn_increments(d)
        dd = torch.from_numpy(delta.view(np.int32)).to(DEV)
        qd, kd = to_dev(q, 0), to_dev(k, 0)
        qo = torch.empty((b, hq, s, d), dtype=torch.float16, device=DEV)
        ko = torch.empty((b, hkv, s, d), dtype=torch.float16, device=DEV)
        dims = dict(batch=b, seq=s, hq=hq, hkv=hkv, head_dim=d, pos_offset=pos)
        B.poly_rope_fwd(B.POLY_ROPE_POLY, qd, kd, qo, ko, dd, **dims)
        wq, wk = rope.rope_forward(q, k, delta, pos)
        where = (case, b, s, hq, hkv, d, pos)
        assert np.array_equal(from_dev(qo).reshape(wq.shape), wq), where
        assert np.array_equal(from_dev(ko).reshape(wk.shape), wk), where
        gq = torch.empty((b, s, hq, d), dtype=torch.float16, device=DEV)
        gk = torch.empty((b, s, hkv, d), dtype=torch.float16, device=DEV)
        B.poly_rope_bwd(B.POLY_ROPE_POLY, qo, ko, gq, gk, dd, **dims)
        bq, bk = rope.rope_backward(wq, wk, delta, pos)
        assert np.array_equal(from_dev(gq).reshape(bq.shape), bq), where
        assert np.array_equal(from_dev(gk).reshape(bk.shape), bk), where
        cs, sn = rope.tables(s, delta, pos)
        qo2, ko2 = torch.empty_like(qo), torch.empty_like(ko)
        B.poly_rope_fwd(B.POLY_ROPE_TABLE, qd, kd, qo2, ko2, None,
                        torch.from_numpy(cs.view(np.int16)).to(DEV),
                        torch.from_numpy(sn.view(np.int16)).to(DEV), **dims)
        assert torch.equal(qo2.view(torch.int16), qo.view(torch.int16)), where
        assert torch.equal(ko2.view(torch.int16), ko.view(torch.int16)), where


def test_rope_mufu_variant_accuracy():
    from oracle import rope
    b, s, hq, hkv, d = 1, 512, 4, 2, 128
    rng = np.random.default_rng(5)
    q, k = _rope_case(rng, b, s, hq, hkv, d)
    dd = torch.from_numpy(rope.turn_increments(d).view(np.int32)).to(DEV)
    qo = torch.empty((b, hq, s, d), dtype=torch.float16, device=DEV)
    ko = torch.empty((b, hkv, s, d), dtype=torch.float16, device=DEV)
    B.poly_rope_fwd(B.POLY_ROPE_MUFU, to_dev(q, 0), to_dev(k, 0), qo, ko, dd, batch=b, seq=s,
                    hq=hq, hkv=hkv, head_dim=d)
    qv = tf.decode(q, "f16")
    z = qv[..., 0::2] + 1j * qv[..., 1::2]
    omega = 10000.0 ** (-2.0 * np.arange(d // 2) / d)
    zr = z * np.exp(1j * np.arange(s)[None, :, None, None] * omega)
    want = np.empty_like(qv)
    want[..., 0::2], want[..., 1::2] = zr.real, zr.imag
    got = tf.decode(from_dev(qo).reshape(b, hq, s, d), "f16").transpose(0, 2, 1, 3)
    assert np.max(np.abs(got - want)) < 2e-2


def test_rope_full_size_sampled():
    """B = 4, S = 4096, Hq = 32, Hkv = 8, D = 128 (the paper's GQA geometry at
    batch 4): sampled rows of every output head."""
    from oracle import rope
    b, s, hq, hkv, d = 4, 4096, 32, 8, 128
    rng = np.random.default_rng(11)
    qd = torch.randn((b, s, hq, d), generator=torch.Generator(device=DEV).manual_seed(1),
                     device=DEV, dtype=torch.float32).to(torch.float16)
    kd = torch.randn((b, s, hkv, d), generator=torch.Generator(device=DEV).manual_seed(2),
                     device=DEV, dtype=torch.float32).to(torch.float16)
    delta = rope.turn_increments(d)
    dd = torch.from_numpy(delta.view(np.int32)).to(DEV)
    qo = torch.empty((b, hq, s, d), dtype=torch.float16, device=DEV)
    ko = torch.empty((b, hkv, s, d), dtype=torch.float16, device=DEV)
    B.poly_rope_fwd(B.POLY_ROPE_POLY, qd, kd, qo, ko, dd)
    cs, sn = rope.tables(s, delta)
    for _ in range(64):
        bb, ss = int(rng.integers(0, b)), int(rng.integers(0, s))
        xq = from_dev(qd[bb, ss])                           # [Hq, D]
        want = rope.rotate(xq, cs[ss][None, :], sn[ss][None, :])
        assert np.array_equal(from_dev(qo[bb, :, ss, :]), want)
        xk = from_dev(kd[bb, ss])
        assert np.array_equal(from_dev(ko[bb, :, ss, :]), rope.rotate(xk, cs[ss][None, :], sn[ss][None, :]))


def test_rope_above_2_31_elements():
    """q of 2^31 + 2^25 elements (B = 1, S = 65,792, Hq = 256, D = 128, plus
    Hkv = 4), forward and backward: 64-bit element offsets in both layouts;
    sampled positions (the last ones included) against the oracle, a late
    position offset making the phases wrap."""
    from oracle import rope
    b, s, hq, hkv, d = 1, 65_792, 256, 4, 128
    assert b * s * hq * d > 1 << 31
    pos0 = 3_000_000_000
    rng = np.random.default_rng(12)
    gen = torch.Generator(device=DEV).manual_seed(3)
    qd = torch.randn((b, s, hq, d), generator=gen, device=DEV, dtype=torch.float32).to(torch.float16)
    kd = torch.randn((b, s, hkv, d), generator=gen, device=DEV, dtype=torch.float32).to(torch.float16)
    delta = rope.turn_increments(d)
    dd = torch.from_numpy(delta.view(np.int32)).to(DEV)
    qo = torch.empty((b, hq, s, d), dtype=torch.float16, device=DEV)
    ko = torch.empty((b, hkv, s, d), dtype=torch.float16, device=DEV)
    B.poly_rope_fwd(B.POLY_ROPE_POLY, qd, kd, qo, ko, dd, pos_offset=pos0)
    picks = sorted(set(int(v) for v in rng.integers(0, s, 24)) | {0, s - 1})
    for ss in picks:
        cs, sn = rope.tables(1, delta, pos0 + ss)
        assert np.array_equal(from_dev(qo[0, :, ss, :]), rope.rotate(from_dev(qd[0, ss]), cs, sn)), ss
        assert np.array_equal(from_dev(ko[0, :, ss, :]), rope.rotate(from_dev(kd[0, ss]), cs, sn)), ss
    gq = torch.empty_like(qd)
    gk = torch.empty_like(kd)
    B.poly_rope_bwd(B.POLY_ROPE_POLY, qo, ko, gq, gk, dd, pos_offset=pos0)
    for ss in picks:
        wq, wk = rope.rope_backward(from_dev(qo[:, :, ss:ss + 1, :]), from_dev(ko[:, :, ss:ss + 1, :]),
                                    delta, pos0 + ss)
        assert np.array_equal(from_dev(gq[:, ss:ss + 1]), wq), ss
        assert np.array_equal(from_dev(gk[:, ss:ss + 1]), wk), ss
    del qd, kd, qo, ko, gq, gk
    torch.cuda.empty_cache()


# ------------------------------------------------------- graphs and streams

def test_cuda_graph_capture_and_replay():
    """Calls captured into a CUDA graph (the launches, with programmatic
    dependent launch, become graph nodes) replay to exactly the oracle's
    values, also after the inputs are rewritten in place."""
    dt, fmt = B.POLY_F16, "f16"
    n = 1_000_003
    rng = np.random.default_rng(61)
    x0, x1 = _rand_bits(rng, n, fmt), _rand_bits(rng, n, fmt)
    dy = _rand_bits(rng, n, fmt)
    xd, dyd = to_dev(x0, dt), to_dev(dy, dt)
    y1, y2 = torch.empty_like(xd), torch.empty_like(xd)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                    # warm-up (program fits) outside capture
        B.poly_act_fwd(B.POLY_GELU, dt, xd, y1, n)
        B.poly_act_bwd(B.POLY_TANH, dt, xd, dyd, y2, n)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.poly_act_fwd(B.POLY_GELU, dt, xd, y1, n)
        B.poly_act_bwd(B.POLY_TANH, dt, xd, dyd, y2, n)
    gelu = oracle_program(B.POLY_GELU, B.POLY_FWD, dt)
    tanh_d = oracle_program(B.POLY_TANH, B.POLY_BWD, dt)
    for x in (x0, x1):
        xd.copy_(to_dev(x, dt))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(from_dev(y1), forward(gelu, x))
        assert np.array_equal(from_dev(y2), backward(tanh_d, x, dy))


def test_concurrent_streams():
    """Different programs launched on two streams at once each produce the
    oracle's values (kernels carry their program as a parameter; nothing is
    shared between launches)."""
    dt, fmt = B.POLY_BF16, "bf16"
    n = 3_000_017
    rng = np.random.default_rng(62)
    xa, xb = _rand_bits(rng, n, fmt), _rand_bits(rng, n, fmt)
    da, db = to_dev(xa, dt), to_dev(xb, dt)
    ya, yb = torch.empty_like(da), torch.empty_like(db)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    B.poly_get_program(B.POLY_SIGMOID, B.POLY_FWD, dt)
    B.poly_get_program(B.POLY_SILU, B.POLY_FWD, dt)
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(sa):
            B.poly_act_fwd(B.POLY_SIGMOID, dt, da, ya, n)
        with torch.cuda.stream(sb):
            B.poly_act_fwd(B.POLY_SILU, dt, db, yb, n)
    torch.cuda.synchronize()
    assert np.array_equal(from_dev(ya), forward(oracle_program(B.POLY_SIGMOID, B.POLY_FWD, dt), xa))
    assert np.array_equal(from_dev(yb), forward(oracle_program(B.POLY_SILU, B.POLY_FWD, dt), xb))


def test_host_threads_launch_concurrently():
    """Four host threads, each on its own stream with its own program, launch
    at the same time (the C calls overlap: ctypes releases the GIL); every
    output is the oracle's."""
    import threading
    dt, fmt = B.POLY_F16, "f16"
    n = 1_000_003
    rng = np.random.default_rng(63)
    jobs = []
    for fn, d in ((B.POLY_SIGMOID, 0), (B.POLY_TANH, 0), (B.POLY_GELU, 0), (B.POLY_SILU, 1)):
        x, dy = _rand_bits(rng, n, fmt), _rand_bits(rng, n, fmt)
        B.poly_get_program(fn, d, dt)
        jobs.append((fn, d, x, dy, to_dev(x, dt), to_dev(dy, dt)))
    outs = [torch.empty_like(j[4]) for j in jobs]
    torch.cuda.synchronize()
    errors = []

    def work(i):
        try:
            fn, d, _, _, xd, dyd = jobs[i]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(50):
                    if d == 0:
                        B.poly_act_fwd(fn, dt, xd, outs[i])
                    else:
                        B.poly_act_bwd(fn, dt, xd, dyd, outs[i])
            st.synchronize()
        except BaseException as e:
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    torch.cuda.synchronize()
    for (fn, d, x, dy, _, _), o in zip(jobs, outs):
        op = oracle_program(fn, d, dt)
        want = forward(op, x) if d == 0 else backward(op, x, dy)
        assert np.array_equal(from_dev(o), want), (fn, d)


# ------------------------------------------------------------------ autograd

def test_autograd_wrappers_match_direct_calls():
    """The torch.autograd wrappers return exactly what the C-ABI calls give."""
    from polynomial_activation_gb300 import ops
    from oracle import rope
    rng = np.random.default_rng(77)
    for dt in DTS:
        x = to_dev(_rand_bits(rng, 10_000, FMT[dt]), dt).requires_grad_(True)
        dy = to_dev(_rand_bits(rng, 10_000, FMT[dt]), dt)
        for name, f in [("sigmoid", ops.sigmoid), ("tanh", ops.tanh), ("silu", ops.silu),
                        ("gelu", ops.gelu)]:
            x.grad = None
            y = f(x)
            y.backward(dy)
            assert torch.equal(y.detach().view(torch.int16), ops.act_fwd(name, x.detach()).view(torch.int16))
            assert torch.equal(x.grad.view(torch.int16), ops.act_bwd(name, x.detach(), dy).view(torch.int16))
        g = to_dev(_rand_bits(rng, 64 * 256, FMT[dt]), dt).view(64, 256).requires_grad_(True)
        u = to_dev(_rand_bits(rng, 64 * 256, FMT[dt]), dt).view(64, 256).requires_grad_(True)
        dyy = to_dev(_rand_bits(rng, 64 * 256, FMT[dt]), dt).view(64, 256)
        y = ops.swiglu(g, u)
        y.backward(dyy)
        dg, du = ops.swiglu_bwd(g.detach(), u.detach(), dyy)
        assert torch.equal(g.grad.view(torch.int16), dg.view(torch.int16))
        assert torch.equal(u.grad.view(torch.int16), du.view(torch.int16))
        # a [batch, tokens, hidden] input is read as [batch * tokens, hidden]
        g3 = g.detach().reshape(4, 16, 256).requires_grad_(True)
        y3 = ops.swiglu(g3, u.detach().reshape(4, 16, 256))
        assert y3.shape == (4, 16, 256)
        assert torch.equal(y3.detach().reshape(64, 256).view(torch.int16),
                           ops.swiglu_fwd(g.detach(), u.detach()).view(torch.int16))
        # ragged: rows [0, 40) of a 64-row capacity; the rest stay zero
        seg = torch.tensor([0, 10, 10, 40], dtype=torch.int32, device=DEV)
        g.grad, u.grad = None, None
        y = ops.swiglu_ragged(g, u, seg)
        y.backward(dyy)
        dg, du = ops.swiglu_bwd(g.detach()[:40], u.detach()[:40], dyy[:40])
        assert torch.equal(y.detach()[:40].view(torch.int16),
                           ops.swiglu_fwd(g.detach()[:40], u.detach()[:40]).view(torch.int16))
        assert torch.equal(g.grad[:40].view(torch.int16), dg.view(torch.int16))
        assert torch.equal(u.grad[:40].view(torch.int16), du.view(torch.int16))
        for t in (y.detach(), g.grad, u.grad):
            assert not bool(t[40:].view(torch.int16).any())
        x.grad = None
        y = ops.softcap(x, 30.0)
        y.backward(dy)
        ref = torch.empty_like(dy)
        B.poly_softcap_bwd(dt, 30.0, x.detach(), dy, ref)
        assert torch.equal(x.grad.view(torch.int16), ref.view(torch.int16))
    q = torch.randn(2, 16, 4, 64, device=DEV).half().requires_grad_(True)
    k = torch.randn(2, 16, 2, 64, device=DEV).half().requires_grad_(True)
    delta = torch.from_numpy(rope.turn_increments(64).view(np.int32)).to(DEV)
    qo, ko = ops.rope(q, k, delta, 5)
    (qo.float().sum() + 2 * ko.float().sum()).backward()
    gq, gk = rope.rope_backward(np.ones((2, 4, 16, 64), np.uint16) * 0x3C00,
                                np.ones((2, 2, 16, 64), np.uint16) * 0x4000, rope.turn_increments(64), 5)
    assert np.array_equal(from_dev(q.grad).reshape(gq.shape), gq)
    assert np.array_equal(from_dev(k.grad).reshape(gk.shape), gk)


def test_wrappers_without_autograd_match_recorded_calls():
    """With no gradient to record (inputs without requires_grad, or under
    torch.no_grad / inference_mode) the wrappers call the kernels directly:
    same bits as the recorded path, no autograd node, ragged rows outside the
    range still zero."""
    from polynomial_activation_gb300 import ops
    from oracle import rope
    rng = np.random.default_rng(78)
    for dt in DTS:
        x = to_dev(_rand_bits(rng, 10_001, FMT[dt]), dt)
        g = to_dev(_rand_bits(rng, 64 * 256, FMT[dt]), dt).view(64, 256)
        u = to_dev(_rand_bits(rng, 64 * 256, FMT[dt]), dt).view(64, 256)
        seg = torch.tensor([0, 10, 10, 40], dtype=torch.int32, device=DEV)
        calls = [lambda a: ops.sigmoid(a), lambda a: ops.tanh(a), lambda a: ops.silu(a),
                 lambda a: ops.gelu(a), lambda a: ops.softcap(a, 30.0)]
        for f in calls:
            want = f(x.clone().requires_grad_(True))
            assert want.grad_fn is not None
            for mode in ("plain", "no_grad", "inference"):
                if mode == "plain":
                    got = f(x)
                elif mode == "no_grad":
                    with torch.no_grad():
                        got = f(x.clone().requires_grad_(True))
                else:
                    with torch.inference_mode():
                        got = f(x)
                assert got.grad_fn is None and not got.requires_grad
                assert torch.equal(got.view(torch.int16), want.detach().view(torch.int16)), mode
        want = ops.swiglu(g.clone().requires_grad_(True), u)
        got = ops.swiglu(g, u)
        assert got.grad_fn is None
        assert torch.equal(got.view(torch.int16), want.detach().view(torch.int16))
        with torch.no_grad():
            got3 = ops.swiglu(g.reshape(4, 16, 256), u.reshape(4, 16, 256))
        assert got3.shape == (4, 16, 256)
        assert torch.equal(got3.reshape(64, 256).view(torch.int16), got.view(torch.int16))
        want = ops.swiglu_ragged(g.clone().requires_grad_(True), u, seg)
        got = ops.swiglu_ragged(g, u, seg)
        assert got.grad_fn is None
        assert torch.equal(got.view(torch.int16), want.detach().view(torch.int16))
        assert not bool(got[40:].view(torch.int16).any())
    q = torch.randn(2, 16, 4, 64, device=DEV).half()
    k = torch.randn(2, 16, 2, 64, device=DEV).half()
    delta = torch.from_numpy(rope.turn_increments(64).view(np.int32)).to(DEV)
    wq, wk = ops.rope(q.clone().requires_grad_(True), k, delta, 7)
    gq, gk = ops.rope(q, k, delta, 7)
    assert gq.grad_fn is None and gk.grad_fn is None
    assert torch.equal(gq.view(torch.int16), wq.detach().view(torch.int16))
    assert torch.equal(gk.view(torch.int16), wk.detach().view(torch.int16))


@pytest.mark.parametrize("variant", [B.POLY_SWIGLU_DIRECT, B.POLY_SWIGLU_SIGMOID])
def test_swiglu_packed_gate_up_buffer(variant):
    """ops.swiglu_packed on a fused [.., 2H] gate-up buffer: the same bits as
    the separate-tensor SwiGLU, forward and backward, with the gradient
    written as one [.., 2H] tensor; 2-D and 3-D, recorded and not, and
    2-D views of wider buffers (a leading dimension above 2H, at an aligned
    and at an odd element offset); under both SwiGLU rules."""
    from polynomial_activation_gb300 import ops
    rng = np.random.default_rng(79)
    B.poly_set_swiglu_variant(variant)
    try:
        _packed_cases(ops, rng)
    finally:
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)


def _packed_cases(ops, rng):
    for dt in DTS:
        for shape, pad, off in (((64, 2 * 200), 0, 0), ((3, 7, 2 * 48), 0, 0),
                                ((40, 2 * 64), 24, 8), ((40, 2 * 64), 24, 3)):
            m = int(np.prod(shape))
            if pad:
                rows, w = shape
                big = to_dev(_rand_bits(rng, rows * (w + pad), FMT[dt]), dt).view(rows, w + pad)
                gu = big[:, off:off + w]
            else:
                gu = to_dev(_rand_bits(rng, m, FMT[dt]), dt).view(*shape)
            dy = to_dev(_rand_bits(rng, m // 2, FMT[dt]), dt).view(*shape[:-1], shape[-1] // 2)
            h = shape[-1] // 2
            g, u = gu[..., :h].contiguous(), gu[..., h:].contiguous()
            want = ops.swiglu_fwd(g.reshape(-1, h), u.reshape(-1, h)).view(*shape[:-1], h)
            got = ops.swiglu_packed(gu)
            assert got.shape == want.shape and got.grad_fn is None
            assert torch.equal(got.view(torch.int16), want.view(torch.int16))
            if pad:   # the recorded input is itself a view of the wider buffer
                bigr = big.clone().requires_grad_(True)
                gur = bigr[:, off:off + shape[1]]
            else:
                gur = gu.clone().requires_grad_(True)
            y = ops.swiglu_packed(gur)
            assert torch.equal(y.detach().view(torch.int16), want.view(torch.int16))
            y.backward(dy)
            grad = bigr.grad[:, off:off + shape[1]] if pad else gur.grad
            dg, du = ops.swiglu_bwd(g.reshape(-1, h), u.reshape(-1, h), dy.reshape(-1, h))
            assert grad.shape == gu.shape
            assert torch.equal(grad[..., :h].reshape(-1, h).view(torch.int16), dg.view(torch.int16))
            assert torch.equal(grad[..., h:].reshape(-1, h).view(torch.int16), du.view(torch.int16))
            if pad:
                assert not bool(bigr.grad[:, :off].any()) and not bool(bigr.grad[:, off + shape[1]:].any())


def test_swiglu_on_chunked_halves_takes_the_fused_path():
    """ops.swiglu(*gu.chunk(2, -1)) with a gate-up buffer in the graph runs on
    the buffer itself (one gradient buffer): the same bits as separate
    leaves, also through a reshape of the buffer and with the gate used
    elsewhere in the graph too."""
    from polynomial_activation_gb300 import ops
    rng = np.random.default_rng(81)
    for dt in DTS:
        rows, h = 48, 96
        gu0 = to_dev(_rand_bits(rng, rows * 2 * h, FMT[dt]), dt).view(rows, 2 * h)
        dy = to_dev(_rand_bits(rng, rows * h, FMT[dt]), dt).view(rows, h)
        g0, u0 = gu0[:, :h].contiguous(), gu0[:, h:].contiguous()
        want_y = ops.swiglu_fwd(g0, u0)
        want_dg, want_du = ops.swiglu_bwd(g0, u0, dy)
        # a leaf buffer, chunked
        gu = gu0.clone().requires_grad_(True)
        g, u = gu.chunk(2, dim=-1)
        assert ops._fused_base(g, u) is gu
        y = ops.swiglu(g, u)
        assert torch.equal(y.detach().view(torch.int16), want_y.view(torch.int16))
        y.backward(dy)
        assert torch.equal(gu.grad[:, :h].view(torch.int16), want_dg.view(torch.int16))
        assert torch.equal(gu.grad[:, h:].view(torch.int16), want_du.view(torch.int16))
        # a non-leaf buffer reshaped to [4, 12, 2H] before chunking; the gate
        # also feeds a second term of the loss (finite normal inputs: the
        # gradients from the two paths are summed by autograd)
        gu1 = to_dev(workloads.normal(rows * 2 * h, 82, 1.0, FMT[dt]), dt).view(rows, 2 * h)
        dy1 = to_dev(workloads.normal(rows * h, 83, 1.0, FMT[dt]), dt).view(rows, h)
        src = gu1.float().requires_grad_(True)
        x = src.to(TDT[dt]).view(4, rows // 4, 2 * h)
        g, u = x.chunk(2, dim=-1)
        assert ops._fused_base(g, u) is not None
        y = ops.swiglu(g, u)
        assert y.shape == (4, rows // 4, h)
        ((y * dy1.view(4, rows // 4, h)).float().sum() + g.float().sum()).backward()
        # reference with separate leaves
        gl = gu1[:, :h].contiguous().requires_grad_(True)
        ul = gu1[:, h:].contiguous().requires_grad_(True)
        yl = ops.swiglu(gl, ul)
        ((yl * dy1).float().sum() + gl.float().sum()).backward()
        got = src.grad.to(TDT[dt])
        assert torch.equal(got[:, :h].view(torch.int16), gl.grad.view(torch.int16))
        assert torch.equal(got[:, h:].view(torch.int16), ul.grad.view(torch.int16))


def test_swiglu_ragged_padding_free():
    """With padding_free (the offsets cover every row) the ragged wrapper
    skips the zero fill and gives the same bits, recorded and not."""
    from polynomial_activation_gb300 import ops
    rng = np.random.default_rng(80)
    for dt in DTS:
        rows, cols = 96, 136
        g = to_dev(_rand_bits(rng, rows * cols, FMT[dt]), dt).view(rows, cols)
        u = to_dev(_rand_bits(rng, rows * cols, FMT[dt]), dt).view(rows, cols)
        dy = to_dev(_rand_bits(rng, rows * cols, FMT[dt]), dt).view(rows, cols)
        seg = torch.tensor([0, 30, 30, 77, rows], dtype=torch.int32, device=DEV)
        want = ops.swiglu_ragged(g, u, seg)
        got = ops.swiglu_ragged(g, u, seg, padding_free=True)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))
        assert torch.equal(want.view(torch.int16), ops.swiglu_fwd(g, u).view(torch.int16))
        grads = []
        for pf in (False, True):
            gr, ur = g.clone().requires_grad_(True), u.clone().requires_grad_(True)
            y = ops.swiglu_ragged(gr, ur, seg, padding_free=pf)
            y.backward(dy)
            grads.append((y.detach(), gr.grad, ur.grad))
        for a, b in zip(*grads):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        dg, du = ops.swiglu_bwd(g, u, dy)
        assert torch.equal(grads[1][1].view(torch.int16), dg.view(torch.int16))
        assert torch.equal(grads[1][2].view(torch.int16), du.view(torch.int16))


def test_ragged_zero_outside():
    """poly_ragged_zero_outside zeroes exactly the rows outside the clamped
    range [max(seg[0], 0), min(seg[E], cap)) (empty when the offsets cross),
    leaves the range and the guard bands untouched, for row widths that are
    and are not multiples of 8 and for buffers on and off the 16-byte grid."""
    G = 64
    cases = [[0, 10, 30], [5, 10, 30], [0, 37], [10, 5], [-3, 50], [7], [0, 0, 36], [36, 37],
             [50], [40, 45], [-9, -2]]
    for cols in (8, 21, 2048, 3):
        cap = 37
        n = cap * cols
        for seg in cases:
            for off in (0, 1, 5):
                buf = torch.full((2 * G + off + n,), 0x5A5A, dtype=torch.int16, device=DEV)
                out = buf[G + off:G + off + n].view(cap, cols)
                segd = torch.tensor(seg, dtype=torch.int32, device=DEV)
                B.poly_ragged_zero_outside(out, segd)
                lo = min(max(seg[0], 0), cap)
                hi = max(min(seg[-1], cap), lo)
                got = from_dev(out).reshape(cap, cols)
                assert not got[:lo].any() and not got[hi:].any(), (cols, seg, off)
                assert (got[lo:hi] == 0x5A5A).all(), (cols, seg, off)
                b = from_dev(buf)
                assert (b[:G + off] == 0x5A5A).all() and (b[G + off + n:] == 0x5A5A).all()
    # full size: the ragged workload inside a capacity of 3,000 more rows
    g, u, dy, seg = workloads.ragged_swiglu("bf16")
    rows, cols = g.shape
    cap = rows + 3000
    y = torch.full((cap, cols), 0x5A5A, dtype=torch.int16, device=DEV)
    B.poly_ragged_zero_outside(y, torch.from_numpy(seg).to(DEV))
    assert bool((y[:rows] == 0x5A5A).all()) and not bool(y[rows:].any())
    del y


def test_calls_use_the_current_stream():
    """With no stream argument the binding launches on the current stream of
    the current device, inside and outside a torch.cuda.stream context."""
    side = torch.cuda.Stream()
    assert B._stream(None) == torch.cuda.current_stream().cuda_stream
    with torch.cuda.stream(side):
        assert B._stream(None) == side.cuda_stream
        assert B._stream(None) == torch.cuda.current_stream().cuda_stream
    assert B._stream(None) == torch.cuda.current_stream().cuda_stream


def test_every_degree_every_program_exhaustive():
    """Programs of every degree D3-D6 (fitted by the library, installed with
    poly_set_program) for every function, direction and format, over all
    65,536 inputs against the oracle replay of the same descriptor; then
    SwiGLU with non-default SiLU / SiLU' degree pairs."""
    from oracle import fit
    rng = np.random.default_rng(95)
    try:
        for dt in DTS:
            fmt = FMT[dt]
            xd = to_dev(X_ALL, dt)
            dy = _rand_bits(rng, X_ALL.size, fmt)
            dyd = to_dev(dy, dt)
            out = torch.empty_like(xd)
            for fn, d in PROGRAMS:
                for D in (3, 4, 5, 6):
                    p = B.poly_fit(fn, d, dt, D)
                    B.poly_set_program(p)
                    op = fit.make_program(fn, d, fmt, p.degree, p.li, p.lc, p.coefficients())
                    if d == B.POLY_FWD:
                        B.poly_act_fwd(fn, dt, xd, out)
                        want = forward(op, X_ALL)
                    else:
                        B.poly_act_bwd(fn, dt, xd, dyd, out)
                        want = backward(op, X_ALL, dy)
                    assert np.array_equal(from_dev(out), want), (fn, d, fmt, D)
                    # one element off the 16-byte grid: the general kernel's head / body / tail
                    if d == B.POLY_FWD:
                        B.poly_act_fwd(fn, dt, xd[1:], out[1:])
                    else:
                        B.poly_act_bwd(fn, dt, xd[1:], dyd[1:], out[1:])
                    assert np.array_equal(from_dev(out[1:]), want[1:]), (fn, d, fmt, D, "offset")
            g = _rand_bits(rng, 48 * 80, fmt).reshape(48, 80)
            u = _rand_bits(rng, 48 * 80, fmt).reshape(48, 80)
            gd, ud = to_dev(g, dt).view(48, 80), to_dev(u, dt).view(48, 80)
            for DS, DD in ((6, 3), (4, 6), (5, 5)):
                ps, pd = B.poly_fit(B.POLY_SILU, 0, dt, DS), B.poly_fit(B.POLY_SILU, 1, dt, DD)
                B.poly_set_program(ps)
                B.poly_set_program(pd)
                s_op = fit.make_program(B.POLY_SILU, 0, fmt, DS, ps.li, ps.lc, ps.coefficients())
                d_op = fit.make_program(B.POLY_SILU, 1, fmt, DD, pd.li, pd.lc, pd.coefficients())
                y, dg, du = (torch.empty_like(gd) for _ in range(3))
                B.poly_swiglu_fwd(dt, gd, ud, y)
                B.poly_swiglu_bwd(dt, gd, ud, ud, dg, du)
                wdg, wdu = swiglu_backward(s_op, d_op, g, u, u)
                assert np.array_equal(from_dev(y).reshape(48, 80), swiglu_forward(s_op, g, u))
                assert np.array_equal(from_dev(dg).reshape(48, 80), wdg), (DS, DD)
                assert np.array_equal(from_dev(du).reshape(48, 80), wdu), (DS, DD)
            # the sigmoid rule with sigmoid programs of degree 4-6
            from oracle.replay import swiglu_sigmoid_backward, swiglu_sigmoid_forward
            B.poly_set_swiglu_variant(B.POLY_SWIGLU_SIGMOID)
            for D in (4, 5, 6):
                p = B.poly_fit(B.POLY_SIGMOID, 0, dt, D)
                B.poly_set_program(p)
                sig = fit.make_program(B.POLY_SIGMOID, 0, fmt, D, p.li, p.lc, p.coefficients())
                y, dg, du = (torch.empty_like(gd) for _ in range(3))
                B.poly_swiglu_fwd(dt, gd, ud, y)
                B.poly_swiglu_bwd(dt, gd, ud, ud, dg, du)
                wdg, wdu = swiglu_sigmoid_backward(sig, g, u, u)
                assert np.array_equal(from_dev(y).reshape(48, 80), swiglu_sigmoid_forward(sig, g, u))
                assert np.array_equal(from_dev(dg).reshape(48, 80), wdg), D
                assert np.array_equal(from_dev(du).reshape(48, 80), wdu), D
            B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)
            # the softcap with tanh and tanh' programs of degree 3, 5 and 6
            from oracle.replay import softcap_backward, softcap_forward
            for D in (3, 5, 6):
                pf, pb = B.poly_fit(B.POLY_TANH, 0, dt, D), B.poly_fit(B.POLY_TANH, 1, dt, D)
                B.poly_set_program(pf)
                B.poly_set_program(pb)
                tf_op = fit.make_program(B.POLY_TANH, 0, fmt, D, pf.li, pf.lc, pf.coefficients())
                tb_op = fit.make_program(B.POLY_TANH, 1, fmt, D, pb.li, pb.lc, pb.coefficients())
                B.poly_softcap_fwd(dt, 30.0, xd, out)
                assert np.array_equal(from_dev(out), softcap_forward(tf_op, 30.0, X_ALL)), D
                B.poly_softcap_bwd(dt, 30.0, xd, dyd, out)
                assert np.array_equal(from_dev(out), softcap_backward(tb_op, 30.0, X_ALL, dy)), D
    finally:
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)
        B.poly_reset_programs()


def _random_program(rng, fn, d, dt, D):
    """A descriptor the library accepts with arbitrary coefficient bits:
    ordinary, subnormal, huge, infinite and NaN patterns mixed in."""
    fmt = FMT[dt]
    p = B.PolyProgram()
    p.fn, p.dir, p.dtype, p.degree = fn, d, dt, D
    p.form = B.lib().poly_form_of(fn, d)
    coef = _rand_bits(rng, D + 1, fmt)
    sp = np.array([0x0001, 0x8003, 0x7BFF, 0xFC00, 0x7E01] if fmt == "f16" else
                  [0x0001, 0x8003, 0x7F7F, 0xFF80, 0x7FC1], dtype=np.uint16)
    pick = rng.random(D + 1) < 0.25
    coef[pick] = sp[rng.integers(0, sp.size, int(pick.sum()))]
    if p.form != B.POLY_FORM_E:
        coef[0] = 0                                  # c0 = f(0) = 0 for these forms
    for j in range(D + 1):
        p.coef[j] = int(coef[j])
    lc = float(rng.uniform(0.25, 20.0))
    p.lc_bits = int(tf.from_f64(lc, fmt))
    p.lc = float(tf.decode(np.uint16(p.lc_bits), fmt))
    p.li = p.lc
    p.version = 1
    return p


def test_random_descriptors_exhaustive():
    """Any descriptor the library accepts -- here random coefficient bits,
    specials included, with a random clamp -- is evaluated bit-exactly: every
    form and degree D3-D6, both formats, all 65,536 inputs, three descriptors
    each."""
    from oracle import fit
    rng = np.random.default_rng(99)
    try:
        for dt in DTS:
            fmt = FMT[dt]
            xd = to_dev(X_ALL, dt)
            dy = _rand_bits(rng, X_ALL.size, fmt)
            dyd = to_dev(dy, dt)
            out = torch.empty_like(xd)
            for fn, d in PROGRAMS:
                for D in (3, 4, 5, 6):
                    for _ in range(3):
                        p = _random_program(rng, fn, d, dt, D)
                        B.poly_set_program(p)
                        op = fit.make_program(fn, d, fmt, D, p.li, p.lc, p.coefficients())
                        assert op.lc_bits == p.lc_bits
                        if d == B.POLY_FWD:
                            B.poly_act_fwd(fn, dt, xd, out)
                            want = forward(op, X_ALL)
                        else:
                            B.poly_act_bwd(fn, dt, xd, dyd, out)
                            want = backward(op, X_ALL, dy)
                        assert np.array_equal(from_dev(out), want), (fn, d, fmt, D, p.coefficients())
            # the fused kernels with random descriptors: SwiGLU (both rules), softcap
            from oracle.replay import (softcap_backward, softcap_forward,
                                       swiglu_sigmoid_backward, swiglu_sigmoid_forward)
            g = _rand_bits(rng, 32 * 64, fmt).reshape(32, 64)
            u = _rand_bits(rng, 32 * 64, fmt).reshape(32, 64)
            gd, ud = to_dev(g, dt).view(32, 64), to_dev(u, dt).view(32, 64)
            mk = lambda q: fit.make_program(q.fn, q.dir, fmt, q.degree, q.li, q.lc, q.coefficients())
            for D in (3, 5, 6):
                ps = _random_program(rng, B.POLY_SILU, 0, dt, D)
                pd = _random_program(rng, B.POLY_SILU, 1, dt, 9 - D)
                psig = _random_program(rng, B.POLY_SIGMOID, 0, dt, D)
                for q in (ps, pd, psig):
                    B.poly_set_program(q)
                y, dg, du = (torch.empty_like(gd) for _ in range(3))
                B.poly_swiglu_fwd(dt, gd, ud, y)
                B.poly_swiglu_bwd(dt, gd, ud, ud, dg, du)
                wdg, wdu = swiglu_backward(mk(ps), mk(pd), g, u, u)
                assert np.array_equal(from_dev(y).reshape(32, 64), swiglu_forward(mk(ps), g, u))
                assert np.array_equal(from_dev(dg).reshape(32, 64), wdg)
                assert np.array_equal(from_dev(du).reshape(32, 64), wdu)
                B.poly_set_swiglu_variant(B.POLY_SWIGLU_SIGMOID)
                try:
                    B.poly_swiglu_fwd(dt, gd, ud, y)
                    B.poly_swiglu_bwd(dt, gd, ud, ud, dg, du)
                finally:
                    B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)
                wdg, wdu = swiglu_sigmoid_backward(mk(psig), g, u, u)
                assert np.array_equal(from_dev(y).reshape(32, 64),
                                      swiglu_sigmoid_forward(mk(psig), g, u))
                assert np.array_equal(from_dev(dg).reshape(32, 64), wdg)
                assert np.array_equal(from_dev(du).reshape(32, 64), wdu)
                pt, ptd = (_random_program(rng, B.POLY_TANH, dd, dt, D) for dd in (0, 1))
                B.poly_set_program(pt)
                B.poly_set_program(ptd)
                B.poly_softcap_fwd(dt, 30.0, xd, out)
                assert np.array_equal(from_dev(out), softcap_forward(mk(pt), 30.0, X_ALL))
                B.poly_softcap_bwd(dt, 30.0, xd, dyd, out)
                assert np.array_equal(from_dev(out), softcap_backward(mk(ptd), 30.0, X_ALL, dy))
    finally:
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)
        B.poly_reset_programs()


def test_must_fail_perturbed_program_on_gpu():
    """The parity check can fail: install a program whose c_2 is one ulp off
    and the GPU output no longer equals the oracle's replay of the fitted
    program (while it equals the replay of the perturbed one)."""
    from oracle import fit
    dt = B.POLY_BF16
    p = B.poly_get_program(B.POLY_SIGMOID, B.POLY_FWD, dt)
    bad = B.PolyProgram.from_buffer_copy(bytes(p))
    bad.coef[2] += 1
    B.poly_set_program(bad)
    try:
        xd = to_dev(X_ALL, dt)
        out = torch.empty_like(xd)
        B.poly_act_fwd(B.POLY_SIGMOID, dt, xd, out)
        got = from_dev(out)
        good = fit.make_program(0, 0, "bf16", p.degree, p.li, p.lc, p.coefficients())
        perturbed = fit.make_program(0, 0, "bf16", bad.degree, bad.li, bad.lc, bad.coefficients())
        assert not np.array_equal(got, forward(good, X_ALL))
        assert np.array_equal(got, forward(perturbed, X_ALL))
    finally:
        B.poly_reset_programs()


def test_bench_line_keeps_its_contract():
    """bench.py on a small case prints one JSON line with every key its
    readers rely on, with consistent values."""
    import json as _json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--elements", str(1 << 22),
                        "--steps", "5", "--warmup", "3", "--no-extras", "--cpu-sample", "65536"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = _json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches", "env"):
        assert k in d, k
    assert d["steps"] == 5 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["value"] > 0
    assert d["gpu_launches"] == 6 * 5 and d["higher_is_better"] is True
    assert abs(d["value"] - 6 * (1 << 22) / (d["ms_per_step"] * 1e-3) / 1e9) < 1e-6 * d["value"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is None                      # recorded only for the full-size step
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["unit"] == d["unit"]
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 2 * 2 * (1 << 22) and e["d2h_bytes_per_step"] == 6 * 2 * (1 << 22)
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert "workload" in d["config"]

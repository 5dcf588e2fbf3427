"""GPU tests of the per-call variants: the packed-target-format MUFU control
(one tanh.approx per pair) against the FP64 functions, the SwiGLU rule passed
per call (bit-exact against the oracle whatever the process default, also
from concurrent host threads with different rules), and the streaming-
bandwidth probe's output.

Tolerance of the packed control.  Every packed operation rounds once (half an
ulp of its result) and tanh.approx carries its own error dt, a few ulps of 1
at most in the target format (u1 = the spacing just below 1: 2^-11 FP16,
2^-8 BF16).  A control y built from t = tanh.approx(.) then errs by at most
  tanh, sigmoid, sigma', tanh'  a few u1 plus 2 ulps of the value;
  SiLU = h + h t, h = x/2       |h| dt: the error grows with |x| (the exact
                                product h t cancels against h for x < 0);
  SiLU' = p + x p (1 - p)       |x| dp with dp = dt / 2;
  GELU (tanh form)              the same as SiLU plus the form's own
                                distance from exact GELU (4.8e-4; 8.7e-4 for
                                its derivative) and, in the derivative,
                                (1 - t^2) h z' where z' grows like x^2.
The tests assert |y - f| <= 2 ulp(f) + K u1 (1 + |x| / 2) (+ the tanh form's
distance for GELU) with K = 4 (forward) and 8 (backward) over every finite
input with |x| < 60 -- bounds that hold for a tanh.approx within 2 u1 -- and
report the measured maxima.  GELU' is tested on |x| <= 6 (where 1 - t^2 is not
yet rounded away) with K = 32: its error is |h z'| dt there.
"""
import threading

import numpy as np
import pytest
import torch

from gpu_util import DEV, FMT, TDT, from_dev, guards_intact, oracle_program, sentinel_buffer, to_dev
from oracle import reference as ref
from oracle import tformat as tf
from oracle.replay import swiglu_backward, swiglu_forward
from oracle.replay import swiglu_sigmoid_backward, swiglu_sigmoid_forward
from polynomial_activation_gb300 import binding as B

pytestmark = pytest.mark.gpu

DTS = [B.POLY_BF16, B.POLY_F16]
FNS = [B.POLY_SIGMOID, B.POLY_TANH, B.POLY_SILU, B.POLY_GELU]
X_ALL = tf.all_patterns()
U1 = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}
GELU_TANH_FORM = {B.POLY_FWD: 4.8e-4, B.POLY_BWD: 8.7e-4}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available()
    torch.cuda.set_device(DEV)
    B.poly_reset_programs()
    yield
    torch.cuda.synchronize()


def _ulp(f, fmt):
    a = np.abs(f)
    if fmt == "f16":
        return np.spacing(a.astype(np.float16)).astype(np.float64)
    return np.spacing(a.astype(np.float32)).astype(np.float64) * 2.0 ** 16


def _rand_bits(rng, n, fmt):
    b = rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    k = n // 2
    b[:k] = tf.from_f64(rng.normal(0, 4, k), fmt)
    return b


@pytest.mark.parametrize("dt", DTS)
@pytest.mark.parametrize("d", [B.POLY_FWD, B.POLY_BWD])
@pytest.mark.parametrize("fn", FNS)
def test_packed_control_accuracy(fn, d, dt):
    """The packed control approximates the true function within the bound
    derived in the module docstring, on every finite input with |x| < 60."""
    fmt = FMT[dt]
    x = X_ALL[tf.finite_mask(X_ALL, fmt)]
    xv = tf.decode(x, fmt)
    lim = 6.0 if (fn == B.POLY_GELU and d == B.POLY_BWD) else 60.0
    keep = np.abs(xv) <= lim
    x, xv = x[keep], xv[keep]
    xd = to_dev(x, dt)
    out = torch.empty_like(xd)
    if d == B.POLY_FWD:
        B.poly_ctrl_act_fwd_v(B.POLY_CTRL_PACKED, fn, dt, xd, out)
    else:
        ones = to_dev(tf.from_f64(np.ones(x.size), fmt), dt)
        B.poly_ctrl_act_bwd_v(B.POLY_CTRL_PACKED, fn, dt, xd, ones, out)
    y = tf.decode(from_dev(out), fmt)
    f = ref.function(fn, d)(xv)
    k = 4.0 if d == B.POLY_FWD else 8.0
    model = 0.0
    if fn == B.POLY_GELU:
        model = GELU_TANH_FORM[d]
        if d == B.POLY_BWD:
            k = 32.0
    tol = 2 * _ulp(f, fmt) + k * U1[fmt] * (1 + np.abs(xv) / 2) + model
    err = np.abs(y - f)
    worst = int(np.argmax(err / tol))
    assert np.all(np.isfinite(y)), (fn, d, fmt)
    assert np.all(err <= tol), (fn, d, fmt, float(xv[worst]), float(y[worst]), float(f[worst]),
                                float(np.max(err)))


@pytest.mark.parametrize("dt", DTS)
def test_packed_control_specials(dt):
    """NaN in, NaN out; signed zeros give the function's value at 0."""
    fmt = FMT[dt]
    nan, pz, nz = (int(v) for v in tf.from_f64(np.array([np.nan, 0.0, -0.0]), fmt))
    x = np.array([nan, pz, nz], dtype=np.uint16)
    xd = to_dev(x, dt)
    ones = to_dev(tf.from_f64(np.ones(3), fmt), dt)
    out = torch.empty_like(xd)
    for fn in FNS:
        B.poly_ctrl_act_fwd_v(B.POLY_CTRL_PACKED, fn, dt, xd, out)
        y = tf.decode(from_dev(out), fmt)
        assert np.isnan(y[0]) and y[1] == ref.function(fn, 0)(np.array([0.0]))[0], fn
        B.poly_ctrl_act_bwd_v(B.POLY_CTRL_PACKED, fn, dt, xd, ones, out)
        y = tf.decode(from_dev(out), fmt)
        assert np.isnan(y[0]) and y[1] == y[2] == ref.function(fn, 1)(np.array([0.0]))[0], fn


@pytest.mark.parametrize("dt", DTS)
def test_packed_control_is_position_independent(dt):
    """The packed control runs through the same streaming kernels as the
    programs: at every size 1..67 and misalignment 0..7 (scalar head and
    tail, one-lane evaluation) each element equals the aligned full-tensor
    result bit for bit, and nothing outside the output is written."""
    fmt = FMT[dt]
    rng = np.random.default_rng(21)
    x = _rand_bits(rng, 4096, fmt)
    dy = _rand_bits(rng, 4096, fmt)
    xd, dyd = to_dev(x, dt), to_dev(dy, dt)
    ref_f = {fn: torch.empty_like(xd) for fn in FNS}
    ref_b = {fn: torch.empty_like(xd) for fn in FNS}
    for fn in FNS:
        B.poly_ctrl_act_fwd_v(B.POLY_CTRL_PACKED, fn, dt, xd, ref_f[fn])
        B.poly_ctrl_act_bwd_v(B.POLY_CTRL_PACKED, fn, dt, xd, dyd, ref_b[fn])
    G = 16
    for n in (1, 2, 7, 8, 9, 15, 16, 17, 31, 33, 64, 67):
        for off in range(8):
            for fn in FNS:
                buf, o = sentinel_buffer(n, G, dt, off)
                B.poly_ctrl_act_fwd_v(B.POLY_CTRL_PACKED, fn, dt, xd[off:off + n], o, n)
                assert guards_intact(buf, n, G, off) and torch.equal(
                    o.view(torch.int16), ref_f[fn][off:off + n].view(torch.int16)), (fn, n, off)
                buf, o = sentinel_buffer(n, G, dt, off)
                B.poly_ctrl_act_bwd_v(B.POLY_CTRL_PACKED, fn, dt, xd[off:off + n],
                                      dyd[off:off + n], o, n)
                assert guards_intact(buf, n, G, off) and torch.equal(
                    o.view(torch.int16), ref_b[fn][off:off + n].view(torch.int16)), (fn, n, off)


@pytest.mark.parametrize("dt", DTS)
def test_packed_swiglu_control(dt):
    """y = SiLU(g) u, dg = (dy u) SiLU'(g), du = dy SiLU(g) with the packed
    control: within the SiLU bounds above (scaled by |u|, |dy u|) plus the
    products' roundings, on dense and fused-half layouts."""
    fmt = FMT[dt]
    rng = np.random.default_rng(8)
    rows, cols = 64, 256
    g = tf.from_f64(rng.normal(0, 3, rows * cols), fmt).reshape(rows, cols)
    u = tf.from_f64(rng.normal(0, 1, rows * cols), fmt).reshape(rows, cols)
    dy = tf.from_f64(rng.normal(0, 1, rows * cols), fmt).reshape(rows, cols)
    gd, ud, dyd = (to_dev(a, dt).view(rows, cols) for a in (g, u, dy))
    gv, uv, dv = (tf.decode(a, fmt) for a in (g, u, dy))
    u1 = U1[fmt]
    y = torch.empty_like(gd)
    B.poly_ctrl_swiglu_fwd_v(B.POLY_CTRL_PACKED, dt, gd, ud, y)
    want = ref.silu(gv) * uv
    tol = 3 * _ulp(want, fmt) + 4 * u1 * (1 + np.abs(gv) / 2) * np.abs(uv)
    got = tf.decode(from_dev(y).reshape(rows, cols), fmt)
    assert np.all(np.abs(got - want) <= tol)
    dg, du = torch.empty_like(gd), torch.empty_like(gd)
    B.poly_ctrl_swiglu_bwd_v(B.POLY_CTRL_PACKED, dt, gd, ud, dyd, dg, du)
    wdg = dv * uv * ref.dsilu(gv)
    wdu = dv * ref.silu(gv)
    tdg = 4 * _ulp(wdg, fmt) + 8 * u1 * (1 + np.abs(gv)) * np.abs(dv * uv)
    tdu = 3 * _ulp(wdu, fmt) + 4 * u1 * (1 + np.abs(gv) / 2) * np.abs(dv)
    assert np.all(np.abs(tf.decode(from_dev(dg).reshape(rows, cols), fmt) - wdg) <= tdg)
    assert np.all(np.abs(tf.decode(from_dev(du).reshape(rows, cols), fmt) - wdu) <= tdu)
    # gate and up as the halves of one fused buffer: the same values
    gu = torch.cat([gd, ud], dim=1)
    y2 = torch.empty_like(gd)
    B.poly_ctrl_swiglu_fwd_v(B.POLY_CTRL_PACKED, dt, gu[:, :cols], gu[:, cols:], y2)
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    # the FP32 control through the _v entry point equals the plain call
    y3 = torch.empty_like(gd)
    B.poly_ctrl_swiglu_fwd_v(B.POLY_CTRL_FP32, dt, gd, ud, y3)
    B.poly_ctrl_swiglu_fwd(dt, gd, ud, y)
    assert torch.equal(y3.view(torch.int16), y.view(torch.int16))


def _other(variant):
    return B.POLY_SWIGLU_SIGMOID if variant == B.POLY_SWIGLU_DIRECT else B.POLY_SWIGLU_DIRECT


def _want(variant, dt, g, u, dy):
    if variant == B.POLY_SWIGLU_DIRECT:
        ps = oracle_program(B.POLY_SILU, B.POLY_FWD, dt)
        pd = oracle_program(B.POLY_SILU, B.POLY_BWD, dt)
        return (swiglu_forward(ps, g, u),) + tuple(swiglu_backward(ps, pd, g, u, dy))
    sig = oracle_program(B.POLY_SIGMOID, B.POLY_FWD, dt)
    return (swiglu_sigmoid_forward(sig, g, u),) + tuple(swiglu_sigmoid_backward(sig, g, u, dy))


@pytest.mark.parametrize("variant", [B.POLY_SWIGLU_DIRECT, B.POLY_SWIGLU_SIGMOID])
@pytest.mark.parametrize("dt", DTS)
def test_swiglu_rule_per_call(dt, variant):
    """poly_swiglu_*_v compute the rule they are given, bit for bit, with the
    process-wide default set to the other rule: dense, strided (fused
    halves) and ragged layouts."""
    fmt = FMT[dt]
    rng = np.random.default_rng(40 + variant)
    rows, cols = 37, 1032
    g = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
    u = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
    dy = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
    wy, wdg, wdu = _want(variant, dt, g, u, dy)
    B.poly_set_swiglu_variant(_other(variant))
    try:
        gd, ud, dyd = (to_dev(a, dt).view(rows, cols) for a in (g, u, dy))
        y, dg, du = (torch.empty_like(gd) for _ in range(3))
        B.poly_swiglu_fwd_v(variant, dt, gd, ud, y)
        B.poly_swiglu_bwd_v(variant, dt, gd, ud, dyd, dg, du)
        assert np.array_equal(from_dev(y).reshape(rows, cols), wy)
        assert np.array_equal(from_dev(dg).reshape(rows, cols), wdg)
        assert np.array_equal(from_dev(du).reshape(rows, cols), wdu)
        gu = torch.cat([gd, ud], dim=1)
        dgu = torch.empty_like(gu)
        B.poly_swiglu_fwd_v(variant, dt, gu[:, :cols], gu[:, cols:], y)
        B.poly_swiglu_bwd_v(variant, dt, gu[:, :cols], gu[:, cols:], dyd, dgu[:, :cols],
                            dgu[:, cols:])
        assert np.array_equal(from_dev(y).reshape(rows, cols), wy)
        assert np.array_equal(from_dev(dgu[:, :cols]).reshape(rows, cols), wdg)
        assert np.array_equal(from_dev(dgu[:, cols:]).reshape(rows, cols), wdu)
        seg = torch.tensor([0, 5, 5, 30], dtype=torch.int32, device=DEV)
        status = torch.full((1,), 7, dtype=torch.int32, device=DEV)
        yr = torch.full((rows, cols), 0x5A5A, dtype=torch.int16, device=DEV).view(TDT[dt])
        dgr, dur = yr.clone(), yr.clone()
        B.poly_swiglu_fwd_ragged_v(variant, dt, gd, ud, yr, seg, status=status)
        B.poly_swiglu_bwd_ragged_v(variant, dt, gd, ud, dyd, dgr, dur, seg)
        assert int(status.item()) == 0
        assert np.array_equal(from_dev(yr).reshape(rows, cols)[:30], wy[:30])
        assert np.array_equal(from_dev(dgr).reshape(rows, cols)[:30], wdg[:30])
        assert np.array_equal(from_dev(dur).reshape(rows, cols)[:30], wdu[:30])
        for t in (yr, dgr, dur):
            assert np.all(from_dev(t).reshape(rows, cols)[30:] == 0x5A5A)
        assert B.poly_get_swiglu_variant() == _other(variant)
    finally:
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)


def test_swiglu_rules_from_concurrent_threads():
    """Four host threads on their own streams launch SwiGLU forward and
    backward at the same time, two with each rule (while a fifth thread keeps
    flipping the process-wide default); every output is its rule's oracle
    result."""
    dt, fmt = B.POLY_BF16, "bf16"
    rows, cols = 256, 2048
    rng = np.random.default_rng(77)
    jobs = []
    for i in range(4):
        variant = (B.POLY_SWIGLU_DIRECT, B.POLY_SWIGLU_SIGMOID)[i % 2]
        g = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
        u = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
        dy = _rand_bits(rng, rows * cols, fmt).reshape(rows, cols)
        dev = tuple(to_dev(a, dt).view(rows, cols) for a in (g, u, dy))
        outs = tuple(torch.empty_like(dev[0]) for _ in range(3))
        jobs.append((variant, (g, u, dy), dev, outs))
    for variant in (B.POLY_SWIGLU_DIRECT, B.POLY_SWIGLU_SIGMOID):   # fit outside the race
        _want(variant, dt, *jobs[0][1])
    torch.cuda.synchronize()
    errors, stop = [], threading.Event()

    def work(i):
        try:
            variant, _, (gd, ud, dyd), (y, dg, du) = jobs[i]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                for _ in range(40):
                    B.poly_swiglu_fwd_v(variant, dt, gd, ud, y)
                    B.poly_swiglu_bwd_v(variant, dt, gd, ud, dyd, dg, du)
            st.synchronize()
        except BaseException as e:
            errors.append(e)

    def flip():
        k = 0
        while not stop.is_set():
            B.poly_set_swiglu_variant(k % 2)
            k += 1

    flipper = threading.Thread(target=flip)
    flipper.start()
    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    try:
        for t in threads:
            t.start()
        for t in threads:
            t.join(timeout=120)
    finally:
        stop.set()
        flipper.join(timeout=30)
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)
    assert not errors, errors
    torch.cuda.synchronize()
    for variant, (g, u, dy), _, (y, dg, du) in jobs:
        wy, wdg, wdu = _want(variant, dt, g, u, dy)
        assert np.array_equal(from_dev(y).reshape(rows, cols), wy), variant
        assert np.array_equal(from_dev(dg).reshape(rows, cols), wdg), variant
        assert np.array_equal(from_dev(du).reshape(rows, cols), wdu), variant


@pytest.mark.parametrize("n", [8, 4096, 1 << 20, (1 << 22) + 8 * 37])
def test_stream_peak_probe_output(n):
    """The bandwidth probe writes out = a (one input) or a ^ b (two inputs)
    at every element after several rotated passes, and nothing else."""
    rng = np.random.default_rng(5)
    a = torch.from_numpy(rng.integers(-32768, 32767, n, dtype=np.int16)).to(DEV)
    b = torch.from_numpy(rng.integers(-32768, 32767, n, dtype=np.int16)).to(DEV)
    G = 64
    for nin in (1, 2):
        for inflight in (1, 2, 4, 8):
            for reps in (1, 3, 8):
                buf = torch.full((n + 2 * G,), 0x5A5A, dtype=torch.int16, device=DEV)
                out = buf[G:G + n]
                B.poly_diag_stream_peak(nin, a, b if nin == 2 else None, out, n, reps=reps,
                                        inflight=inflight)
                want = a if nin == 1 else a ^ b
                assert torch.equal(out, want), (nin, inflight, reps)
                assert bool((buf[:G] == 0x5A5A).all() and (buf[G + n:] == 0x5A5A).all())


@pytest.mark.parametrize("inflight", [2, 4])
def test_stream_peak_probe_l2_passes(inflight):
    """Two hundred rotated passes over L2-resident buffers (the launch the
    bench's L2 roof comes from) leave out = a ^ b everywhere."""
    n = 4_194_304
    rng = np.random.default_rng(9)
    a = torch.from_numpy(rng.integers(-32768, 32767, n, dtype=np.int16)).to(DEV)
    b = torch.from_numpy(rng.integers(-32768, 32767, n, dtype=np.int16)).to(DEV)
    out = torch.zeros_like(a)
    for _ in range(3):
        B.poly_diag_stream_peak(2, a, b, out, n, reps=200, inflight=inflight)
    assert torch.equal(out, a ^ b)


@pytest.mark.parametrize("rule", [B.POLY_SWIGLU_DIRECT, B.POLY_SWIGLU_SIGMOID])
def test_autograd_swiglu_keeps_its_rule(rule):
    """ops.swiglu / swiglu_packed / swiglu_ragged fix the SwiGLU rule when the
    forward runs: with the process default switched to the other rule before
    backward(), the gradients are still the chosen rule's, bit for bit."""
    from polynomial_activation_gb300 import ops
    dt, fmt = B.POLY_BF16, "bf16"
    rng = np.random.default_rng(90 + rule)
    rows, h = 64, 264
    g = _rand_bits(rng, rows * h, fmt).reshape(rows, h)
    u = _rand_bits(rng, rows * h, fmt).reshape(rows, h)
    dy = _rand_bits(rng, rows * h, fmt).reshape(rows, h)
    wy, wdg, wdu = _want(rule, dt, g, u, dy)
    dyd = to_dev(dy, dt).view(rows, h)
    try:
        for mode in ("pair", "packed", "chunked", "ragged"):
            B.poly_set_swiglu_variant(_other(rule))
            if mode == "pair":
                gd = to_dev(g, dt).view(rows, h).requires_grad_(True)
                ud = to_dev(u, dt).view(rows, h).requires_grad_(True)
                y = ops.swiglu(gd, ud, rule=rule)
            elif mode == "ragged":
                gd = to_dev(g, dt).view(rows, h).requires_grad_(True)
                ud = to_dev(u, dt).view(rows, h).requires_grad_(True)
                seg = torch.tensor([0, 20, rows], dtype=torch.int32, device=DEV)
                y = ops.swiglu_ragged(gd, ud, seg, rule=rule)
            else:
                gu = torch.cat([to_dev(g, dt).view(rows, h), to_dev(u, dt).view(rows, h)],
                               dim=1).requires_grad_(True)
                y = (ops.swiglu_packed(gu, rule=rule) if mode == "packed"
                     else ops.swiglu(*gu.chunk(2, dim=-1), rule=rule))
            B.poly_set_swiglu_variant(rule)       # flip the default between fwd and bwd
            B.poly_set_swiglu_variant(_other(rule))
            y.backward(dyd)
            assert np.array_equal(from_dev(y.detach()).reshape(rows, h), wy), mode
            if mode in ("pair", "ragged"):
                dg, du = gd.grad, ud.grad
            else:
                dg, du = gu.grad[:, :h], gu.grad[:, h:]
            assert np.array_equal(from_dev(dg).reshape(rows, h), wdg), mode
            assert np.array_equal(from_dev(du).reshape(rows, h), wdu), mode
    finally:
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)

"""Tensor-level conveniences over the C ABI: allocate the output with torch
(device memory only) and call the library's kernel on the current stream."""
from __future__ import annotations

import torch

from . import binding as B


_IDS = {torch.float16: B.POLY_F16, torch.bfloat16: B.POLY_BF16}


def _dt(t):
    dt = _IDS.get(t.dtype)
    if dt is None:
        raise TypeError("FP16 or BF16 tensors only")
    if not t.is_cuda:
        raise ValueError("CUDA tensors only: the library has no CPU path")
    return dt


def _dense(t):
    """t, or a contiguous copy of it (the check is cheaper than a no-op
    .contiguous() call, which goes through the dispatcher)."""
    return t if t.is_contiguous() else t.contiguous()


def act_fwd(fn: str, x: torch.Tensor, out=None, control: bool = False) -> torch.Tensor:
    x = _dense(x)
    y = torch.empty_like(x) if out is None else out
    (B.poly_ctrl_act_fwd if control else B.poly_act_fwd)(B.FN[fn], _dt(x), x, y)
    return y


def act_bwd(fn: str, x: torch.Tensor, dy: torch.Tensor, out=None,
            control: bool = False) -> torch.Tensor:
    x, dy = _dense(x), _dense(dy)
    dx = torch.empty_like(x) if out is None else out
    (B.poly_ctrl_act_bwd if control else B.poly_act_bwd)(B.FN[fn], _dt(x), x, dy, dx)
    return dx


def _rows(t):
    """t itself when it is a row-major 2-D view (any leading dimension, e.g.
    one half of a [T, 2H] gate-up buffer), else a contiguous copy."""
    return t if t.dim() == 2 and t.stride(1) == 1 else t.contiguous()


def _rule(rule):
    """The SwiGLU rule of a call: POLY_SWIGLU_DIRECT or POLY_SWIGLU_SIGMOID,
    or None for the library's process-wide default, read now."""
    if rule is None:
        return B.poly_get_swiglu_variant()
    if rule not in (B.POLY_SWIGLU_DIRECT, B.POLY_SWIGLU_SIGMOID):
        raise ValueError(f"unknown SwiGLU rule {rule!r}")
    return rule


def swiglu_fwd(g, u, out=None, control: bool = False, rule=None):
    """y = SiLU(g) * u under `rule` (None: the process default), or with the
    FP32 MUFU control."""
    y = torch.empty(g.shape, dtype=g.dtype, device=g.device) if out is None else out
    if control:
        B.poly_ctrl_swiglu_fwd(_dt(g), g, u, y)
    else:
        B.poly_swiglu_fwd_v(_rule(rule), _dt(g), g, u, y)
    return y


def swiglu_bwd(g, u, dy, control: bool = False, rule=None):
    dg = torch.empty(g.shape, dtype=g.dtype, device=g.device)
    du = torch.empty(g.shape, dtype=g.dtype, device=g.device)
    if control:
        B.poly_ctrl_swiglu_bwd(_dt(g), g, u, dy, dg, du)
    else:
        B.poly_swiglu_bwd_v(_rule(rule), _dt(g), g, u, dy, dg, du)
    return dg, du


def swiglu_fwd_ragged(g, u, seg_off, out=None, status=None, rule=None):
    y = torch.empty_like(g) if out is None else out
    B.poly_swiglu_fwd_ragged_v(_rule(rule), _dt(g), g, u, y, seg_off, status=status)
    return y


def swiglu_bwd_ragged(g, u, dy, seg_off, dg=None, du=None, status=None, rule=None):
    dg = torch.empty_like(g) if dg is None else dg
    du = torch.empty_like(g) if du is None else du
    B.poly_swiglu_bwd_ragged_v(_rule(rule), _dt(g), g, u, dy, dg, du, seg_off, status=status)
    return dg, du


# ---- autograd: drop-in modules for training code --------------------------
# Each forward saves its inputs and the backward recomputes the programs from
# them (the paper's backward constructions evaluate from x, §4.2, §5.2.4), so
# no activation tensor is kept.

class PolyActivation(torch.autograd.Function):
    """y = program_fwd(fn)(x); dx = dy * program_bwd(fn)(x)."""

    @staticmethod
    def forward(ctx, x, fn: str):
        x = _dense(x)
        ctx.save_for_backward(x)
        ctx.fn = fn
        return act_fwd(fn, x)

    @staticmethod
    def backward(ctx, dy):
        (x,) = ctx.saved_tensors
        return act_bwd(ctx.fn, x, _dense(dy)), None


def _grad(*ts):
    """True when autograd has to record the call; otherwise the wrappers below
    call the kernels directly (the autograd node costs ~10 us of host time)."""
    return torch.is_grad_enabled() and any(t.requires_grad for t in ts)


def _act(x, fn):
    return PolyActivation.apply(x, fn) if _grad(x) else act_fwd(fn, x)


def sigmoid(x):
    return _act(x, "sigmoid")


def tanh(x):
    return _act(x, "tanh")


def silu(x):
    return _act(x, "silu")


def gelu(x):
    return _act(x, "gelu")


class PolySwiGLU(torch.autograd.Function):
    """y = SiLU(g) * u under a SwiGLU rule fixed at forward time (the
    backward uses the same rule whatever the process default is by then)."""

    @staticmethod
    def forward(ctx, g, u, rule=None):
        g, u = _rows(g), _rows(u)
        ctx.save_for_backward(g, u)
        ctx.rule = _rule(rule)
        return swiglu_fwd(g, u, rule=ctx.rule)

    @staticmethod
    def backward(ctx, dy):
        g, u = ctx.saved_tensors
        return swiglu_bwd(g, u, _rows(dy), rule=ctx.rule) + (None,)


def _fused_base(g, u):
    """The contiguous [..., 2H] buffer whose two halves g and u are (as from
    gu.chunk(2, dim=-1), possibly through a reshape of gu), or None."""
    b = g._base
    if b is None or u._base is not b or not b.is_contiguous() or g.dim() == 0:
        return None
    # differentiable views of a buffer that is itself in the graph
    if not (b.requires_grad and g.grad_fn is not None and u.grad_fn is not None):
        return None
    h = g.shape[-1]
    if g.shape != u.shape or b.shape[-1] != 2 * h or b.numel() != 2 * g.numel():
        return None
    es = g.element_size()
    if g.data_ptr() != b.data_ptr() or u.data_ptr() != b.data_ptr() + h * es:
        return None
    # g and u must be rows of h elements, one every 2h, in row-major order
    want = 2 * h
    for d in range(g.dim() - 2, -1, -1):
        if g.stride(d) != want and g.shape[d] != 1:
            return None
        want *= g.shape[d]
    if g.stride(-1) != 1 or g.stride() != u.stride():
        return None
    return b


def swiglu(g, u, rule=None):
    """SiLU(g) * u under `rule` (POLY_SWIGLU_DIRECT, POLY_SWIGLU_SIGMOID, or
    None for the process default at the time of the call; the backward
    keeps that rule).  When g and u are the two halves of one fused gate-up
    buffer (gu.chunk(2, dim=-1)), the recorded path runs on that buffer so
    that the backward writes one [..., 2H] gradient (see swiglu_packed)."""
    rule = _rule(rule)
    if not _grad(g, u):
        return swiglu_fwd(_rows(g), _rows(u), rule=rule)
    b = _fused_base(g, u)
    if b is not None:
        y = PolySwiGLUPacked.apply(b, rule)
        return y if y.shape == g.shape else y.view(g.shape)
    return PolySwiGLU.apply(g, u, rule)


def _halves(gu):
    """[rows, 2H] row-major view of a fused gate-up buffer, H, the leading
    dimension, and the addresses of the two halves (raw addresses rather
    than slice tensors: two slices cost more host time than the call)."""
    two_h = gu.shape[-1]
    if two_h % 2:
        raise ValueError("the last dimension of a fused gate-up buffer must be even")
    gu2 = gu if gu.dim() == 2 and gu.stride(1) == 1 else _dense(gu).view(-1, two_h)
    h = two_h // 2
    p = gu2.data_ptr()
    return gu2, h, gu2.stride(0), p, p + h * gu2.element_size()


def _packed_fwd(gu, rule):
    gu2, h, ld, gp, up = _halves(gu)
    rows = gu2.shape[0]
    y = torch.empty((rows, h), dtype=gu.dtype, device=gu.device)
    # the halves lie inside gu2 by construction; y carries the device check
    B.poly_swiglu_fwd_v(rule, _dt(gu), gp, up, y, rows=rows, cols=h, ldg=ld, ldu=ld, ldy=h)
    return y.view(*gu.shape[:-1], h)


class PolySwiGLUPacked(torch.autograd.Function):
    """y = SiLU(gu[..., :H]) * gu[..., H:] for a fused gate-up buffer
    [..., 2H] (one projection producing both halves).  The backward writes
    dgate and dup straight into the two halves of one [..., 2H] gradient, so
    no slice gradients are assembled afterwards."""

    @staticmethod
    def forward(ctx, gu, rule=None):
        ctx.save_for_backward(gu)
        ctx.rule = _rule(rule)
        return _packed_fwd(gu, ctx.rule)

    @staticmethod
    def backward(ctx, dy):
        (gu,) = ctx.saved_tensors
        gu2, h, ld, gp, up = _halves(gu)
        rows = gu2.shape[0]
        dgu = torch.empty((rows, 2 * h), dtype=gu.dtype, device=gu.device)
        dyv = _dense(dy).view(-1, h)
        dp = dgu.data_ptr()
        B.poly_swiglu_bwd_v(ctx.rule, _dt(gu), gp, up, dyv, dp, dp + h * dgu.element_size(),
                            rows=rows, cols=h, ldg=ld, ldu=ld, lddy=h, lddg=2 * h, lddu=2 * h)
        return dgu.view(gu.shape), None


def swiglu_packed(gu, rule=None):
    """SwiGLU of a fused gate-up buffer [..., 2H] -> [..., H] under `rule`
    (None: the process default at the time of the call)."""
    rule = _rule(rule)
    return PolySwiGLUPacked.apply(gu, rule) if _grad(gu) else _packed_fwd(gu, rule)


class PolySwiGLURagged(torch.autograd.Function):
    """Routed-expert SwiGLU over rows [seg_off[0], seg_off[E]) of [cap_rows,
    cols] gate / up buffers (offsets stay on the device); rows outside the
    range are zero in the output and in both gradients (written once, by
    poly_ragged_zero_outside).  With padding_free the caller guarantees
    seg_off[0] = 0 and seg_off[E] = cap_rows, so the kernel writes every row
    and the zeroing launch is skipped."""

    @staticmethod
    def forward(ctx, g, u, seg_off, padding_free, rule=None):
        g, u = _dense(g), _dense(u)
        ctx.save_for_backward(g, u, seg_off)
        ctx.padding_free = padding_free
        ctx.rule = _rule(rule)
        return _ragged_fwd(g, u, seg_off, padding_free, ctx.rule)

    @staticmethod
    def backward(ctx, dy):
        g, u, seg_off = ctx.saved_tensors
        dg, du = swiglu_bwd_ragged(g, u, _dense(dy), seg_off, rule=ctx.rule)
        if not ctx.padding_free:
            B.poly_ragged_zero_outside(dg, seg_off)
            B.poly_ragged_zero_outside(du, seg_off)
        return dg, du, None, None, None


def _ragged_fwd(g, u, seg_off, padding_free=False, rule=None):
    y = swiglu_fwd_ragged(g, u, seg_off, rule=rule)
    if not padding_free:
        B.poly_ragged_zero_outside(y, seg_off)
    return y


def swiglu_ragged(g, u, seg_off, padding_free: bool = False, rule=None):
    """Rows outside [seg_off[0], seg_off[E]) of the output (and of the
    gradients) are zero: one extra launch zeroes them on the device, writing
    nothing when the segments cover every row.  padding_free=True (seg_off[0]
    = 0 and seg_off[E] = g.shape[0]) skips that launch; rows outside the range
    would then be left uninitialised, so pass it only when that holds.  (A
    padding-free call covers every row, so it computes exactly what swiglu
    does; for gate and up halves of one fused [rows, 2H] buffer, which the
    ragged calls do not take, use swiglu or swiglu_packed.)"""
    rule = _rule(rule)
    if _grad(g, u):
        return PolySwiGLURagged.apply(g, u, seg_off, padding_free, rule)
    return _ragged_fwd(_dense(g), _dense(u), seg_off, padding_free, rule)


class PolySoftcap(torch.autograd.Function):
    """alpha * tanh(x / alpha) (attention-logit softcap)."""

    @staticmethod
    def forward(ctx, x, alpha: float):
        x = _dense(x)
        ctx.save_for_backward(x)
        ctx.alpha = alpha
        return _softcap_fwd(x, alpha)

    @staticmethod
    def backward(ctx, dy):
        (x,) = ctx.saved_tensors
        dx = torch.empty_like(x)
        B.poly_softcap_bwd(_dt(x), ctx.alpha, x, _dense(dy), dx)
        return dx, None


def _softcap_fwd(x, alpha):
    y = torch.empty_like(x)
    B.poly_softcap_fwd(_dt(x), alpha, x, y)
    return y


def softcap(x, alpha: float):
    return PolySoftcap.apply(x, alpha) if _grad(x) else _softcap_fwd(_dense(x), alpha)


class PolyRoPE(torch.autograd.Function):
    """q [B, S, Hq, D], k [B, S, Hkv, D] (FP16) -> rotated q [B, Hq, S, D],
    k [B, Hkv, S, D] with polynomial sine / cosine."""

    @staticmethod
    def forward(ctx, q, k, delta, pos_offset: int):
        qo, ko = _rope_fwd(q, k, delta, pos_offset)
        ctx.save_for_backward(delta)
        ctx.meta = (q.shape[0], q.shape[1], q.shape[2], k.shape[2], q.shape[3], pos_offset)
        return qo, ko

    @staticmethod
    def backward(ctx, dqo, dko):
        (delta,) = ctx.saved_tensors
        b, s, hq, hkv, d, pos = ctx.meta
        dqo = torch.zeros((b, hq, s, d), dtype=torch.float16, device=delta.device) \
            if dqo is None else _dense(dqo)
        dko = torch.zeros((b, hkv, s, d), dtype=torch.float16, device=delta.device) \
            if dko is None else _dense(dko)
        dq = torch.empty((b, s, hq, d), dtype=dqo.dtype, device=dqo.device)
        dk = torch.empty((b, s, hkv, d), dtype=dko.dtype, device=dko.device)
        B.poly_rope_bwd(B.POLY_ROPE_POLY, dqo, dko, dq, dk, delta, pos_offset=pos)
        return dq, dk, None, None


def _rope_fwd(q, k, delta, pos_offset):
    q, k = _dense(q), _dense(k)
    b, s, hq, d = q.shape
    hkv = k.shape[2]
    qo = torch.empty((b, hq, s, d), dtype=q.dtype, device=q.device)
    ko = torch.empty((b, hkv, s, d), dtype=k.dtype, device=k.device)
    B.poly_rope_fwd(B.POLY_ROPE_POLY, q, k, qo, ko, delta, pos_offset=pos_offset)
    return qo, ko


def rope(q, k, delta, pos_offset: int = 0):
    """delta: device uint32/int32 tensor of D/2 turn increments
    (``binding.poly_rope_turn_increments``)."""
    if _grad(q, k):
        return PolyRoPE.apply(q, k, delta, pos_offset)
    return _rope_fwd(q, k, delta, pos_offset)

"""Tensor-level conveniences over the C ABI: allocate the output with torch
(device memory only) and call the library's kernel on the current stream."""
from __future__ import annotations

import torch

from . import binding as B


def _dt(t):
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("FP16 or BF16 tensors only")
    if not t.is_cuda:
        raise ValueError("CUDA tensors only: the library has no CPU path")
    return B.POLY_F16 if t.dtype == torch.float16 else B.POLY_BF16


def act_fwd(fn: str, x: torch.Tensor, out=None, control: bool = False) -> torch.Tensor:
    x = x.contiguous()
    y = torch.empty_like(x) if out is None else out
    (B.poly_ctrl_act_fwd if control else B.poly_act_fwd)(B.FN[fn], _dt(x), x, y)
    return y


def act_bwd(fn: str, x: torch.Tensor, dy: torch.Tensor, out=None,
            control: bool = False) -> torch.Tensor:
    x, dy = x.contiguous(), dy.contiguous()
    dx = torch.empty_like(x) if out is None else out
    (B.poly_ctrl_act_bwd if control else B.poly_act_bwd)(B.FN[fn], _dt(x), x, dy, dx)
    return dx


def swiglu_fwd(g, u, out=None, control: bool = False):
    y = torch.empty(g.shape, dtype=g.dtype, device=g.device) if out is None else out
    (B.poly_ctrl_swiglu_fwd if control else B.poly_swiglu_fwd)(_dt(g), g, u, y)
    return y


def swiglu_bwd(g, u, dy, control: bool = False):
    dg = torch.empty(g.shape, dtype=g.dtype, device=g.device)
    du = torch.empty(g.shape, dtype=g.dtype, device=g.device)
    (B.poly_ctrl_swiglu_bwd if control else B.poly_swiglu_bwd)(_dt(g), g, u, dy, dg, du)
    return dg, du


def swiglu_fwd_ragged(g, u, seg_off, out=None, status=None):
    y = torch.empty_like(g) if out is None else out
    B.poly_swiglu_fwd_ragged(_dt(g), g, u, y, seg_off, status=status)
    return y


def swiglu_bwd_ragged(g, u, dy, seg_off, dg=None, du=None, status=None):
    dg = torch.empty_like(g) if dg is None else dg
    du = torch.empty_like(g) if du is None else du
    B.poly_swiglu_bwd_ragged(_dt(g), g, u, dy, dg, du, seg_off, status=status)
    return dg, du

"""Helpers for the GPU tests: host <-> device transfer of 16-bit patterns and
the oracle program matching a library program (after checking that the
library's fitter produced exactly the oracle's program)."""
import numpy as np
import torch

import golden_programs as gp
from oracle import fit
from polynomial_activation_gb300 import binding as B

FMT = {B.POLY_F16: "f16", B.POLY_BF16: "bf16"}
TDT = {B.POLY_F16: torch.float16, B.POLY_BF16: torch.bfloat16}
DEV = torch.device("cuda:0")


def to_dev(bits: np.ndarray, dt: int) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV)
    return t.view(TDT[dt])


def from_dev(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_program(fn: int, d: int, dt: int):
    """The library's installed program, as an oracle Program, asserted equal to
    the oracle fitter's own program (tests/golden/programs.json)."""
    p = B.poly_get_program(fn, d, dt)
    g = gp.get(fn, d, FMT[dt], p.degree)
    assert p.coefficients() == list(g.coef) and p.lc_bits == g.lc_bits, (fn, d, dt)
    return fit.make_program(fn, d, FMT[dt], p.degree, p.li, p.lc, p.coefficients())


def sentinel_buffer(n: int, guard: int, dt: int, offset: int = 0):
    """A device buffer of guard + offset + n + guard elements filled with a
    sentinel; returns (buffer, view of the n output elements)."""
    buf = torch.full((2 * guard + offset + n,), 0x5A5A, dtype=torch.int16, device=DEV)
    buf = buf.view(TDT[dt])
    return buf, buf[guard + offset: guard + offset + n]


def guards_intact(buf: torch.Tensor, n: int, guard: int, offset: int = 0) -> bool:
    b = buf.view(torch.int16)
    return bool((b[:guard + offset] == 0x5A5A).all() and (b[guard + offset + n:] == 0x5A5A).all())

"""Thin ctypes binding of libpolyact (include/polyact.h).

Argument marshalling only: every function here has the name of the C entry
point it calls, turns tensors into device pointers and sizes, passes the
current torch CUDA stream unless one is given, and raises ``PolyError`` on a
non-zero status.  All computation happens in the library's CUDA kernels (and,
for ``poly_fit``, in its host fitter); there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpolyact.so")

POLY_F16, POLY_BF16 = 0, 1
POLY_SIGMOID, POLY_TANH, POLY_SILU, POLY_GELU = 0, 1, 2, 3
POLY_FWD, POLY_BWD = 0, 1
POLY_FORM_CO, POLY_FORM_O, POLY_FORM_E, POLY_FORM_HX = 0, 1, 2, 3
POLY_OK, POLY_EINVAL, POLY_ENOPROG, POLY_ECUDA, POLY_ENOFIT = 0, -1, -2, -3, -4
POLY_MAX_DEGREE = 6
POLY_PROGRAM_VERSION = 1
FN = {"sigmoid": POLY_SIGMOID, "tanh": POLY_TANH, "silu": POLY_SILU, "gelu": POLY_GELU}
FN_NAMES = {v: k for k, v in FN.items()}

# version of include/polyact.h this binding marshals for (poly_abi_version)
ABI_VERSION = 4

# every function declared in include/polyact.h
EXPORTS = [
    "poly_status_str", "poly_last_cuda_error", "poly_abi_version", "poly_form_of",
    "poly_default_degree", "poly_fit_defaults", "poly_fit", "poly_set_program",
    "poly_get_program", "poly_reset_programs", "poly_act_fwd", "poly_act_bwd",
    "poly_swiglu_fwd", "poly_swiglu_bwd", "poly_swiglu_fwd_ragged", "poly_swiglu_bwd_ragged",
    "poly_ragged_zero_outside",
    "poly_ctrl_act_fwd", "poly_ctrl_act_bwd", "poly_ctrl_swiglu_fwd", "poly_ctrl_swiglu_bwd",
    "poly_diag_packed", "poly_set_swiglu_variant", "poly_get_swiglu_variant",
    "poly_debug_fail_launches",
    "poly_derive_program", "poly_softcap_fwd", "poly_softcap_bwd", "poly_exp2",
    "poly_ctrl_exp2", "poly_rope_fwd", "poly_rope_bwd", "poly_rope_turn_increments",
    "poly_rope_programs",
    "poly_swiglu_fwd_v", "poly_swiglu_bwd_v", "poly_swiglu_fwd_ragged_v",
    "poly_swiglu_bwd_ragged_v", "poly_ctrl_act_fwd_v", "poly_ctrl_act_bwd_v",
    "poly_ctrl_swiglu_fwd_v", "poly_ctrl_swiglu_bwd_v", "poly_diag_stream_peak",
]
POLY_ROPE_POLY, POLY_ROPE_MUFU, POLY_ROPE_TABLE = 0, 1, 2
POLY_EXP2_D1, POLY_EXP2_PWL2, POLY_EXP2_D2, POLY_EXP2_D3 = 0, 1, 2, 3
POLY_SWIGLU_DIRECT, POLY_SWIGLU_SIGMOID = 0, 1
POLY_CTRL_FP32, POLY_CTRL_PACKED = 0, 1
POLY_DIAG_FMA, POLY_DIAG_MUL, POLY_DIAG_MIN_NAN, POLY_DIAG_MAX, POLY_DIAG_GT = 0, 1, 2, 3, 4


class PolyProgram(ctypes.Structure):
    _fields_ = [
        ("fn", ctypes.c_int32), ("dir", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("form", ctypes.c_int32), ("degree", ctypes.c_int32),
        ("coef", ctypes.c_uint16 * (POLY_MAX_DEGREE + 1)), ("lc_bits", ctypes.c_uint16),
        ("li", ctypes.c_double), ("lc", ctypes.c_double),
        ("search_score", ctypes.c_double), ("deployed_score", ctypes.c_double),
        ("stated_max_abs_err", ctypes.c_double), ("table2", ctypes.c_double),
        ("rank", ctypes.c_int32), ("version", ctypes.c_uint32),
    ]

    def coefficients(self):
        return [int(self.coef[j]) for j in range(self.degree + 1)]


class PolyFitOpts(ctypes.Structure):
    _fields_ = [
        ("li_min", ctypes.c_double), ("li_max", ctypes.c_double), ("li_step", ctypes.c_double),
        ("lc_min", ctypes.c_double), ("lc_step", ctypes.c_double),
        ("n_nodes", ctypes.c_int32), ("n_score", ctypes.c_int32),
        ("score_hi", ctypes.c_double), ("top_k", ctypes.c_int32),
        ("lc_refine_ulps", ctypes.c_int32),
    ]


class PolyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().poly_status_str(status).decode()
        if status == POLY_ECUDA:
            msg += f" (cudaError {lib().poly_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


_LIB = None

_i, _i64, _p = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p


def lib():
    """Load libpolyact.so (built by ``__graft_entry__.build()``); fails loudly
    if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    L.poly_status_str.restype = ctypes.c_char_p
    L.poly_status_str.argtypes = [_i]
    L.poly_set_swiglu_variant.argtypes = [_i]
    L.poly_derive_program.argtypes = [ctypes.POINTER(PolyProgram), ctypes.POINTER(PolyProgram)]
    L.poly_exp2.argtypes = [_i, _p, _p, _i64, _p]
    for name in ("poly_rope_fwd", "poly_rope_bwd"):
        getattr(L, name).argtypes = [_i, _p, _p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64,
                                     _i64, _i64, _p]
    L.poly_rope_turn_increments.argtypes = [_i, ctypes.c_double, _p]
    L.poly_rope_programs.argtypes = [_p, _p]
    L.poly_ctrl_exp2.argtypes = [_p, _p, _i64, _p]
    L.poly_softcap_fwd.argtypes = [_i, ctypes.c_double, _p, _p, _i64, _p]
    L.poly_softcap_bwd.argtypes = [_i, ctypes.c_double, _p, _p, _p, _i64, _p]
    for name in ("poly_last_cuda_error", "poly_abi_version", "poly_reset_programs",
                 "poly_get_swiglu_variant"):
        getattr(L, name).restype = _i
        getattr(L, name).argtypes = []
    L.poly_form_of.argtypes = [_i, _i]
    L.poly_default_degree.argtypes = [_i, _i]
    L.poly_fit_defaults.argtypes = [ctypes.POINTER(PolyFitOpts)]
    L.poly_fit.argtypes = [_i, _i, _i, _i, ctypes.POINTER(PolyFitOpts), ctypes.POINTER(PolyProgram)]
    L.poly_set_program.argtypes = [ctypes.POINTER(PolyProgram)]
    L.poly_get_program.argtypes = [_i, _i, _i, ctypes.POINTER(PolyProgram)]
    for name in ("poly_act_fwd", "poly_ctrl_act_fwd"):
        getattr(L, name).argtypes = [_i, _i, _p, _p, _i64, _p]
    for name in ("poly_act_bwd", "poly_ctrl_act_bwd"):
        getattr(L, name).argtypes = [_i, _i, _p, _p, _p, _i64, _p]
    for name in ("poly_swiglu_fwd", "poly_ctrl_swiglu_fwd"):
        getattr(L, name).argtypes = [_i, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _p]
    for name in ("poly_swiglu_bwd", "poly_ctrl_swiglu_bwd"):
        getattr(L, name).argtypes = [_i, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64,
                                     _i64, _i64, _p]
    L.poly_swiglu_fwd_ragged.argtypes = [_i, _p, _p, _p, _p, _i, _i64, _i64, _p, _p]
    L.poly_swiglu_bwd_ragged.argtypes = [_i, _p, _p, _p, _p, _p, _p, _i, _i64, _i64, _p, _p]
    L.poly_ragged_zero_outside.argtypes = [_p, _p, _i, _i64, _i64, _p]
    L.poly_diag_packed.argtypes = [_i, _i, _p, _p, _p, _p, _i64, _p]
    L.poly_diag_stream_peak.argtypes = [_i, _i, _p, _p, _p, _i64, _i, _p]
    L.poly_ctrl_act_fwd_v.argtypes = [_i, _i, _i, _p, _p, _i64, _p]
    L.poly_ctrl_act_bwd_v.argtypes = [_i, _i, _i, _p, _p, _p, _i64, _p]
    for name in ("poly_swiglu_fwd_v", "poly_ctrl_swiglu_fwd_v"):
        getattr(L, name).argtypes = [_i, _i, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _p]
    for name in ("poly_swiglu_bwd_v", "poly_ctrl_swiglu_bwd_v"):
        getattr(L, name).argtypes = [_i, _i, _p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64,
                                     _i64, _i64, _p]
    L.poly_swiglu_fwd_ragged_v.argtypes = [_i, _i, _p, _p, _p, _p, _i, _i64, _i64, _p, _p]
    L.poly_swiglu_bwd_ragged_v.argtypes = [_i, _i, _p, _p, _p, _p, _p, _p, _i, _i64, _i64, _p,
                                           _p]
    L.poly_debug_fail_launches.argtypes = [_i, _i]
    for name in EXPORTS:
        if name not in ("poly_status_str",):
            getattr(L, name).restype = _i
    if L.poly_abi_version() != ABI_VERSION:
        raise RuntimeError(f"{LIB_PATH}: ABI version {L.poly_abi_version()}, "
                           f"this binding expects {ABI_VERSION}; rebuild the library")
    _LIB = L
    return L


# ---- marshalling helpers ----------------------------------------------------

def _ptr(t):
    """Device (or host) address of a tensor, an int address, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


_CURRENT_STREAM = None


def _current_stream_fn():
    """A function returning the current device's current CUDA stream handle.
    torch's raw-stream query skips building a torch.cuda.Stream object (about
    2 us per call); where this torch lacks it, the public API is used."""
    global _CURRENT_STREAM
    torch = _torch()
    C = torch._C
    if hasattr(C, "_cuda_getCurrentRawStream") and hasattr(C, "_cuda_getDevice"):
        torch.cuda.init()
        raw, device = C._cuda_getCurrentRawStream, C._cuda_getDevice
        _CURRENT_STREAM = lambda: raw(device())
    else:
        _CURRENT_STREAM = lambda: torch.cuda.current_stream().cuda_stream
    return _CURRENT_STREAM


def _stream(stream):
    if stream is None:
        return (_CURRENT_STREAM or _current_stream_fn())()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != POLY_OK:
        raise PolyError(status, where)


_TORCH = None
_NDEV = None
_HALF_IDS = {}              # torch half dtypes -> POLY_F16 / POLY_BF16


def _torch():
    global _TORCH, _NDEV
    if _TORCH is None:
        import torch
        _HALF_IDS.update({torch.float16: POLY_F16, torch.bfloat16: POLY_BF16})
        _NDEV = torch.cuda.device_count() if torch.cuda.is_available() else 0
        _TORCH = torch
    return _TORCH


def _room(t, nbytes, where, name, esize=2, dtype=None):
    """Check a tensor argument before its address crosses the C ABI (which
    sees only pointers): memory of the current device or pinned host memory,
    elements of esize bytes, a declared FP16 / BF16 type that agrees with the
    call's dtype, and at least nbytes from its first element to the end of
    its storage.  Raw integer addresses are the caller's responsibility."""
    if t is None or isinstance(t, int):
        return
    torch = _torch()
    if t.is_cuda:
        if _NDEV > 1 and t.device.index != torch.cuda.current_device():
            raise ValueError(f"{where}: {name} is on cuda:{t.device.index}, the kernels run on "
                             f"the current device cuda:{torch.cuda.current_device()}")
    elif not t.is_pinned():
        raise ValueError(f"{where}: {name} must be a CUDA tensor or pinned host memory")
    tdt = t.dtype
    declared = _HALF_IDS.get(tdt)
    if declared is not None:
        if esize != 2:
            raise ValueError(f"{where}: {name} has 2-byte elements, expected {esize}")
        if dtype is not None and declared != dtype:
            raise ValueError(f"{where}: {name} is {tdt}, which is not the call's dtype")
    elif t.element_size() != esize:
        raise ValueError(f"{where}: {name} has {t.element_size()}-byte elements, expected {esize}")
    if nbytes > 0 and not (t.is_contiguous() and t.numel() * esize >= nbytes):
        # views: judge by the storage from the first element on (an expanded,
        # stride-0 tensor is judged by what it owns, not by its shape)
        avail = t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()
        if avail < nbytes:
            raise ValueError(f"{where}: {name} has {avail} bytes from its first element; the "
                             f"call touches {nbytes}")


def _extent(rows, cols, ld):
    """Elements spanned by rows x cols with leading dimension ld."""
    return (rows - 1) * ld + cols if rows > 0 and cols > 0 else 0


def _rows(t, cols):
    """Rows of a 2-D row-major view, or of a contiguous tensor of any rank
    read as [numel / cols, cols] (e.g. [batch, tokens, hidden])."""
    if t.dim() == 2:
        return t.shape[0]
    if t.is_contiguous() and cols > 0:
        return t.numel() // cols
    raise ValueError("tensor must be 2-D row-major or contiguous")


def _ld(t, cols):
    """Leading dimension (elements) of a 2-D row-major view."""
    if t is None or isinstance(t, int):
        return cols
    if t.dim() == 2 and t.stride(1) == 1:
        return t.stride(0)
    if t.is_contiguous():
        return cols
    raise ValueError("tensor must be row-major with unit column stride")


# ---- entry points (same names as the C ABI) ----------------------------------

def poly_fit_defaults():
    o = PolyFitOpts()
    _check(lib().poly_fit_defaults(ctypes.byref(o)), "poly_fit_defaults")
    return o


def poly_fit(fn, direction, dtype, degree, opts=None):
    p = PolyProgram()
    st = lib().poly_fit(fn, direction, dtype, degree,
                        ctypes.byref(opts) if opts is not None else None, ctypes.byref(p))
    _check(st, "poly_fit")
    return p


def poly_set_program(p: PolyProgram):
    _check(lib().poly_set_program(ctypes.byref(p)), "poly_set_program")


def poly_get_program(fn, direction, dtype):
    p = PolyProgram()
    _check(lib().poly_get_program(fn, direction, dtype, ctypes.byref(p)), "poly_get_program")
    return p


def poly_reset_programs():
    _check(lib().poly_reset_programs(), "poly_reset_programs")


def poly_set_swiglu_variant(variant):
    _check(lib().poly_set_swiglu_variant(variant), "poly_set_swiglu_variant")


def poly_get_swiglu_variant():
    return lib().poly_get_swiglu_variant()


def poly_act_fwd(fn, dtype, x, y, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (y, "y")):
        _room(t, 2 * n, "poly_act_fwd", nm, dtype=dtype)
    _check(lib().poly_act_fwd(fn, dtype, _ptr(x), _ptr(y), n, _stream(stream)), "poly_act_fwd")


def poly_act_bwd(fn, dtype, x, dy, dx, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (dy, "dy"), (dx, "dx")):
        _room(t, 2 * n, "poly_act_bwd", nm, dtype=dtype)
    _check(lib().poly_act_bwd(fn, dtype, _ptr(x), _ptr(dy), _ptr(dx), n, _stream(stream)),
           "poly_act_bwd")


def poly_ctrl_act_fwd(fn, dtype, x, y, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (y, "y")):
        _room(t, 2 * n, "poly_ctrl_act_fwd", nm, dtype=dtype)
    _check(lib().poly_ctrl_act_fwd(fn, dtype, _ptr(x), _ptr(y), n, _stream(stream)),
           "poly_ctrl_act_fwd")


def poly_ctrl_act_bwd(fn, dtype, x, dy, dx, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (dy, "dy"), (dx, "dx")):
        _room(t, 2 * n, "poly_ctrl_act_bwd", nm, dtype=dtype)
    _check(lib().poly_ctrl_act_bwd(fn, dtype, _ptr(x), _ptr(dy), _ptr(dx), n, _stream(stream)),
           "poly_ctrl_act_bwd")


def poly_ctrl_act_fwd_v(variant, fn, dtype, x, y, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (y, "y")):
        _room(t, 2 * n, "poly_ctrl_act_fwd_v", nm, dtype=dtype)
    _check(lib().poly_ctrl_act_fwd_v(variant, fn, dtype, _ptr(x), _ptr(y), n, _stream(stream)),
           "poly_ctrl_act_fwd_v")


def poly_ctrl_act_bwd_v(variant, fn, dtype, x, dy, dx, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (dy, "dy"), (dx, "dx")):
        _room(t, 2 * n, "poly_ctrl_act_bwd_v", nm, dtype=dtype)
    _check(lib().poly_ctrl_act_bwd_v(variant, fn, dtype, _ptr(x), _ptr(dy), _ptr(dx), n,
                                     _stream(stream)), "poly_ctrl_act_bwd_v")


def _swiglu_fwd(cfn, dtype, g, u, y, rows, cols, ldg, ldu, ldy, stream, name):
    cols = g.shape[-1] if cols is None else cols
    rows = _rows(g, cols) if rows is None else rows
    ldg = _ld(g, cols) if ldg is None else ldg
    ldu = _ld(u, cols) if ldu is None else ldu
    ldy = _ld(y, cols) if ldy is None else ldy
    for t, nm, ld in ((g, "g", ldg), (u, "u", ldu), (y, "y", ldy)):
        _room(t, 2 * _extent(rows, cols, ld), name, nm, dtype=dtype)
    _check(cfn(dtype, _ptr(g), _ptr(u), _ptr(y), rows, cols, ldg, ldu, ldy, _stream(stream)),
           name)


def poly_swiglu_fwd(dtype, g, u, y, rows=None, cols=None, ldg=None, ldu=None, ldy=None,
                    stream=None):
    _swiglu_fwd(lib().poly_swiglu_fwd, dtype, g, u, y, rows, cols, ldg, ldu, ldy, stream,
                "poly_swiglu_fwd")


def poly_ctrl_swiglu_fwd(dtype, g, u, y, rows=None, cols=None, ldg=None, ldu=None, ldy=None,
                         stream=None):
    _swiglu_fwd(lib().poly_ctrl_swiglu_fwd, dtype, g, u, y, rows, cols, ldg, ldu, ldy, stream,
                "poly_ctrl_swiglu_fwd")


def poly_swiglu_fwd_v(variant, dtype, g, u, y, rows=None, cols=None, ldg=None, ldu=None,
                      ldy=None, stream=None):
    cfn = lambda *a: lib().poly_swiglu_fwd_v(variant, *a)
    _swiglu_fwd(cfn, dtype, g, u, y, rows, cols, ldg, ldu, ldy, stream, "poly_swiglu_fwd_v")


def poly_ctrl_swiglu_fwd_v(variant, dtype, g, u, y, rows=None, cols=None, ldg=None, ldu=None,
                           ldy=None, stream=None):
    cfn = lambda *a: lib().poly_ctrl_swiglu_fwd_v(variant, *a)
    _swiglu_fwd(cfn, dtype, g, u, y, rows, cols, ldg, ldu, ldy, stream, "poly_ctrl_swiglu_fwd_v")


def _swiglu_bwd(cfn, dtype, g, u, dy, dg, du, rows, cols, lds, stream, name):
    cols = g.shape[-1] if cols is None else cols
    rows = _rows(g, cols) if rows is None else rows
    ts = (g, u, dy, dg, du)
    lds = [(_ld(t, cols) if l is None else l) for t, l in zip(ts, lds)]
    for t, nm, ld in zip(ts, ("g", "u", "dy", "dg", "du"), lds):
        _room(t, 2 * _extent(rows, cols, ld), name, nm, dtype=dtype)
    _check(cfn(dtype, _ptr(g), _ptr(u), _ptr(dy), _ptr(dg), _ptr(du), rows, cols, *lds,
               _stream(stream)), name)


def poly_swiglu_bwd(dtype, g, u, dy, dg, du, rows=None, cols=None, ldg=None, ldu=None,
                    lddy=None, lddg=None, lddu=None, stream=None):
    _swiglu_bwd(lib().poly_swiglu_bwd, dtype, g, u, dy, dg, du, rows, cols,
                (ldg, ldu, lddy, lddg, lddu), stream, "poly_swiglu_bwd")


def poly_ctrl_swiglu_bwd(dtype, g, u, dy, dg, du, rows=None, cols=None, ldg=None, ldu=None,
                         lddy=None, lddg=None, lddu=None, stream=None):
    _swiglu_bwd(lib().poly_ctrl_swiglu_bwd, dtype, g, u, dy, dg, du, rows, cols,
                (ldg, ldu, lddy, lddg, lddu), stream, "poly_ctrl_swiglu_bwd")


def poly_swiglu_bwd_v(variant, dtype, g, u, dy, dg, du, rows=None, cols=None, ldg=None,
                      ldu=None, lddy=None, lddg=None, lddu=None, stream=None):
    cfn = lambda *a: lib().poly_swiglu_bwd_v(variant, *a)
    _swiglu_bwd(cfn, dtype, g, u, dy, dg, du, rows, cols, (ldg, ldu, lddy, lddg, lddu), stream,
                "poly_swiglu_bwd_v")


def poly_ctrl_swiglu_bwd_v(variant, dtype, g, u, dy, dg, du, rows=None, cols=None, ldg=None,
                           ldu=None, lddy=None, lddg=None, lddu=None, stream=None):
    cfn = lambda *a: lib().poly_ctrl_swiglu_bwd_v(variant, *a)
    _swiglu_bwd(cfn, dtype, g, u, dy, dg, du, rows, cols, (ldg, ldu, lddy, lddg, lddu), stream,
                "poly_ctrl_swiglu_bwd_v")


def _ragged_room(where, dtype, ts, names, seg_off, num_segments, cap_rows, cols, status):
    for t, nm in zip(ts, names):
        _room(t, 2 * cap_rows * cols, where, nm, dtype=dtype)
    _room(seg_off, 4 * (num_segments + 1), where, "seg_off", esize=4)
    _room(status, 4, where, "status", esize=4)


def poly_swiglu_fwd_ragged(dtype, g, u, y, seg_off, num_segments=None, cap_rows=None,
                           cols=None, status=None, stream=None):
    num_segments = seg_off.numel() - 1 if num_segments is None else num_segments
    cols = g.shape[-1] if cols is None else cols
    cap_rows = _rows(g, cols) if cap_rows is None else cap_rows
    _ragged_room("poly_swiglu_fwd_ragged", dtype, (g, u, y), ("g", "u", "y"), seg_off,
                 num_segments, cap_rows, cols, status)
    _check(lib().poly_swiglu_fwd_ragged(dtype, _ptr(g), _ptr(u), _ptr(y), _ptr(seg_off),
                                        num_segments, cap_rows, cols, _ptr(status),
                                        _stream(stream)), "poly_swiglu_fwd_ragged")


def poly_swiglu_bwd_ragged(dtype, g, u, dy, dg, du, seg_off, num_segments=None, cap_rows=None,
                           cols=None, status=None, stream=None):
    num_segments = seg_off.numel() - 1 if num_segments is None else num_segments
    cols = g.shape[-1] if cols is None else cols
    cap_rows = _rows(g, cols) if cap_rows is None else cap_rows
    _ragged_room("poly_swiglu_bwd_ragged", dtype, (g, u, dy, dg, du), ("g", "u", "dy", "dg", "du"),
                 seg_off, num_segments, cap_rows, cols, status)
    _check(lib().poly_swiglu_bwd_ragged(dtype, _ptr(g), _ptr(u), _ptr(dy), _ptr(dg), _ptr(du),
                                        _ptr(seg_off), num_segments, cap_rows, cols,
                                        _ptr(status), _stream(stream)),
           "poly_swiglu_bwd_ragged")


def poly_swiglu_fwd_ragged_v(variant, dtype, g, u, y, seg_off, num_segments=None,
                             cap_rows=None, cols=None, status=None, stream=None):
    num_segments = seg_off.numel() - 1 if num_segments is None else num_segments
    cols = g.shape[-1] if cols is None else cols
    cap_rows = _rows(g, cols) if cap_rows is None else cap_rows
    _ragged_room("poly_swiglu_fwd_ragged_v", dtype, (g, u, y), ("g", "u", "y"), seg_off,
                 num_segments, cap_rows, cols, status)
    _check(lib().poly_swiglu_fwd_ragged_v(variant, dtype, _ptr(g), _ptr(u), _ptr(y),
                                          _ptr(seg_off), num_segments, cap_rows, cols,
                                          _ptr(status), _stream(stream)),
           "poly_swiglu_fwd_ragged_v")


def poly_swiglu_bwd_ragged_v(variant, dtype, g, u, dy, dg, du, seg_off, num_segments=None,
                             cap_rows=None, cols=None, status=None, stream=None):
    num_segments = seg_off.numel() - 1 if num_segments is None else num_segments
    cols = g.shape[-1] if cols is None else cols
    cap_rows = _rows(g, cols) if cap_rows is None else cap_rows
    _ragged_room("poly_swiglu_bwd_ragged_v", dtype, (g, u, dy, dg, du),
                 ("g", "u", "dy", "dg", "du"), seg_off, num_segments, cap_rows, cols, status)
    _check(lib().poly_swiglu_bwd_ragged_v(variant, dtype, _ptr(g), _ptr(u), _ptr(dy), _ptr(dg),
                                          _ptr(du), _ptr(seg_off), num_segments, cap_rows, cols,
                                          _ptr(status), _stream(stream)),
           "poly_swiglu_bwd_ragged_v")


def poly_diag_stream_peak(nin, a, b, out, n=None, reps=1, inflight=2, stream=None):
    """reps streaming passes out = a (nin 1) or a ^ b (nin 2) over n 16-bit
    elements with `inflight` 16-byte chunks per input in flight per thread
    (the bandwidth probe)."""
    n = a.numel() if n is None else n
    for t, nm in ((a, "a"), (b, "b"), (out, "out")):
        _room(t, 2 * n, "poly_diag_stream_peak", nm)
    _check(lib().poly_diag_stream_peak(nin, inflight, _ptr(a), _ptr(b), _ptr(out), n, reps,
                                       _stream(stream)), "poly_diag_stream_peak")


def poly_ragged_zero_outside(out, seg_off, num_segments=None, cap_rows=None, cols=None,
                             stream=None):
    """Zero the rows of out [cap_rows, cols] outside [seg_off[0], seg_off[E])."""
    num_segments = seg_off.numel() - 1 if num_segments is None else num_segments
    cap_rows = out.shape[0] if cap_rows is None else cap_rows
    cols = out.shape[1] if cols is None else cols
    _room(out, 2 * cap_rows * cols, "poly_ragged_zero_outside", "out")
    _room(seg_off, 4 * (num_segments + 1), "poly_ragged_zero_outside", "seg_off", esize=4)
    _check(lib().poly_ragged_zero_outside(_ptr(out), _ptr(seg_off), num_segments, cap_rows, cols,
                                          _stream(stream)), "poly_ragged_zero_outside")


def poly_diag_packed(op, dtype, a, b, c, out, n=None, stream=None):
    n = a.numel() if n is None else n
    for t, nm in ((a, "a"), (b, "b"), (c, "c"), (out, "out")):
        _room(t, 2 * n, "poly_diag_packed", nm, dtype=dtype)
    _check(lib().poly_diag_packed(op, dtype, _ptr(a), _ptr(b), _ptr(c), _ptr(out), n,
                                  _stream(stream)), "poly_diag_packed")


def poly_debug_fail_launches(cuda_error, count):
    """Make the next `count` launches report `cuda_error` without running;
    returns how many injected failures were still pending."""
    st = lib().poly_debug_fail_launches(cuda_error, count)
    if st < 0:
        _check(st, "poly_debug_fail_launches")
    return st


def poly_derive_program(fwd: PolyProgram):
    out = PolyProgram()
    _check(lib().poly_derive_program(ctypes.byref(fwd), ctypes.byref(out)), "poly_derive_program")
    return out


def poly_softcap_fwd(dtype, alpha, x, y, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (y, "y")):
        _room(t, 2 * n, "poly_softcap_fwd", nm, dtype=dtype)
    _check(lib().poly_softcap_fwd(dtype, float(alpha), _ptr(x), _ptr(y), n, _stream(stream)),
           "poly_softcap_fwd")


def poly_softcap_bwd(dtype, alpha, x, dy, dx, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (dy, "dy"), (dx, "dx")):
        _room(t, 2 * n, "poly_softcap_bwd", nm, dtype=dtype)
    _check(lib().poly_softcap_bwd(dtype, float(alpha), _ptr(x), _ptr(dy), _ptr(dx), n,
                                  _stream(stream)), "poly_softcap_bwd")


def poly_exp2(core, x, y, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (y, "y")):
        _room(t, 4 * n, "poly_exp2", nm, esize=4)
    _check(lib().poly_exp2(core, _ptr(x), _ptr(y), n, _stream(stream)), "poly_exp2")


def poly_ctrl_exp2(x, y, n=None, stream=None):
    n = x.numel() if n is None else n
    for t, nm in ((x, "x"), (y, "y")):
        _room(t, 4 * n, "poly_ctrl_exp2", nm, esize=4)
    _check(lib().poly_ctrl_exp2(_ptr(x), _ptr(y), n, _stream(stream)), "poly_ctrl_exp2")


def poly_rope_turn_increments(head_dim, base=10000.0):
    """Host array of the D/2 Q0.32 turn increments (numpy uint32)."""
    import numpy as np
    out = np.zeros(head_dim // 2, dtype=np.uint32)
    _check(lib().poly_rope_turn_increments(head_dim, float(base), out.ctypes.data),
           "poly_rope_turn_increments")
    return out


def poly_rope_programs():
    s = (ctypes.c_uint16 * 3)()
    c = (ctypes.c_uint16 * 3)()
    _check(lib().poly_rope_programs(ctypes.cast(s, ctypes.c_void_p), ctypes.cast(c, ctypes.c_void_p)),
           "poly_rope_programs")
    return list(s), list(c)


def _rope(fn, name, variant, q, k, q_out, k_out, delta, cos_tab, sin_tab, shape,
          pos_offset, stream):
    batch, seq, hq, hkv, head_dim = shape
    nq, nk = batch * seq * hq * head_dim, batch * seq * hkv * head_dim
    for t, nm, cnt in ((q, "q", nq), (k, "k", nk), (q_out, "q_out", nq), (k_out, "k_out", nk),
                       (cos_tab, "cos_tab", seq * head_dim // 2),
                       (sin_tab, "sin_tab", seq * head_dim // 2)):
        _room(t, 2 * cnt, name, nm, dtype=POLY_F16)          # the RoPE kernels are FP16
    _room(delta, 4 * (head_dim // 2), name, "delta", esize=4)
    _check(fn(variant, _ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), _ptr(delta), _ptr(cos_tab),
              _ptr(sin_tab), batch, seq, hq, hkv, head_dim, pos_offset, _stream(stream)), name)


def poly_rope_fwd(variant, q, k, q_out, k_out, delta, cos_tab=None, sin_tab=None, batch=None,
                  seq=None, hq=None, hkv=None, head_dim=None, pos_offset=0, stream=None):
    """q [B, S, Hq, D], k [B, S, Hkv, D] -> q_out [B, Hq, S, D], k_out [B, Hkv, S, D]."""
    shape = (batch if batch is not None else q.shape[0], seq if seq is not None else q.shape[1],
             hq if hq is not None else q.shape[2], hkv if hkv is not None else k.shape[2],
             head_dim if head_dim is not None else q.shape[3])
    _rope(lib().poly_rope_fwd, "poly_rope_fwd", variant, q, k, q_out, k_out, delta, cos_tab,
          sin_tab, shape, pos_offset, stream)


def poly_rope_bwd(variant, dq, dk, dq_out, dk_out, delta, cos_tab=None, sin_tab=None, batch=None,
                  seq=None, hq=None, hkv=None, head_dim=None, pos_offset=0, stream=None):
    """dq [B, Hq, S, D], dk [B, Hkv, S, D] -> dq_out [B, S, Hq, D], dk_out [B, S, Hkv, D]."""
    shape = (batch if batch is not None else dq.shape[0], seq if seq is not None else dq.shape[2],
             hq if hq is not None else dq.shape[1], hkv if hkv is not None else dk.shape[1],
             head_dim if head_dim is not None else dq.shape[3])
    _rope(lib().poly_rope_bwd, "poly_rope_bwd", variant, dq, dk, dq_out, dk_out, delta, cos_tab,
          sin_tab, shape, pos_offset, stream)

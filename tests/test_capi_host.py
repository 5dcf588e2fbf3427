"""Host-side tests of libpolyact: symbol exports, argument validation and the
C++ fitter.  No compute call reaches the GPU: every device entry point is
called only with arguments that fail validation (or with n == 0), which the
library rejects on the host before any CUDA call."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import golden_programs as gp
from polynomial_activation_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "polyact.h")


@pytest.fixture(scope="module")
def L():
    return B.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(poly_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    declared = header_functions()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(B.EXPORTS) == declared


def test_status_strings(L):
    for st in (B.POLY_OK, B.POLY_EINVAL, B.POLY_ENOPROG, B.POLY_ECUDA, B.POLY_ENOFIT):
        assert L.poly_status_str(st).startswith(b"POLY_")
    assert L.poly_status_str(12345) == b"unknown status"


def test_forms_and_default_degrees(L):
    assert [L.poly_form_of(f, 0) for f in range(4)] == [B.POLY_FORM_CO, B.POLY_FORM_O,
                                                        B.POLY_FORM_HX, B.POLY_FORM_HX]
    assert [L.poly_form_of(f, 1) for f in range(4)] == [B.POLY_FORM_E, B.POLY_FORM_E,
                                                        B.POLY_FORM_CO, B.POLY_FORM_CO]
    assert [L.poly_default_degree(f, 0) for f in range(4)] == [3, 4, 3, 5]
    assert [L.poly_default_degree(f, 1) for f in range(4)] == [4, 4, 4, 4]
    assert L.poly_form_of(7, 0) == B.POLY_EINVAL
    assert L.poly_default_degree(0, 2) == B.POLY_EINVAL


@pytest.mark.parametrize("k", sorted(json.load(open(gp.PATH))))
def test_cpp_fitter_reproduces_oracle_programs(k):
    """The library's C++ fitter (independent code: integer soft-float,
    Householder QR) accepts exactly the program the oracle fitter accepts."""
    g = json.load(open(gp.PATH))[k]
    dt = B.POLY_F16 if g["fmt"] == "f16" else B.POLY_BF16
    p = B.poly_fit(g["fn"], g["direction"], dt, g["degree"])
    assert p.coefficients() == g["coef"]
    assert p.lc_bits == g["lc_bits"] and p.li == g["li"] and p.lc == g["lc"]
    assert p.form == B.lib().poly_form_of(g["fn"], g["direction"])
    assert p.rank == g["rank"]
    assert p.stated_max_abs_err == pytest.approx(g["stated_max_abs_err"], rel=1e-12)
    assert p.search_score == pytest.approx(g["search_score"], rel=1e-12)
    assert p.table2 == pytest.approx(g["table2"], rel=1e-9)


@pytest.mark.parametrize("fn,D,top_k,refine", [(0, 3, 8, 0), (3, 5, 8, 0), (0, 4, 0, 2),
                                                (1, 4, 3, 1)])
def test_cpp_fitter_options_match_oracle(fn, D, top_k, refine):
    """top_k (deployed replay of the k best split-order candidates) and
    lc_refine_ulps (clamp moved by up to k BF16 ulps) select the same program
    in the C++ fitter as in the oracle fitter."""
    from oracle import fit
    o = B.poly_fit_defaults()
    assert (o.top_k, o.lc_refine_ulps) == (0, 0)
    o.top_k, o.lc_refine_ulps = top_k, refine
    p = B.poly_fit(fn, 0, B.POLY_BF16, D, o)
    q = fit.search(fn, 0, "bf16", D, top_k=top_k, lc_refine_ulps=refine)
    assert p.coefficients() == [int(c) for c in q.coef]
    assert (p.li, p.lc, p.lc_bits, p.rank) == (q.li, q.lc, int(q.lc_bits), q.info["rank"])
    assert p.deployed_score == q.info["deployed_score"]


def test_fit_is_deterministic_and_registry_roundtrip():
    a = B.poly_fit(B.POLY_TANH, B.POLY_FWD, B.POLY_BF16, 4)
    b = B.poly_fit(B.POLY_TANH, B.POLY_FWD, B.POLY_BF16, 4)
    assert bytes(a) == bytes(b)
    B.poly_reset_programs()
    got = B.poly_get_program(B.POLY_TANH, B.POLY_FWD, B.POLY_BF16)
    assert bytes(got) == bytes(a)
    # install a different-degree program and read it back
    c = B.poly_fit(B.POLY_TANH, B.POLY_FWD, B.POLY_BF16, 6)
    B.poly_set_program(c)
    assert B.poly_get_program(B.POLY_TANH, B.POLY_FWD, B.POLY_BF16).degree == 6
    B.poly_reset_programs()
    assert B.poly_get_program(B.POLY_TANH, B.POLY_FWD, B.POLY_BF16).degree == 4


def test_fit_argument_errors(L):
    p = B.PolyProgram()
    assert L.poly_fit(9, 0, 0, 3, None, ctypes.byref(p)) == B.POLY_EINVAL
    assert L.poly_fit(0, 2, 0, 3, None, ctypes.byref(p)) == B.POLY_EINVAL
    assert L.poly_fit(0, 0, 5, 3, None, ctypes.byref(p)) == B.POLY_EINVAL
    assert L.poly_fit(0, 0, 0, 2, None, ctypes.byref(p)) == B.POLY_EINVAL
    assert L.poly_fit(0, 0, 0, 7, None, ctypes.byref(p)) == B.POLY_EINVAL
    assert L.poly_fit(0, 0, 0, 3, None, None) == B.POLY_EINVAL
    o = B.poly_fit_defaults()
    o.li_step = 0.0
    assert L.poly_fit(0, 0, 0, 3, ctypes.byref(o), ctypes.byref(p)) == B.POLY_EINVAL
    assert L.poly_fit_defaults(None) == B.POLY_EINVAL
    for field, value in (("top_k", -1), ("lc_refine_ulps", -1), ("lc_refine_ulps", 65)):
        o = B.poly_fit_defaults()
        setattr(o, field, value)
        assert L.poly_fit(0, 0, 0, 3, ctypes.byref(o), ctypes.byref(p)) == B.POLY_EINVAL
    assert L.poly_abi_version() == B.ABI_VERSION == 4
    # no admissible clamp at all: Lc starts above Li + 1
    o = B.poly_fit_defaults()
    o.li_max, o.lc_min = 2.0, 5.0
    assert L.poly_fit(0, 0, 1, 3, ctypes.byref(o), ctypes.byref(p)) == B.POLY_ENOFIT


def test_set_program_rejects_inconsistent_descriptors(L):
    good = B.poly_fit(B.POLY_SIGMOID, B.POLY_FWD, B.POLY_BF16, 3)
    for field, value in (("form", B.POLY_FORM_E), ("degree", 2), ("degree", 7),
                         ("version", 99), ("fn", 8), ("dtype", 4)):
        bad = B.PolyProgram.from_buffer_copy(bytes(good))
        setattr(bad, field, value)
        assert L.poly_set_program(ctypes.byref(bad)) == B.POLY_ENOPROG, field
    bad = B.PolyProgram.from_buffer_copy(bytes(good))
    bad.coef[0] = 0x3F80                                # c_0 must be 0 for the CO form
    assert L.poly_set_program(ctypes.byref(bad)) == B.POLY_ENOPROG
    assert L.poly_set_program(None) == B.POLY_EINVAL
    B.poly_reset_programs()


def test_set_program_rejects_bad_clamps(L):
    """The clamp Lc must be a finite positive target-format value equal to
    lc, no further than Li + 1 (§3.2 step 6): a descriptor breaking any of
    these would make every later call return NaN or unclamped values."""
    good = B.poly_fit(B.POLY_SIGMOID, B.POLY_FWD, B.POLY_BF16, 3)
    assert L.poly_set_program(ctypes.byref(good)) == B.POLY_OK
    cases = [
        ("lc_bits", 0x7FC0, None, None),          # NaN
        ("lc_bits", 0x7F80, None, None),          # +inf
        ("lc_bits", 0xFF80, None, None),          # -inf
        ("lc_bits", 0xBF80, None, None),          # -1
        ("lc_bits", 0x0000, None, None),          # +0
        ("lc_bits", 0x8000, None, None),          # -0
        ("lc", good.lc + 0.25, None, None),       # lc disagrees with lc_bits
        ("li", good.lc - 1.5, None, None),        # Lc > Li + 1
        ("li", float("nan"), None, None),
        ("li", -1.0, None, None),
    ]
    try:
        for field, value, _, _ in cases:
            bad = B.PolyProgram.from_buffer_copy(bytes(good))
            setattr(bad, field, value)
            if field == "lc_bits":
                bad.lc = float("nan") if value in (0x7FC0,) else bad.lc
            assert L.poly_set_program(ctypes.byref(bad)) == B.POLY_ENOPROG, (field, value)
        # the boundary Lc = Li + 1 itself is accepted
        edge = B.PolyProgram.from_buffer_copy(bytes(good))
        edge.li = good.lc - 1.0
        assert L.poly_set_program(ctypes.byref(edge)) == B.POLY_OK
        # derivation checks the forward program the same way
        bad = B.PolyProgram.from_buffer_copy(bytes(good))
        bad.lc_bits = 0x7F80
        out = B.PolyProgram()
        assert L.poly_derive_program(ctypes.byref(bad), ctypes.byref(out)) == B.POLY_ENOPROG
    finally:
        B.poly_reset_programs()


FAKE = 0x7F0000001000          # never dereferenced: every call below fails validation


def test_device_calls_reject_bad_arguments_on_host(L):
    s = None
    # bad enums
    assert L.poly_act_fwd(9, 0, FAKE, FAKE + 4096, 8, s) == B.POLY_EINVAL
    assert L.poly_act_fwd(0, 3, FAKE, FAKE + 4096, 8, s) == B.POLY_EINVAL
    # negative size, null pointers
    assert L.poly_act_fwd(0, 0, FAKE, FAKE + 4096, -1, s) == B.POLY_EINVAL
    assert L.poly_act_fwd(0, 0, None, FAKE, 8, s) == B.POLY_EINVAL
    assert L.poly_act_bwd(0, 0, FAKE, None, FAKE + 4096, 8, s) == B.POLY_EINVAL
    # odd (misaligned for 16-bit elements) addresses
    assert L.poly_act_fwd(0, 0, FAKE + 1, FAKE + 4096, 8, s) == B.POLY_EINVAL
    # partial overlap of output and input
    assert L.poly_act_fwd(0, 0, FAKE, FAKE + 2, 8, s) == B.POLY_EINVAL
    assert L.poly_act_bwd(0, 0, FAKE, FAKE + 4096, FAKE + 4098, 8, s) == B.POLY_EINVAL
    # SwiGLU: ld < cols, overlapping outputs, negative rows
    assert L.poly_swiglu_fwd(1, FAKE, FAKE + 8192, FAKE + 16384, 4, 16, 8, 16, 16, s) == B.POLY_EINVAL
    assert L.poly_swiglu_fwd(1, FAKE, FAKE + 8192, FAKE + 16384, -1, 16, 16, 16, 16, s) == B.POLY_EINVAL
    assert L.poly_swiglu_bwd(1, FAKE, FAKE + 8192, FAKE + 16384, FAKE + 24576, FAKE + 24578,
                             4, 16, 16, 16, 16, 16, 16, s) == B.POLY_EINVAL
    assert L.poly_swiglu_fwd(7, FAKE, FAKE + 8192, FAKE + 16384, 4, 16, 16, 16, 16, s) == B.POLY_EINVAL
    # ragged: null offsets, negative segments
    assert L.poly_swiglu_fwd_ragged(1, FAKE, FAKE + 8192, FAKE + 16384, None, 4, 4, 16, None, s) == B.POLY_EINVAL
    assert L.poly_swiglu_fwd_ragged(1, FAKE, FAKE + 8192, FAKE + 16384, FAKE + 30000, -1, 4, 16, None, s) == B.POLY_EINVAL
    # zero fill outside the segments: null / odd buffer, null offsets, negative sizes
    assert L.poly_ragged_zero_outside(None, FAKE, 4, 4, 16, s) == B.POLY_EINVAL
    assert L.poly_ragged_zero_outside(FAKE + 1, FAKE + 30000, 4, 4, 16, s) == B.POLY_EINVAL
    assert L.poly_ragged_zero_outside(FAKE, None, 4, 4, 16, s) == B.POLY_EINVAL
    assert L.poly_ragged_zero_outside(FAKE, FAKE + 30000, -1, 4, 16, s) == B.POLY_EINVAL
    assert L.poly_ragged_zero_outside(FAKE, FAKE + 30000, 4, -4, 16, s) == B.POLY_EINVAL
    assert L.poly_ragged_zero_outside(FAKE, FAKE + 30000, 4, 1 << 40, 1 << 40, s) == B.POLY_EINVAL
    # controls share the validation
    assert L.poly_ctrl_act_fwd(0, 0, FAKE + 1, FAKE + 4096, 8, s) == B.POLY_EINVAL
    assert L.poly_ctrl_swiglu_bwd(1, FAKE, FAKE + 8192, FAKE + 16384, FAKE + 24576, FAKE + 24578,
                                  4, 16, 16, 16, 16, 16, 16, s) == B.POLY_EINVAL
    # diagnostic: FMA needs c, bad op
    assert L.poly_diag_packed(0, 0, FAKE, FAKE + 4096, None, FAKE + 8192, 8, s) == B.POLY_EINVAL
    assert L.poly_diag_packed(9, 0, FAKE, FAKE + 4096, FAKE, FAKE + 8192, 8, s) == B.POLY_EINVAL
    # per-call variants: unknown SwiGLU rule or control variant
    assert L.poly_swiglu_fwd_v(2, 1, FAKE, FAKE + 8192, FAKE + 16384, 4, 16, 16, 16, 16,
                               s) == B.POLY_EINVAL
    assert L.poly_swiglu_bwd_v(-1, 1, FAKE, FAKE + 8192, FAKE + 16384, FAKE + 24576,
                               FAKE + 32768, 4, 16, 16, 16, 16, 16, 16, s) == B.POLY_EINVAL
    assert L.poly_swiglu_fwd_ragged_v(5, 1, FAKE, FAKE + 8192, FAKE + 16384, FAKE + 30000, 4, 4,
                                      16, None, s) == B.POLY_EINVAL
    assert L.poly_swiglu_bwd_ragged_v(5, 1, FAKE, FAKE + 8192, FAKE + 16384, FAKE + 24576,
                                      FAKE + 32768, FAKE + 40000, 4, 4, 16, None,
                                      s) == B.POLY_EINVAL
    assert L.poly_ctrl_act_fwd_v(2, 0, 0, FAKE, FAKE + 4096, 8, s) == B.POLY_EINVAL
    assert L.poly_ctrl_act_bwd_v(-1, 0, 0, FAKE, FAKE + 4096, FAKE + 8192, 8, s) == B.POLY_EINVAL
    assert L.poly_ctrl_swiglu_fwd_v(3, 1, FAKE, FAKE + 8192, FAKE + 16384, 4, 16, 16, 16, 16,
                                    s) == B.POLY_EINVAL
    assert L.poly_ctrl_swiglu_bwd_v(3, 1, FAKE, FAKE + 8192, FAKE + 16384, FAKE + 24576,
                                    FAKE + 32768, 4, 16, 16, 16, 16, 16, 16, s) == B.POLY_EINVAL
    # the packed control shares the validation
    assert L.poly_ctrl_act_fwd_v(1, 0, 0, FAKE + 1, FAKE + 4096, 8, s) == B.POLY_EINVAL
    assert L.poly_ctrl_act_fwd_v(1, 0, 0, FAKE, FAKE + 2, 8, s) == B.POLY_EINVAL
    # streaming probe: nin, n a multiple of 8, reps range, 16-byte alignment, overlap
    for args in ((3, 2, FAKE, FAKE, FAKE + 8192, 64, 1), (1, 2, FAKE, None, FAKE + 8192, 60, 1),
                 (1, 2, FAKE, None, FAKE + 8192, 64, 0), (1, 2, FAKE, None, FAKE + 8192, 64, 1 << 21),
                 (1, 2, FAKE + 8, None, FAKE + 8192, 64, 1),
                 (2, 2, FAKE, FAKE + 4104, FAKE + 8192, 64, 1),
                 (2, 2, FAKE, None, FAKE + 8192, 64, 1), (1, 2, FAKE, None, FAKE + 64, 64, 1),
                 (1, 2, FAKE, None, FAKE + 8192, -8, 1), (1, 2, FAKE, None, FAKE + 8192, 1 << 34, 1),
                 (1, 3, FAKE, None, FAKE + 8192, 64, 1), (1, 16, FAKE, None, FAKE + 8192, 64, 1),
                 (1, 0, FAKE, None, FAKE + 8192, 64, 1)):
        assert L.poly_diag_stream_peak(*args, s) == B.POLY_EINVAL, args


def test_oversized_and_wrapping_arguments_are_rejected(L):
    """Extents above 2^46 elements, products that would overflow and spans
    that would wrap the address space fail validation on the host."""
    s = None
    before = L.poly_last_cuda_error()
    top = 0xFFFFFFFFFFFFF000                    # even; 4,096 FP16 elements wrap past 2^64
    assert L.poly_act_fwd(0, 0, FAKE, FAKE + (1 << 49), 1 << 47, s) == B.POLY_EINVAL
    assert L.poly_act_fwd(0, 0, top, FAKE, 4096, s) == B.POLY_EINVAL
    assert L.poly_act_bwd(0, 0, FAKE, top, FAKE + 4096, 4096, s) == B.POLY_EINVAL
    assert L.poly_swiglu_fwd(1, FAKE, FAKE + 8192, FAKE + 16384, 1 << 45, 16, 16, 16, 16,
                             s) == B.POLY_EINVAL
    assert L.poly_swiglu_fwd(1, FAKE, FAKE + 8192, FAKE + 16384, 4, 16, 1 << 47, 16, 16,
                             s) == B.POLY_EINVAL
    assert L.poly_swiglu_fwd_ragged(1, FAKE, FAKE + 8192, FAKE + 16384, FAKE + 30000, 4,
                                    1 << 40, 1 << 10, None, s) == B.POLY_EINVAL
    assert L.poly_exp2(B.POLY_EXP2_D1, FAKE, FAKE + (1 << 50), 1 << 47, s) == B.POLY_EINVAL
    assert L.poly_softcap_fwd(0, 30.0, FAKE, FAKE + (1 << 49), 1 << 47, s) == B.POLY_EINVAL
    assert L.poly_diag_packed(1, 0, FAKE, FAKE, None, top, 4096, s) == B.POLY_EINVAL
    for batch, seq, hq, hkv, d, pos in ((1 << 20, 1 << 20, 1 << 10, 0, 128, 0),
                                        (1, 16, 1, 1, 8, 1 << 62),
                                        (1, 1 << 40, 1, 0, 8, 0)):
        assert L.poly_rope_fwd(B.POLY_ROPE_POLY, FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288,
                               FAKE + 16384, None, None, batch, seq, hq, hkv, d, pos,
                               s) == B.POLY_EINVAL
    assert L.poly_last_cuda_error() == before


def test_interleaved_halves_are_disjoint_partial_overlap_is_not(L):
    """Gate and up (and their gradients) as the two halves of one [T, 2H]
    buffer with ld = 2H share no element and pass validation -- shown by an
    injected launch failure, which only a call that reached its launch
    consumes -- while views whose rows overlap by one chunk are refused."""
    T, H = 16, 64
    gu, dgu, dy = FAKE, FAKE + (1 << 20), FAKE + (2 << 20)
    assert L.poly_debug_fail_launches(777, 1) == 0
    try:
        st = L.poly_swiglu_bwd(1, gu, gu + 2 * H, dy, dgu, dgu + 2 * H, T, H, 2 * H, 2 * H, H,
                               2 * H, 2 * H, None)
        assert st == B.POLY_ECUDA and L.poly_last_cuda_error() == 777
        assert L.poly_debug_fail_launches(777, 0) == 0            # consumed by that call
        # du shifted 8 elements left: its rows overlap the end of dg's rows
        assert L.poly_swiglu_bwd(1, gu, gu + 2 * H, dy, dgu, dgu + 2 * (H - 8), T, H, 2 * H,
                                 2 * H, H, 2 * H, 2 * H, None) == B.POLY_EINVAL
        # output over an input's gap-free region: y on top of gate's rows
        assert L.poly_swiglu_fwd(1, gu, gu + 2 * H, gu + 16, T, H, 2 * H, 2 * H, 2 * H,
                                 None) == B.POLY_EINVAL
    finally:
        L.poly_debug_fail_launches(777, 0)


def test_binding_refuses_pageable_host_tensors():
    """The binding passes only device or pinned host memory to the library:
    an ordinary CPU tensor is refused before any call."""
    import torch
    x = torch.zeros(16, dtype=torch.float16)
    with pytest.raises(ValueError, match="pinned"):
        B.poly_act_fwd(B.POLY_SIGMOID, B.POLY_F16, x, x.clone())


def test_empty_calls_are_no_ops(L):
    """n == 0 / rows == 0 return POLY_OK without touching CUDA (no GPU here)."""
    s = None
    before = L.poly_last_cuda_error()
    assert L.poly_act_fwd(0, 0, None, None, 0, s) == B.POLY_OK
    assert L.poly_act_bwd(1, 1, None, None, None, 0, s) == B.POLY_OK
    assert L.poly_ctrl_act_fwd(3, 1, None, None, 0, s) == B.POLY_OK
    assert L.poly_swiglu_fwd(1, None, None, None, 0, 16, 16, 16, 16, s) == B.POLY_OK
    assert L.poly_swiglu_bwd(1, None, None, None, None, None, 5, 0, 0, 0, 0, 0, 0, s) == B.POLY_OK
    assert L.poly_swiglu_fwd_ragged(1, None, None, None, FAKE, 4, 0, 16, None, s) == B.POLY_OK
    assert L.poly_ragged_zero_outside(None, FAKE, 4, 0, 16, s) == B.POLY_OK
    assert L.poly_ragged_zero_outside(None, FAKE, 4, 8, 0, s) == B.POLY_OK
    assert L.poly_diag_packed(0, 0, None, None, None, None, 0, s) == B.POLY_OK
    assert L.poly_ctrl_act_fwd_v(1, 2, 0, None, None, 0, s) == B.POLY_OK
    assert L.poly_ctrl_swiglu_bwd_v(1, 1, None, None, None, None, None, 0, 8, 8, 8, 8, 8, 8,
                                    s) == B.POLY_OK
    assert L.poly_swiglu_fwd_v(1, 1, None, None, None, 0, 16, 16, 16, 16, s) == B.POLY_OK
    assert L.poly_swiglu_bwd_ragged_v(0, 1, None, None, None, None, None, FAKE, 4, 0, 16, None,
                                      s) == B.POLY_OK
    assert L.poly_diag_stream_peak(2, 2, None, None, None, 0, 1, s) == B.POLY_OK
    assert L.poly_last_cuda_error() == before


def test_failure_injection_is_consumed_only_by_launches(L):
    """Injected launch failures (poly_debug_fail_launches) wait for a call
    that would launch: invalid or empty calls leave them pending."""
    assert L.poly_debug_fail_launches(0, 1) == B.POLY_EINVAL
    assert L.poly_debug_fail_launches(-5, 1) == B.POLY_EINVAL
    assert L.poly_debug_fail_launches(701, -1) == B.POLY_EINVAL
    assert L.poly_debug_fail_launches(701, 2) == 0
    before = L.poly_last_cuda_error()            # the last POLY_ECUDA's code, per thread
    try:
        assert L.poly_act_fwd(0, 0, FAKE + 1, FAKE + 4096, 8, None) == B.POLY_EINVAL
        assert L.poly_act_fwd(0, 0, None, None, 0, None) == B.POLY_OK
        assert L.poly_last_cuda_error() == before
    finally:
        assert L.poly_debug_fail_launches(701, 0) == 2       # both still pending; cleared


def test_per_call_swiglu_rule_ignores_the_process_default(L):
    """The _v SwiGLU calls take their rule from the argument: with the
    process-wide default set to either rule, both rules validate and reach
    their launch (shown by consuming an injected launch failure), and an
    unknown rule is refused before any launch."""
    T, H = 4, 16
    g, u, dy, dg, du = (FAKE + (k << 16) for k in range(5))
    seg = FAKE + (6 << 16)
    try:
        for default in (B.POLY_SWIGLU_DIRECT, B.POLY_SWIGLU_SIGMOID):
            B.poly_set_swiglu_variant(default)
            for v in (B.POLY_SWIGLU_DIRECT, B.POLY_SWIGLU_SIGMOID):
                calls = (
                    lambda: L.poly_swiglu_fwd_v(v, 1, g, u, dg, T, H, H, H, H, None),
                    lambda: L.poly_swiglu_bwd_v(v, 0, g, u, dy, dg, du, T, H, H, H, H, H, H, None),
                    lambda: L.poly_swiglu_fwd_ragged_v(v, 1, g, u, dg, seg, 2, T, H, None, None),
                    lambda: L.poly_swiglu_bwd_ragged_v(v, 0, g, u, dy, dg, du, seg, 2, T, H, None,
                                                       None),
                )
                for call in calls:
                    assert L.poly_debug_fail_launches(812, 1) == 0
                    assert call() == B.POLY_ECUDA and L.poly_last_cuda_error() == 812
            assert B.poly_get_swiglu_variant() == default
    finally:
        L.poly_debug_fail_launches(812, 0)
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)


def test_swiglu_variant_switch(L):
    assert B.poly_get_swiglu_variant() == B.POLY_SWIGLU_DIRECT
    try:
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_SIGMOID)
        assert B.poly_get_swiglu_variant() == B.POLY_SWIGLU_SIGMOID
        assert L.poly_set_swiglu_variant(7) == B.POLY_EINVAL
        assert B.poly_get_swiglu_variant() == B.POLY_SWIGLU_SIGMOID
    finally:
        B.poly_set_swiglu_variant(B.POLY_SWIGLU_DIRECT)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("fn,D", [(0, 3), (1, 4), (2, 4), (3, 4)])
def test_derive_program_matches_oracle(L, fmt, fn, D):
    """poly_derive_program (C++) equals the oracle's differentiated program."""
    from oracle.replay import derive
    dt = B.POLY_F16 if fmt == "f16" else B.POLY_BF16
    if fn in (2, 3):        # SiLU / GELU forward are x/2 + even: not differentiable this way
        p = B.poly_fit(fn, 0, dt, 3)
        out = B.PolyProgram()
        assert L.poly_derive_program(ctypes.byref(p), ctypes.byref(out)) == B.POLY_EINVAL
        return
    p = B.poly_fit(fn, 0, dt, D)
    d = B.poly_derive_program(p)
    od = derive(gp.get(fn, 0, fmt, D))
    assert d.form == B.POLY_FORM_E and d.dir == B.POLY_BWD and d.degree == D - 1
    assert d.coefficients() == list(od.coef) and d.lc_bits == od.lc_bits
    from oracle import fit
    assert d.stated_max_abs_err == pytest.approx(fit.exhaustive_error(od)[0], rel=1e-12)
    B.poly_set_program(d)                     # degree 2 / 3 even programs install
    assert B.poly_get_program(fn, 1, dt).degree == D - 1
    B.poly_reset_programs()
    # a backward program cannot be differentiated again
    e = B.PolyProgram()
    assert L.poly_derive_program(ctypes.byref(d), ctypes.byref(e)) == B.POLY_EINVAL
    assert L.poly_derive_program(None, ctypes.byref(e)) == B.POLY_EINVAL


def test_softcap_rejects_bad_alpha(L):
    s = None
    for dt, alpha in [(0, 0.0), (0, -1.0), (0, float("nan")), (0, float("inf")),
                      (0, 1e6), (0, 1e10), (1, 1e39), (1, 1e-39)]:
        assert L.poly_softcap_fwd(dt, alpha, FAKE, FAKE + 4096, 8, s) == B.POLY_EINVAL, (dt, alpha)
        assert L.poly_softcap_bwd(dt, alpha, FAKE, FAKE + 4096, FAKE + 8192, 8, s) == B.POLY_EINVAL
    assert L.poly_softcap_fwd(0, 30.0, None, None, 0, s) == B.POLY_OK
    assert L.poly_softcap_fwd(0, 30.0, FAKE, FAKE + 2, 8, s) == B.POLY_EINVAL
    assert L.poly_softcap_bwd(1, 30.0, FAKE, None, FAKE + 8192, 8, s) == B.POLY_EINVAL


def test_exp2_rejects_bad_arguments(L):
    s = None
    assert L.poly_exp2(9, FAKE, FAKE + 4096, 8, s) == B.POLY_EINVAL
    assert L.poly_exp2(4, FAKE, FAKE + 4096, 8, s) == B.POLY_EINVAL      # control has its own call
    assert L.poly_exp2(1, FAKE + 2, FAKE + 4096, 8, s) == B.POLY_EINVAL  # not 4-byte aligned
    assert L.poly_exp2(1, FAKE, FAKE + 4, 8, s) == B.POLY_EINVAL         # partial overlap
    assert L.poly_exp2(1, None, FAKE, 8, s) == B.POLY_EINVAL
    assert L.poly_exp2(1, FAKE, FAKE, -1, s) == B.POLY_EINVAL
    assert L.poly_exp2(1, None, None, 0, s) == B.POLY_OK
    assert L.poly_ctrl_exp2(FAKE + 2, FAKE + 4096, 8, s) == B.POLY_EINVAL


def test_rope_programs_and_increments_match_oracle(L):
    from oracle import rope
    s, c = B.poly_rope_programs()
    os_, oc = rope.sincos_coefficients()
    assert tuple(s) == os_ and tuple(c) == oc
    for D, base in [(128, 10000.0), (64, 500000.0), (8, 10000.0)]:
        assert np.array_equal(B.poly_rope_turn_increments(D, base), rope.turn_increments(D, base))
    out = np.zeros(4, dtype=np.uint32)
    assert L.poly_rope_turn_increments(7, 10000.0, out.ctypes.data) == B.POLY_EINVAL
    assert L.poly_rope_turn_increments(8, 1.0, out.ctypes.data) == B.POLY_EINVAL
    assert L.poly_rope_programs(None, None) == B.POLY_EINVAL


def test_rope_rejects_bad_arguments(L):
    s = None
    args = lambda **kw: [kw.get("variant", 0), kw.get("q", FAKE), kw.get("k", FAKE + 0x100000),
                         kw.get("qo", FAKE + 0x200000), kw.get("ko", FAKE + 0x300000),
                         kw.get("delta", FAKE + 0x400000), None, None,
                         kw.get("b", 1), kw.get("s", 4), kw.get("hq", 2), kw.get("hkv", 1),
                         kw.get("d", 16), kw.get("pos", 0), s]
    assert L.poly_rope_fwd(*args(variant=3)) == B.POLY_EINVAL
    assert L.poly_rope_fwd(*args(d=12)) == B.POLY_EINVAL               # not a multiple of 8
    assert L.poly_rope_fwd(*args(q=FAKE + 8)) == B.POLY_EINVAL         # not 16-byte aligned
    assert L.poly_rope_fwd(*args(delta=None)) == B.POLY_EINVAL
    assert L.poly_rope_fwd(*args(qo=FAKE + 64)) == B.POLY_EINVAL       # output overlaps input
    assert L.poly_rope_fwd(*args(pos=(1 << 32) - 2)) == B.POLY_EINVAL  # positions past 2^32
    assert L.poly_rope_fwd(*args(variant=2)) == B.POLY_EINVAL          # table variant, no tables
    assert L.poly_rope_bwd(*args(b=-1)) == B.POLY_EINVAL
    assert L.poly_rope_fwd(*args(b=0)) == B.POLY_OK
    assert L.poly_rope_fwd(*args(hq=0, hkv=0)) == B.POLY_OK


def test_packed_control_constants_are_the_nearest_values():
    """The packed MUFU control's constants (csrc/kern_ctrl.cu, PkConst) are the
    FP16 / BF16 values nearest to 1, sqrt(2/pi), 0.044715 sqrt(2/pi),
    3 x 0.044715 sqrt(2/pi) and 16, duplicated in both lanes."""
    import math
    import torch
    src = open(os.path.join(ROOT, "polynomial_activation_gb300", "csrc", "kern_ctrl.cu")).read()
    body = src[src.index("struct PkConst"):src.index("};", src.index("struct PkConst"))]
    k = math.sqrt(2.0 / math.pi)
    want = {"one": 1.0, "k": k, "kc": k * 0.044715, "k3c": 3.0 * k * 0.044715, "sixteen": 16.0}
    for name, value in want.items():
        m = re.search(r"\b%s = DT == kF16 \? 0x([0-9A-F]{8})u : 0x([0-9A-F]{8})u;" % name, body)
        assert m, name
        f16 = int(np.array([value], np.float16).view(np.uint16)[0])
        bf16 = int(torch.tensor([value], dtype=torch.float64).to(torch.bfloat16)
                   .view(torch.int16).item()) & 0xFFFF
        assert int(m.group(1), 16) == f16 * 0x00010001, name
        assert int(m.group(2), 16) == bf16 * 0x00010001, name


def test_fitted_programs_pass_the_clamp_check(L):
    """Whatever the search options (a clamp step the target format cannot
    represent, clamps refined by ulps, a narrow fit-interval range), the
    fitter's programs carry lc equal to their clamp's exact value and
    Lc <= Li + 1, so poly_set_program accepts them."""
    try:
        for dt in (B.POLY_F16, B.POLY_BF16):
            o = B.poly_fit_defaults()
            o.li_min, o.li_max, o.li_step = 2.0, 6.0, 0.5
            o.lc_min, o.lc_step = 1.05, 0.1
            o.lc_refine_ulps = 2
            p = B.poly_fit(B.POLY_SIGMOID, B.POLY_FWD, dt, 3, o)
            assert p.lc <= p.li + 1.0
            assert L.poly_set_program(ctypes.byref(p)) == B.POLY_OK
            d = B.poly_derive_program(p)
            assert L.poly_set_program(ctypes.byref(d)) == B.POLY_OK
    finally:
        B.poly_reset_programs()

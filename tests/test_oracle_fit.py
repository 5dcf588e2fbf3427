"""Pins of the oracle fitter (oracle/fit.py).

Against: the endpoint conditions of eq. 7 (exact at 0, to rounding at Li);
the normal equations of least squares; an independent 40-digit solve of the
same constrained problem (Lagrange multipliers, mpmath); the roots of the
Chebyshev polynomial; the printed Table 2 values and Figure 2 configuration
(tests/golden/); the qualitative claim of Figures 4 and 5; and the golden
programs file being what the oracle produces today.
"""
import json
import os

import numpy as np
import pytest
from numpy.polynomial import chebyshev as cheb

import golden_programs as gp
from oracle import fit, reference as ref, tformat as tf
from oracle.replay import evaluate

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
CASES = [(ref.SIGMOID, ref.FWD, 3, 5.0), (ref.TANH, ref.FWD, 4, 3.0),
         (ref.SILU, ref.FWD, 3, 4.75), (ref.GELU, ref.FWD, 5, 2.25),
         (ref.SIGMOID, ref.BWD, 4, 4.75), (ref.TANH, ref.BWD, 4, 2.25),
         (ref.SILU, ref.BWD, 4, 7.25), (ref.SIGMOID, ref.FWD, 6, 12.0)]


@pytest.mark.parametrize("fn,d,D,li", CASES)
def test_endpoint_constraints_eq7(fn, d, D, li):
    c = fit.fit_coefficients(fn, d, D, li)
    f = ref.residual(fn, d)
    assert c[0] == ref.residual_at_zero(fn, d)                        # P(0) = f(0)
    pl = np.polyval(c[::-1], li)
    assert abs(pl - float(f(li))) <= 1e-12 * max(1.0, abs(float(f(li))))   # P(Li) = f(Li)


@pytest.mark.parametrize("fn,d,D,li", CASES)
def test_least_squares_normal_equations(fn, d, D, li):
    """The residual is orthogonal to every free basis term x^j - x Li^(j-1)."""
    c = fit.fit_coefficients(fn, d, D, li)
    x = fit.chebyshev_nodes(li)
    r = ref.residual(fn, d)(x) - np.polyval(c[::-1], x)
    for j in range(2, D + 1):
        col = x ** j - x * li ** (j - 1)
        assert abs(col @ r) <= 1e-9 * np.linalg.norm(col) * max(np.linalg.norm(r), 1e-12)


def test_chebyshev_nodes_are_roots():
    li = 3.7
    x = fit.chebyshev_nodes(li, 64)
    tn = cheb.chebval(2 * x / li - 1, [0] * 64 + [1])
    assert np.max(np.abs(tn)) < 1e-12
    assert np.all((x > 0) & (x < li))


@pytest.mark.parametrize("fn,d,D,li", [(ref.SIGMOID, ref.FWD, 3, 5.0),
                                       (ref.SIGMOID, ref.BWD, 4, 4.75)])
def test_constrained_ls_vs_mpmath_lagrange(fn, d, D, li):
    """Same problem solved independently: minimise ||V c - f||^2 over the full
    monomial basis subject to P(0) = f(0), P(Li) = f(Li), via the KKT system
    in 40-digit arithmetic."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    x = fit.chebyshev_nodes(li)[::10]          # a subsample: same problem shape
    # the oracle on the same subsample
    f = ref.residual(fn, d)
    f0, fl = ref.residual_at_zero(fn, d), float(f(li))
    base = f0 + x * (fl - f0) / li
    A = np.stack([x ** j - x * li ** (j - 1) for j in range(2, D + 1)], 1)
    a = np.linalg.lstsq(A, f(x) - base, rcond=None)[0]
    c_or = np.zeros(D + 1)
    c_or[0], c_or[1] = f0, (fl - f0) / li - sum(a[j - 2] * li ** (j - 1) for j in range(2, D + 1))
    c_or[2:] = a
    n = D + 1
    V = mp.matrix([[mp.mpf(float(xi)) ** j for j in range(n)] for xi in x])
    y = mp.matrix([mp.mpf(float(v)) for v in f(x)])
    C = mp.matrix([[1] + [0] * D, [mp.mpf(li) ** j for j in range(n)]])
    K = mp.zeros(n + 2, n + 2)
    VtV = V.T * V
    for i in range(n):
        for j in range(n):
            K[i, j] = 2 * VtV[i, j]
        K[i, n], K[i, n + 1] = C[0, i], C[1, i]
        K[n, i], K[n + 1, i] = C[0, i], C[1, i]
    rhs = mp.matrix([2 * v for v in (V.T * y)] + [mp.mpf(f0), mp.mpf(fl)])
    sol = mp.lu_solve(K, rhs)
    for j in range(n):
        assert abs(c_or[j] - float(sol[j])) <= 1e-9 * max(1.0, abs(float(sol[j])))


def _table2_rows():
    rows = []
    with open(os.path.join(GOLDEN, "table2_bf16.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                d, name, D, form, v = line.split()
                rows.append((d, name, int(D), form, float(v) * 1e-3))
    return rows


# How close the accepted program's Table 2 metric must come to the printed
# value.  sigma' D4 and the D3 centred sigmoid land within 1 % of the paper's
# values.  For the other three the accepted program is not the paper's: the
# Sollya column bounds the paper's clamps (test_sollya_column_bounds_the_clamp)
# and shows SiLU's and GELU's below the ones accepted here, which the score of
# §3.2 step 6 with the exact relu tail cannot select
# (test_accepted_clamps_against_the_sollya_bound); tanh keeps the paper's clamp
# but a different fit interval.  Their factors are the measured gaps (1.173,
# 1.465, 2.826) with 0.5 % of margin, so that any change to the fitter or the
# metric that moves them fails.
T2_FACTOR = {("bwd", "sigmoid"): 1.01, ("fwd", "sigmoid"): 1.01, ("fwd", "tanh"): 1.18,
             ("fwd", "silu"): 1.472, ("fwd", "gelu"): 2.84}


@pytest.mark.parametrize("row", _table2_rows())
def test_table2_magnitudes(row):
    d, name, D, form, printed = row
    fn = gp.NAMES[name]
    direction = ref.FWD if d == "fwd" else ref.BWD
    assert ref.form_of(fn, direction) == form
    p = gp.get(fn, direction, "bf16", D)
    m = fit.table2_metric(p)
    k = T2_FACTOR[(d, name)]
    assert printed / k <= m <= printed * k, (name, m, printed)


def _sollya_rows():
    rows = []
    with open(os.path.join(GOLDEN, "table2_sollya_bf16.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                d, name, D, form, v, lc = line.split()
                rows.append((d, name, int(D), form, float(v) * 1e-3, float(lc)))
    return rows


def _monomials(form, D):
    """Powers of t the row's polynomial carries (§3.1: no constant term
    except for the even form)."""
    return list(range(0, D + 1)) if form == "E" else list(range(1, D + 1))


def _fp64_minimax(fn, direction, form, D, lc, m=3000):
    """Smallest max |P(t) - r(t)| over m points of [0, Lc] for P in the
    row's monomial span, r the half-domain residual: a linear program
    (scipy's HiGHS), independent of the oracle's least-squares code."""
    from scipy.optimize import linprog
    t = np.linspace(0.0, lc, m)
    V = np.stack([t ** p for p in _monomials(form, D)], axis=1)
    y = ref.residual(fn, direction)(t)
    k = V.shape[1]
    A = np.vstack([np.hstack([V, -np.ones((m, 1))]), np.hstack([-V, -np.ones((m, 1))])])
    res = linprog(np.r_[np.zeros(k), 1.0], A_ub=A, b_ub=np.r_[y, -y],
                  bounds=[(None, None)] * k + [(0, None)], method="highs")
    assert res.status == 0
    return float(res.x[-1])


@pytest.mark.parametrize("row", _sollya_rows())
def test_sollya_column_bounds_the_clamp(row):
    """The printed Sollya minimax errors (Table 2) bound each row's clamp:
    an fpminimax fit with BF16 coefficients errs at least as much as the
    unconstrained FP64 minimax on the same interval, which grows with Lc.
    The FP64 minimax at the golden clamp stays below the printed value and,
    except for the centred sigmoid (whose D3 minimax plateaus near 5.3e-3
    for Lc in [5.75, 7]), exceeds it 0.25 further out -- so the paper's Lc
    lies below that point.  A wrong residual, form or monomial set moves the
    crossing and fails here."""
    d, name, D, form, printed, lc = row
    fn = gp.NAMES[name]
    direction = ref.FWD if d == "fwd" else ref.BWD
    assert ref.form_of(fn, direction) == form
    assert _fp64_minimax(fn, direction, form, D, lc) <= printed
    assert _fp64_minimax(fn, direction, form, D, lc + 0.25) > printed


def _ls_error(fn, direction, D, li, lc, rounded):
    """Table 2 metric of the eq. 8 fit on [0, Li] clamped at Lc, with FP64 or
    BF16-rounded coefficients."""
    c = fit.fit_coefficients(fn, direction, D, li)
    if rounded:
        return fit.table2_metric(fit.make_program(fn, direction, "bf16", D, li, lc,
                                                  tf.from_f64(c, "bf16")))
    from oracle.replay import evaluate_real
    x = np.linspace(-lc, lc, 20001)
    y = evaluate_real(ref.form_of(fn, direction), c, lc, x)
    return float(np.max(np.abs(y - ref.function(fn, direction)(x))))


@pytest.mark.parametrize("row", _table2_rows())
def test_table2_least_squares_value_is_bracketed(row):
    """At the clamp the Sollya column allows (fit interval = clamp), the
    printed least-squares value lies between this fitter's FP64 error and its
    BF16-rounded error: the eq. 8 fit agrees with the paper's, and the gap to
    the printed value is coefficient rounding (tanh D4, GELU D5, sigma' D4).
    SiLU D3's printed value falls between the FP64 errors of the grid clamps
    4.25 and 4.5 (an off-grid clamp, like Figure 2's 5.28125); the centred
    sigmoid's accepted program matches it to 1 %."""
    d, name, D, form, printed = row
    fn = gp.NAMES[name]
    direction = ref.FWD if d == "fwd" else ref.BWD
    lc = {r[1]: r[5] for r in _sollya_rows() if r[0] == d}[name]
    if (d, name) == ("fwd", "sigmoid"):
        p = gp.get(fn, direction, "bf16", D)
        assert abs(fit.table2_metric(p) / printed - 1) <= 0.01
    elif (d, name) == ("fwd", "silu"):
        assert (_ls_error(fn, direction, D, 4.25, 4.25, False) < printed
                < _ls_error(fn, direction, D, 4.5, 4.5, False))
    else:
        assert (_ls_error(fn, direction, D, lc, lc, False) <= printed
                <= _ls_error(fn, direction, D, lc, lc, True))


def test_accepted_clamps_against_the_sollya_bound():
    """tanh D4 and sigma' D4 are accepted at the largest clamp the Sollya
    column allows.  SiLU D3 and GELU D5 are accepted above it: every clamp
    below the bound leaves an exact-relu tail error just above the clamp
    (x sigma(-x), x (1 - Phi(x)), evaluated at the bound, where they are
    smallest) larger than the accepted program's whole deployed error, so
    the maximum-error score over [0, 12] (§3.2 step 6) with the exact tail
    cannot select the paper's clamp -- the paper's selection weighed that
    tail differently, which its text does not state."""
    bound = {(r[0], r[1]): r[5] + 0.25 for r in _sollya_rows()}
    for d, name, D in (("fwd", "tanh", 4), ("bwd", "sigmoid", 4)):
        fn = gp.NAMES[name]
        p = gp.get(fn, ref.FWD if d == "fwd" else ref.BWD, "bf16", D)
        assert p.lc == bound[(d, name)] - 0.25
    for name, D, tail in (("silu", 3, lambda x: x * ref.sigmoid(-x)),
                          ("gelu", 5, lambda x: x * ref.Phi(-x))):
        p = gp.get(gp.NAMES[name], ref.FWD, "bf16", D)
        b = bound[("fwd", name)]
        assert p.lc >= b
        assert float(tail(np.array([b]))[0]) > p.info["deployed_score"]


def test_figure2_configuration_is_reproduced():
    """The D4 centred sigmoid search lands on the fit interval of the paper's
    selected (Li, Lc) = (5.0, 5.28125) (Fig. 2b) and on a clamp one BF16 ulp
    below it (the printed Lc is off the 0.25 grid), with exactly the same
    maximum error over every finite BF16 input; allowing the clamp to move by
    one ulp finds no better program (the three clamps tie in deployed order,
    and the Table 2 tie-break takes one of them)."""
    with open(os.path.join(GOLDEN, "figure2_selected.txt")) as f:
        name, d, D, li, lc = [l for l in f if not l.startswith("#")][0].split()
    li, lc, D = float(li), float(lc), int(D)
    assert int(tf.from_f64(lc, "bf16")) == int(tf.from_f64(5.25, "bf16")) + 1
    cb = tf.from_f64(fit.fit_coefficients(ref.SIGMOID, ref.FWD, D, li), "bf16")
    p = fit.make_program(ref.SIGMOID, ref.FWD, "bf16", D, li, lc, cb)
    err_fig2 = fit.exhaustive_error(p)[0]
    ours = fit.search(ref.SIGMOID, ref.FWD, "bf16", D)
    assert ours.li == li and int(ours.lc_bits) == int(tf.from_f64(lc, "bf16")) - 1
    assert err_fig2 == ours.info["stated_max_abs_err"] < 6e-3
    refined = fit.search(ref.SIGMOID, ref.FWD, "bf16", D, lc_refine_ulps=1)
    assert refined.li == li and abs(int(refined.lc_bits) - int(ours.lc_bits)) <= 1
    assert refined.info["deployed_score"] == ours.info["deployed_score"]


def test_top_k_restricts_the_deployed_replay():
    """Keeping only the 8 best split-order candidates for the deployed replay
    can only do as well as replaying them all (the D3 centred sigmoid and the
    D5 GELU do strictly worse with 8)."""
    for fn, D in ((ref.SIGMOID, 3), (ref.GELU, 5)):
        every = gp.get(fn, ref.FWD, "bf16", D)        # the default search's program
        top8 = fit.search(fn, ref.FWD, "bf16", D, top_k=8)
        assert every.info["deployed_score"] < top8.info["deployed_score"]
        assert top8.info["rank"] < 8 <= every.info["rank"]


def _stated_bound(args):
    fn, d, D = args
    return fit.search(fn, d, "bf16", D).info["stated_max_abs_err"]


@pytest.mark.slow
def test_higher_degree_can_be_worse_figs_4_5():
    """In each of the six BF16 sweeps (sigmoid, tanh, SiLU forward; their
    derivatives backward), at least one higher-degree program has a larger
    maximum error than a lower-degree one after replay (§5.1, Figs. 4-5)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    sweeps = [(fn, d) for fn in (ref.SIGMOID, ref.TANH, ref.SILU) for d in (ref.FWD, ref.BWD)]
    jobs = [(fn, d, D) for fn, d in sweeps for D in (3, 4, 5, 6)]
    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    with cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn")) as ex:
        bounds = list(ex.map(_stated_bound, jobs))
    for i, (fn, d) in enumerate(sweeps):
        errs = bounds[4 * i:4 * i + 4]
        assert any(errs[j] > errs[i2] for i2 in range(4) for j in range(i2 + 1, 4)), (fn, d, errs)


@pytest.mark.slow
@pytest.mark.parametrize("k", ["sigmoid.fwd.bf16.D3", "silu.bwd.f16.D4", "gelu.fwd.bf16.D5"])
def test_golden_programs_are_current(k):
    """tests/golden/programs.json is exactly what the oracle fitter produces."""
    with open(gp.PATH) as f:
        g = json.load(f)[k]
    p = fit.search(g["fn"], g["direction"], g["fmt"], g["degree"])
    assert (p.li, p.lc, list(p.coef), p.lc_bits) == (g["li"], g["lc"], g["coef"], g["lc_bits"])
    assert p.info["stated_max_abs_err"] == g["stated_max_abs_err"]


def test_search_gates_hold_on_golden_programs():
    """Every accepted program respects the gates it was selected under."""
    for k, p in gp.load().items():
        x = fit.score_grid(p.fmt)
        y = tf.decode(evaluate(p.form, p.coef, p.lc_bits, x, p.fmt), p.fmt)
        assert np.all(np.isfinite(y))
        rng = ref.value_range(p.fn, p.direction)
        if rng:
            assert y.min() >= rng[0] and y.max() <= rng[1], k
        assert p.lc <= p.li + 1


def _gate(fn, d, fmt, coef, lc):
    """The search's gates for one candidate (split-order replay on the score
    grid, as the search applies them)."""
    x = fit.score_grid(fmt)
    cb = np.asarray(tf.from_f64(np.asarray(coef, dtype=np.float64), fmt))
    lc_bits = tf.from_f64(lc, fmt)
    y = evaluate(ref.form_of(fn, d), tuple(int(b) for b in cb), lc_bits, x, fmt, fused=False)
    return bool(fit._gates(fn, d, y, fmt, cb, lc, x))


def test_gates_reject_each_violation():
    """§3.2 rejects shape or boundary violations: each gate alone turns away
    a candidate built to break only it, and the accepted program passes."""
    S, T, F = ref.SIGMOID, ref.TANH, ref.FWD
    g = gp.load()["sigmoid.fwd.bf16.D3"]
    assert _gate(S, F, "bf16", tf.decode(np.array(g.coef, np.uint16), "bf16"), g.lc)
    # range: y = 1/2 + t/2 reaches 1.25 at Lc = 1.5 (monotone, finite, P(0) exact)
    assert not _gate(S, F, "bf16", [0.0, 0.5, 0.0, 0.0], 1.5)
    assert _gate(S, F, "bf16", [0.0, 0.25, 0.0, 0.0], 1.5)      # 1/2 + t/4 <= 0.875: passes
    # shape: 1/2 + 0.25 t - 0.2 t^2 rises then falls, inside [0, 1] up to Lc = 1.5
    assert not _gate(S, F, "bf16", [0.0, 0.25, -0.2, 0.0], 1.5)
    # boundary: sigma' with P(0) = 0.2 instead of 1/4 (inside [0, 1/4], decreasing)
    assert not _gate(S, ref.BWD, "bf16", [0.2, 0.0, -0.01, 0.0, 0.0], 4.0)
    assert _gate(S, ref.BWD, "bf16", [0.25, 0.0, -0.01, 0.0, 0.0], 4.0)
    # finite: an FP16 SiLU' (no exact range, not monotone, so no other gate
    # applies) whose Horner chain overflows before the clamp
    assert not _gate(ref.SILU, ref.BWD, "f16", [0.0, 0.0, 0.0, 60000.0], 4.0)
    assert _gate(ref.SILU, ref.BWD, "f16", [0.0, 0.0, 0.0, 0.01], 4.0)


@pytest.mark.parametrize("fn,D,li", [(ref.SIGMOID, 3, 1.0), (ref.SILU, 3, 2.0)])
def test_clamp_bound_is_enforced(fn, D, li):
    """Lc <= Li + 1 (§3.2): with a single short fit interval the best clamp
    would lie beyond the bound, so the search must stop exactly at it."""
    p = fit.search(fn, ref.FWD, "bf16", D, li_grid=[li])
    assert p.lc == li + 1.0

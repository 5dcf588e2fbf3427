"""CPU replay oracle for the packed-polynomial activation programs.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product (``polynomial_activation_gb300``) never imports it, and
it never imports the product: the two share no code, no tables and no
constant generators.  Inputs reach both sides from ``workloads.py`` only.

What the oracle computes (all citations are to "Fast Polynomial
Transcendentals for LLMs", arXiv 2610.00049):

* ``tformat``   -- IEEE binary16 (FP16) and bfloat16 (BF16) arithmetic written
  out from the format definitions: every operation rounds its exact result
  once, to nearest with ties to even, with subnormals kept (§3.2, the
  "packed-FMA-style replay that rounds once per multiply-add", Fig. 2c).
* ``reference`` -- FP64 reference functions and the reduced residuals of
  §3.1 (eq. 2-6) and §3.3 (eq. 9-11).
* ``replay``    -- the programs replayed in deployed order (one rounding per
  packed FMA), in the fitter's split order (one rounding per multiply and per
  add, §3.2 step 4) and in real arithmetic (the Table 2 metric).
* ``fit``       -- the endpoint-constrained least-squares fitter and the
  (Li, Lc) search of §3.2 (eq. 7-8, steps 1-7).
* ``exp2``      -- 2^x with the FP32 range reduction, packed-FP16 fractional
  cores and exponent-bit reconstruction of Appendix B.1 (Table 8).
* ``rope``      -- Q0.32 turn increments, the folded Q15 phase, the paired
  FP16 sine / cosine programs and the rotation of Appendix B.2.

Every function is pinned in ``tests/test_oracle_*.py`` against something
other than itself: exact rational arithmetic and a second exact model in
scaled integers (ten million random triples per format), mpmath, printed
values of the paper's Tables 2 and 8 and Figure 2, closed forms and exact
symmetry identities.
Parity unpinned: the exact coefficients chosen by ``fit.search`` (the paper
prints none for these programs; only magnitudes of their errors).
"""

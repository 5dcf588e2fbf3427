"""Write tests/golden/programs.json: the oracle fitter's accepted programs.

Calls only ``oracle/``.  The GPU parity tests replay these programs on the
CPU; the product's own fitter must reproduce them bit for bit
(tests/test_capi_host.py).  Re-run after any change to the oracle fitter:

    python tests/golden/make_programs.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import fit, reference as ref  # noqa: E402

# (fn, direction, degree): the paper's programs (Table 2, Table 3) plus the
# centred SiLU derivative used by the SwiGLU backward and a GELU derivative.
PROGRAMS = [
    (ref.SIGMOID, ref.FWD, 3), (ref.TANH, ref.FWD, 4), (ref.SILU, ref.FWD, 3),
    (ref.GELU, ref.FWD, 5), (ref.SIGMOID, ref.BWD, 4), (ref.TANH, ref.BWD, 4),
    (ref.SILU, ref.BWD, 4), (ref.GELU, ref.BWD, 4),
]


def key(fn, direction, fmt, degree):
    return f"{ref.FN_NAMES[fn]}.{'bwd' if direction else 'fwd'}.{fmt}.D{degree}"


def main():
    out = {}
    for fmt in ("bf16", "f16"):
        for fn, d, D in PROGRAMS:
            p = fit.search(fn, d, fmt, D)
            out[key(fn, d, fmt, D)] = {
                "fn": fn, "direction": d, "fmt": fmt, "degree": D,
                "li": p.li, "lc": p.lc, "lc_bits": p.lc_bits,
                "coef": list(p.coef), **p.info,
            }
            print(key(fn, d, fmt, D), f"Li={p.li} Lc={p.lc}",
                  f"bound={p.info['stated_max_abs_err']:.4e}", flush=True)
    with open(os.path.join(HERE, "programs.json"), "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main()

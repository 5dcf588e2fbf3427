"""Load tests/golden/programs.json (written by tests/golden/make_programs.py,
which calls only the oracle) as oracle ``Program`` objects."""
import json
import os

from oracle import reference as ref
from oracle.replay import Program

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "programs.json")
NAMES = {"sigmoid": ref.SIGMOID, "tanh": ref.TANH, "silu": ref.SILU, "gelu": ref.GELU}


def load():
    with open(PATH) as f:
        raw = json.load(f)
    out = {}
    for k, v in raw.items():
        info = {kk: v[kk] for kk in ("search_score", "deployed_score", "rank",
                                     "stated_max_abs_err", "argmax_bits", "table2")}
        out[k] = Program(fn=v["fn"], direction=v["direction"], fmt=v["fmt"],
                         degree=v["degree"], li=v["li"], lc=v["lc"],
                         coef=tuple(v["coef"]), lc_bits=v["lc_bits"], info=info)
    return out


def key(fn, direction, fmt, degree):
    return f"{ref.FN_NAMES[fn]}.{'bwd' if direction else 'fwd'}.{fmt}.D{degree}"


def get(fn, direction, fmt, degree=None):
    progs = load()
    if degree is None:
        degree = {(ref.SIGMOID, 0): 3, (ref.TANH, 0): 4, (ref.SILU, 0): 3,
                  (ref.GELU, 0): 5}.get((fn, direction), 4)
    return progs[key(fn, direction, fmt, degree)]

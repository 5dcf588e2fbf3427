"""Accepted programs on disk: save, verify, reload, and resumable fitting.

A program (``poly_program``) is small and fully determines the kernels'
arithmetic: function, direction, format, form, degree, the coefficient bit
patterns and the clamp.  This module writes programs to a JSON file with a
format version and, per program, a SHA-256 over exactly those fields, so a
file edited by hand or damaged in transit is refused instead of silently
changing the arithmetic.  The search metadata (Li, Lc, scores, stated bound)
travels with each program.  Host only: nothing here touches the GPU.

``fit_rows`` runs the fitter over (fn, dir, dtype, degree) rows and writes the
file after every row, so an interrupted run resumes with the rows that are
still missing.
"""
from __future__ import annotations

import hashlib
import json
import os

from . import binding as B

FORMAT = "polyact-programs"
FILE_VERSION = 1
_DTYPES = {B.POLY_F16: "f16", B.POLY_BF16: "bf16"}
_DTYPE_IDS = {v: k for k, v in _DTYPES.items()}
_META = ("li", "lc", "search_score", "deployed_score", "stated_max_abs_err", "table2", "rank")


def program_hash(p: B.PolyProgram) -> str:
    """SHA-256 (hex) of the fields that define a program's arithmetic."""
    key = (f"{p.fn}:{p.dir}:{p.dtype}:{p.form}:{p.degree}:"
           + ",".join(f"{c:04x}" for c in p.coefficients()) + f":{p.lc_bits:04x}:{p.version}")
    return hashlib.sha256(key.encode()).hexdigest()


def to_record(p: B.PolyProgram) -> dict:
    rec = {"fn": B.FN_NAMES[p.fn], "dir": "bwd" if p.dir == B.POLY_BWD else "fwd",
           "dtype": _DTYPES[p.dtype], "form": p.form, "degree": p.degree,
           "coef": [f"0x{c:04x}" for c in p.coefficients()], "lc_bits": f"0x{p.lc_bits:04x}",
           "program_version": p.version}
    rec.update({k: getattr(p, k) for k in _META})
    rec["sha256"] = program_hash(p)
    return rec


def from_record(rec: dict) -> B.PolyProgram:
    """Rebuild a program from its record; ValueError if the record is
    incomplete or its hash does not match its fields."""
    try:
        p = B.PolyProgram()
        p.fn = B.FN[rec["fn"]]
        p.dir = B.POLY_BWD if rec["dir"] == "bwd" else B.POLY_FWD
        p.dtype = _DTYPE_IDS[rec["dtype"]]
        p.form = int(rec["form"])
        p.degree = int(rec["degree"])
        coef = [int(c, 16) for c in rec["coef"]]
        if len(coef) != p.degree + 1 or len(coef) > B.POLY_MAX_DEGREE + 1:
            raise ValueError("coefficient count does not match the degree")
        for j, c in enumerate(coef):
            p.coef[j] = c
        p.lc_bits = int(rec["lc_bits"], 16)
        p.version = int(rec["program_version"])
        for k in _META:
            setattr(p, k, rec[k])
    except (KeyError, TypeError) as e:
        raise ValueError(f"incomplete program record: {e}") from None
    if program_hash(p) != rec.get("sha256"):
        raise ValueError(f"program {rec.get('fn')}.{rec.get('dir')}.{rec.get('dtype')}: "
                         "sha256 does not match its fields")
    return p


def save(programs, path: str) -> None:
    """Write programs to path (atomically: a temporary file, then a rename)."""
    doc = {"format": FORMAT, "version": FILE_VERSION,
           "programs": [to_record(p) for p in programs]}
    tmp = path + ".tmp"
    with open(tmp, "w") as f:
        json.dump(doc, f, indent=1)
    os.replace(tmp, path)


def load(path: str):
    """Programs stored in path, each verified against its hash."""
    with open(path) as f:
        doc = json.load(f)
    if doc.get("format") != FORMAT or doc.get("version") != FILE_VERSION:
        raise ValueError(f"{path}: not a {FORMAT} file of version {FILE_VERSION}")
    return [from_record(r) for r in doc["programs"]]


def install(path: str):
    """Load programs and install each in the library's registry (the library
    validates every descriptor again)."""
    progs = load(path)
    for p in progs:
        B.poly_set_program(p)
    return progs


def save_installed(path: str) -> None:
    """Save the program the library uses for every (fn, dir, dtype)."""
    progs = [B.poly_get_program(fn, d, dt) for fn in sorted(B.FN_NAMES)
             for d in (B.POLY_FWD, B.POLY_BWD) for dt in (B.POLY_F16, B.POLY_BF16)]
    save(progs, path)


def _row(p):
    return (p.fn, p.dir, p.dtype, p.degree)


def fit_rows(path: str, rows, opts=None):
    """Fit every (fn, dir, dtype, degree) row not yet in path, writing the
    file after each new row; returns all programs of the file."""
    progs = load(path) if os.path.exists(path) else []
    have = {_row(p) for p in progs}
    for row in rows:
        if tuple(row) in have:
            continue
        fn, d, dt, degree = row
        progs.append(B.poly_fit(fn, d, dt, degree, opts))
        have.add(tuple(row))
        save(progs, path)
    return progs


def _parse_row(text: str):
    """'sigmoid:fwd:bf16:3' -> (fn, dir, dtype, degree)."""
    fn, d, dt, deg = text.split(":")
    return (B.FN[fn], B.POLY_BWD if d == "bwd" else B.POLY_FWD, _DTYPE_IDS[dt], int(deg))


def main(argv=None) -> int:
    """Command line: fit rows into a file (resumable), show or verify one."""
    import argparse
    ap = argparse.ArgumentParser(prog="python -m polynomial_activation_gb300.programs")
    sub = ap.add_subparsers(dest="cmd", required=True)
    f = sub.add_parser("fit", help="fit the missing rows into FILE (rows: fn:dir:dtype:degree)")
    f.add_argument("file")
    f.add_argument("rows", nargs="+")
    for name in ("show", "verify"):
        sub.add_parser(name).add_argument("file")
    a = ap.parse_args(argv)
    if a.cmd == "fit":
        progs = fit_rows(a.file, [_parse_row(r) for r in a.rows])
        print(f"{a.file}: {len(progs)} programs")
        return 0
    progs = load(a.file)                               # verifies every hash
    if a.cmd == "show":
        for p in progs:
            r = to_record(p)
            print(f"{r['fn']}.{r['dir']}.{r['dtype']}.D{r['degree']}  Li={r['li']:g} "
                  f"Lc={r['lc']:g}  bound={r['stated_max_abs_err']:.4e}  {r['sha256'][:12]}")
    else:
        print(f"{a.file}: {len(progs)} programs, every hash verified")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())

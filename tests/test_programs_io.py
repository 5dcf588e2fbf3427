"""Accepted programs on disk (polynomial_activation_gb300/programs.py): the
JSON round trip is exact, a changed coefficient or clamp or a wrong file
version is refused, installed programs come back from the library's
registry, and a fitter run resumes with the rows it has not written yet.
Host only."""
import json

import pytest

from polynomial_activation_gb300 import binding as B
from polynomial_activation_gb300 import programs as P


@pytest.fixture(autouse=True)
def _reset():
    B.poly_reset_programs()
    yield
    B.poly_reset_programs()


def test_round_trip_is_exact(tmp_path):
    progs = [B.poly_get_program(B.POLY_SIGMOID, B.POLY_FWD, B.POLY_BF16),
             B.poly_get_program(B.POLY_TANH, B.POLY_BWD, B.POLY_F16),
             B.poly_fit(B.POLY_GELU, B.POLY_FWD, B.POLY_BF16, 6)]
    path = str(tmp_path / "p.json")
    P.save(progs, path)
    back = P.load(path)
    assert [bytes(a) for a in back] == [bytes(b) for b in progs]


@pytest.mark.parametrize("field,value", [("coef", 1), ("lc_bits", None), ("degree", None)])
def test_tampered_record_is_refused(tmp_path, field, value):
    path = str(tmp_path / "p.json")
    P.save([B.poly_get_program(B.POLY_SILU, B.POLY_FWD, B.POLY_BF16)], path)
    doc = json.load(open(path))
    rec = doc["programs"][0]
    if field == "coef":
        rec["coef"][value] = f"0x{int(rec['coef'][value], 16) ^ 1:04x}"   # one ulp
    elif field == "lc_bits":
        rec["lc_bits"] = f"0x{int(rec['lc_bits'], 16) + 1:04x}"
    else:
        rec["degree"] = rec["degree"] + 1
    json.dump(doc, open(path, "w"))
    with pytest.raises(ValueError):
        P.load(path)


def test_wrong_format_or_version_is_refused(tmp_path):
    path = str(tmp_path / "p.json")
    P.save([], path)
    doc = json.load(open(path))
    doc["version"] = 99
    json.dump(doc, open(path, "w"))
    with pytest.raises(ValueError):
        P.load(path)


def test_install_and_save_installed(tmp_path):
    d6 = B.poly_fit(B.POLY_TANH, B.POLY_FWD, B.POLY_BF16, 6)
    path = str(tmp_path / "one.json")
    P.save([d6], path)
    P.install(path)
    assert bytes(B.poly_get_program(B.POLY_TANH, B.POLY_FWD, B.POLY_BF16)) == bytes(d6)
    every = str(tmp_path / "all.json")
    P.save_installed(every)
    progs = P.load(every)
    assert len(progs) == 16
    assert sum(bytes(p) == bytes(d6) for p in progs) == 1


def test_fit_rows_resumes(tmp_path, monkeypatch):
    path = str(tmp_path / "fit.json")
    rows = [(B.POLY_SIGMOID, B.POLY_FWD, B.POLY_BF16, 3), (B.POLY_TANH, B.POLY_FWD, B.POLY_F16, 4),
            (B.POLY_SILU, B.POLY_BWD, B.POLY_BF16, 4)]
    calls = []
    real = B.poly_fit

    def counting(*a, **k):
        calls.append(a[:4])
        return real(*a, **k)

    monkeypatch.setattr(B, "poly_fit", counting)
    P.fit_rows(path, rows[:2])
    assert len(calls) == 2 and len(P.load(path)) == 2
    progs = P.fit_rows(path, rows)                 # only the missing row is fitted
    assert calls[2:] == [rows[2]]
    assert [(p.fn, p.dir, p.dtype, p.degree) for p in progs] == rows


def test_command_line_fit_show_verify(tmp_path, capsys):
    path = str(tmp_path / "cli.json")
    assert P.main(["fit", path, "tanh:fwd:bf16:4", "sigmoid:bwd:f16:4"]) == 0
    assert P.main(["fit", path, "tanh:fwd:bf16:4", "gelu:fwd:bf16:5"]) == 0   # resumes
    assert len(P.load(path)) == 3
    assert P.main(["show", path]) == 0
    out = capsys.readouterr().out
    assert "tanh.fwd.bf16.D4" in out and "gelu.fwd.bf16.D5" in out
    assert P.main(["verify", path]) == 0
    doc = json.load(open(path))
    doc["programs"][0]["coef"][1] = "0x0000"
    json.dump(doc, open(path, "w"))
    with pytest.raises(ValueError):
        P.main(["verify", path])

"""The C ABI from C: a C99 program that includes include/polyact.h compiles
with -pedantic -Werror, links against libpolyact.so and makes host-side calls
(fit, status strings, version, an empty launch) with the expected results.
No GPU work."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "polynomial_activation_gb300")

PROGRAM = r"""
#include <stdio.h>
#include "polyact.h"

int main(void) {
  poly_fit_opts o;
  poly_program p;
  int st;
  if (poly_fit_defaults(&o) != POLY_OK) return 2;
  st = poly_fit(POLY_SIGMOID, POLY_BWD, POLY_BF16, 4, &o, &p);
  if (st != POLY_OK) return 3;
  printf("fit %s %.2f %.2f %d %d\n", poly_status_str(st), p.li, p.lc, p.degree, p.form);
  printf("abi %d\n", poly_abi_version());
  printf("empty %d\n", poly_act_fwd(POLY_SILU, POLY_BF16, (const void *)0, (void *)0, 0,
                                    (poly_stream_t)0));
  printf("bad %d\n", poly_act_fwd(9, POLY_BF16, (const void *)0, (void *)0, 8, (poly_stream_t)0));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_c_program_uses_the_abi(tmp_path):
    src = tmp_path / "t.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "t"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(ROOT, "include"), str(src), "-L", PKG, "-lpolyact",
           f"-Wl,-rpath,{PKG}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    lines = dict(l.split(" ", 1) for l in out.stdout.strip().splitlines())
    assert lines["fit"].split()[0] == "POLY_OK"
    li, lc, degree, form = lines["fit"].split()[1:]
    assert (float(li), float(lc), int(degree), int(form)) == (4.75, 4.75, 4, 2)   # even form
    assert int(lines["abi"]) == 4
    assert int(lines["empty"]) == 0 and int(lines["bad"]) == -1

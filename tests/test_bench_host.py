"""Host logic of bench.py that needs no GPU: the clock sampler's parsing of
nvidia-smi output, run against a stand-in nvidia-smi on PATH."""
import os
import stat
import sys
import time

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

FAKE = """#!/bin/sh
# stand-in for nvidia-smi --query-gpu ... -lms N: one line per 20 ms
i=0
while [ $i -lt 500 ]; do
  if [ $i -eq 3 ]; then
    echo "1900, 2070, 900.0, Not Active, Not Active, Not Active, Active, 3996"
  else
    echo "2070, 2070, 1000.0, Not Active, Not Active, Not Active, Not Active, 3996"
  fi
  i=$((i + 1))
  sleep 0.02
done
"""


def _fake_smi(tmp_path, monkeypatch):
    exe = tmp_path / "nvidia-smi"
    exe.write_text(FAKE)
    exe.chmod(exe.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")


def test_clock_sampler_parses_samples_and_reasons(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch)
    c = bench.ClockSampler(0)
    c.start()
    assert len(c.lines) >= 1                # start() waited for the first sample
    time.sleep(0.3)
    r = c.stop()
    assert r["samples"] >= 10
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["mem_mhz"] == 3996.0
    assert r["reasons"] == ["sw_power_cap"]   # the fourth line, inside the window
    assert 290 <= r["window_ms"] < 1000


def test_clock_sampler_brackets_a_short_region(tmp_path, monkeypatch):
    """A timed region shorter than the sampling period still gets the last
    sample before it and the first one after it."""
    _fake_smi(tmp_path, monkeypatch)
    c = bench.ClockSampler(0)
    c.start()
    time.sleep(0.1)                          # past the throttled fourth line
    c.t0 = time.monotonic()                  # the region starts now ...
    r = c.stop()                             # ... and ends at once
    assert r["samples"] >= 2 and r["window_ms"] < 20
    assert r["reasons"] == []


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    c = bench.ClockSampler(0)
    c.start()
    assert c.stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}


def test_kernel_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    """Recorded DRAM counters stay valid across comment edits and become
    invalid when the code changes."""
    csrc = tmp_path / "polynomial_activation_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = csrc / "k.cu"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ["k.cu"])
    src.write_text("// a kernel\nint f(int x) { return x + 1; }  /* one */\n")
    h0 = bench.kernel_source_hash()
    src.write_text("// the kernel, reworded\n\nint f(int x) {\n  return x + 1;  // same code\n}\n")
    assert bench.kernel_source_hash() == h0
    src.write_text("int f(int x) { return x + 2; }\n")
    assert bench.kernel_source_hash() != h0


def test_oracle_pool_covers_the_sample():
    """The CPU baseline's worker pool (spawned processes) replays every
    element of the sample once, in one contiguous piece per worker."""
    import bench
    import workloads
    x, dy = workloads.isolated_hbm("f16", n=10_007)
    pool = bench.OraclePool(3)
    try:
        wall, per, sizes = pool.run("six", x, dy)
        assert sum(sizes) == x.size and len(per) == len(sizes) == 3
        assert wall > 0 and all(t > 0 for t in per)
        g, u, d = (np.zeros((7, 24), np.uint16) for _ in range(3))
        wall, per, sizes = pool.run("swiglu", g, u, d)
        assert sum(sizes) == 7 and len(per) == 3
    finally:
        pool.close()

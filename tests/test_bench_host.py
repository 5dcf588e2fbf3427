"""Host logic of bench.py that needs no GPU: the clock sampler's parsing of
nvidia-smi output, run against a stand-in nvidia-smi on PATH."""
import os
import stat
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

FAKE = """#!/bin/sh
# stand-in for nvidia-smi --query-gpu ... -lms 200: one line per 20 ms
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


def test_clock_sampler_parses_samples_and_reasons(tmp_path, monkeypatch):
    exe = tmp_path / "nvidia-smi"
    exe.write_text(FAKE)
    exe.chmod(exe.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    c = bench.ClockSampler(0)
    c.start()
    assert c.skip >= 1                      # start() waited for the first sample
    time.sleep(0.3)
    r = c.stop()
    assert r["samples"] >= 3
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["mem_mhz"] == 3996.0
    assert r["reasons"] == (["sw_power_cap"] if c.skip <= 3 else [])


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    c = bench.ClockSampler(0)
    c.start()
    assert c.stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}

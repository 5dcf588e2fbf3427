import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_sessionstart(session):
    """Build libpolyact.so with nvcc when it is missing or older than any of
    its sources, so that the suite always tests the current kernels."""
    from polynomial_activation_gb300 import build as bld
    srcs = [os.path.join(bld.CSRC, f) for f in os.listdir(bld.CSRC)]
    srcs.append(os.path.join(ROOT, "include", "polyact.h"))
    if os.path.exists(bld.LIB):
        newest = max(os.path.getmtime(f) for f in srcs)
        if os.path.getmtime(bld.LIB) >= newest:
            return
    bld.build(verbose=True)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")

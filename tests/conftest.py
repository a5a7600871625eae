"""Shared test setup.

Markers: ``gpu`` -- needs a CUDA device (parity tests through the C-ABI).
Everything else runs on a CPU-only machine: the oracle's pins, host logic,
and the C-ABI library's load/export check.
"""
import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The count of combine outputs beyond one bf16 ulp of the fp64
    reference in each full comparison (each one within the fp32 summation
    allowance n * 2^-24 * sum|terms|, else its test failed)."""
    gu = sys.modules.get("gpu_util")
    recs = getattr(gu, "ULP_RECORDS", None) if gu else None
    if not recs:
        return
    terminalreporter.section("combine outputs beyond 1 bf16 ulp of the fp64 reference")
    for name, st in recs:
        d = st.as_dict()
        terminalreporter.write_line(
            f"{name:>24}: {d['beyond_1ulp']} of {d['outputs']} outputs "
            f"({d['beyond_1ulp'] / max(d['outputs'], 1):.2e}); largest share of the summation allowance "
            f"used {d['max_allowance_used']:.3f}")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def dyadic(pair):
    """[numerator, log2 denominator] -> float (exact)."""
    n, d = pair
    return float(n) / float(2 ** d)


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.build()
    return o


@pytest.fixture
def rng():
    return np.random.default_rng(20260)

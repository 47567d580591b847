import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def golden_path(name):
    return os.path.join(ROOT, "tests", "golden", name)


def read_golden_kv(name):
    out = {}
    with open(golden_path(name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            k, *v = line.split()
            out[k] = v
    return out


@pytest.fixture(scope="session")
def tqlib():
    """The built library (compiled here if missing or stale)."""
    import rotated_bit_kv_gb300 as tq
    tq.build()
    tq.lib()
    return tq


def pytest_terminal_summary(terminalreporter):
    """Write-side statistics the GPU parity tests collected (if they ran)."""
    mod = sys.modules.get("test_gpu_parity") or sys.modules.get("tests.test_gpu_parity")
    rows = getattr(mod, "STATS", None) if mod else None
    if not rows:
        return
    terminalreporter.write_line("write side vs oracle: workload, B, T, mismatch frac, near-boundary frac "
                                "(normalised), near-boundary frac (scaled)")
    for r in rows:
        terminalreporter.write_line("  %-12s %3d %6d  %.2e  %.2e  %.2e" % r)

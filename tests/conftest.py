"""Shared test configuration.

Markers: ``gpu`` tests need a GB300 and the CUDA library; everything else
runs on a CPU-only machine (oracle pins, host-side validation, symbol
exports, multi-process host logic).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_terminal_summary(terminalreporter):
    """The worst error/bound ratio of every GEMM parity case that ran, and the
    largest overall (written as JSON to $JETFP8_MARGINS_OUT when set)."""
    mod = sys.modules.get("gpu_util")
    margins = getattr(mod, "GEMM_MARGINS", None) if mod else None
    if not margins:
        return
    terminalreporter.write_sep("-", "GEMM parity: worst |gpu - oracle| / bound per case")
    for what, worst, n in margins:
        terminalreporter.write_line(f"{worst:8.4f}  {what}  ({n} elements)")
    top = max(margins, key=lambda m: m[1])
    terminalreporter.write_line(f"largest: {top[1]:.4f} ({top[0]})")
    out = os.environ.get("JETFP8_MARGINS_OUT")
    if out:
        import json
        with open(out, "w") as f:
            json.dump([{"case": w, "worst_ratio": r, "elements": n} for w, r, n in margins], f, indent=1)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running check")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def read_golden(name):
    """Parse a whitespace-separated golden file, skipping '#' comments."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows

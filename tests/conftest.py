import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled libqwm.so")
    config.addinivalue_line("markers", "slow: long CPU-only test")


def golden(name):
    """Parse a tests/golden/*.txt fixture: list of dicts, one per non-comment line."""
    rows = []
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            row = {}
            for tok in line.split():
                k, v = tok.split("=", 1)
                row[k] = v
            rows.append(row)
    return rows

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def golden(name):
    """Parse a ``key = value`` fixture under tests/golden (``case`` keys repeat)."""
    out = {"case": []}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line or "=" not in line:
                continue
            k, v = [s.strip() for s in line.split("=", 1)]
            if k == "case":
                out["case"].append(v)
            else:
                out[k] = v
    return out

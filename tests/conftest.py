import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libckv")


def load_golden(name):
    """key -> float from a tests/golden text fixture (comments after '#')."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split()
            out[k] = float(v)
    return out

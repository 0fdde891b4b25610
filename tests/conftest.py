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


def read_golden_kv(name: str) -> dict:
    """key = value lines of a golden fixture; '#' starts a comment."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            out[key] = val.split()
    return out


def read_golden_rows(name: str) -> list[list[str]]:
    """Whitespace-separated rows of a golden fixture; '#' starts a comment."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def ints(vals) -> np.ndarray:
    return np.array([int(v) for v in vals], np.int64)


def floats(vals) -> np.ndarray:
    return np.array([float(v) for v in vals], np.float64)

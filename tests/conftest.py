import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload")


def load_golden(name):
    """Parse a tests/golden fixture: header keys, then 'name rows cols' blocks of numbers."""
    import numpy as np
    path = os.path.join(ROOT, "tests", "golden", name)
    lines = [l.split("#", 1)[0].strip() for l in open(path, encoding="utf-8")]
    lines = [l for l in lines if l]
    out, i = {}, 0
    while i < len(lines):
        parts = lines[i].split()
        if len(parts) == 2:
            out[parts[0]] = parts[1]
            i += 1
            continue
        name_, r, c = parts[0], int(parts[1]), int(parts[2])
        vals = [float(v) for l in lines[i + 1:i + 1 + r] for v in l.split()]
        out[name_] = np.array(vals, dtype=np.float64).reshape(r, c)
        i += 1 + r
    return out

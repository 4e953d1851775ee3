import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload cases")


def read_golden(name):
    """Parse a golden fixture: '#' comments, records separated by blank lines,
    each line 'key: value'."""
    recs, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line.startswith("#"):
                continue
            if not line:
                if cur:
                    recs.append(cur)
                    cur = {}
                continue
            k, v = line.split(":", 1)
            cur[k.strip()] = v.strip()
    if cur:
        recs.append(cur)
    return recs

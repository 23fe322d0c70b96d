import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libep.so")


def load_golden(name):
    """Parse a whitespace fixture under tests/golden: 'key v v v' lines;
    repeated keys accumulate into a list of rows."""
    path = os.path.join(ROOT, "tests", "golden", name)
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            vals = [int(v) for v in vals]
            out.setdefault(key, []).append(vals)
    return {k: (v[0] if len(v) == 1 else v) for k, v in out.items()}


@pytest.fixture
def golden():
    return load_golden

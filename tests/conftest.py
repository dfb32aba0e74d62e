import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden(name):
    """Parse tests/golden/<name>: '#' lines are comments (the citation);
    every other line is 'key = v1 v2 ...' (numbers)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split("=", 1)
            vals = [float(v) if any(c in v for c in ".e") else int(v) for v in val.split()]
            out[key.strip()] = vals
    return out


@pytest.fixture(scope="session", autouse=True)
def _build_oracle():
    import oracle

    oracle.build()

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture: 'key: a b; c d' -> 2-D int lists."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            out[key.strip()] = [[int(v) for v in row.split()] for row in val.split(";")]
    return out


@pytest.fixture(scope="session")
def golden_worked_example():
    return load_golden("worked_example.txt")

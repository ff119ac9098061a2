import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture: '#' comments, whitespace-separated columns.
    Two-column lines -> {key: value}; three-column lines -> {(k1, k2): value}."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if len(parts) == 2:
                out[parts[0]] = parts[1]
            else:
                out[(parts[0], parts[1])] = parts[2]
    return out


@pytest.fixture(scope="session")
def golden():
    return load_golden

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built extension")


def read_golden(name):
    """Parse a 'key v1 v2 ...' golden file (lines starting with # are comments)."""
    out = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            try:
                rows.append([int(p) for p in parts])
            except ValueError:
                out[parts[0]] = parts[1:]
    if rows:
        out["_rows"] = rows
    return out


@pytest.fixture
def golden():
    return read_golden

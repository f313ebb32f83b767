import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (runs the libkda kernels through the C ABI)")


def read_fixture(name):
    """Parse a tests/golden text fixture: '# comment' lines and 'key: numbers'."""
    path = os.path.join(ROOT, "tests", "golden", name)
    out = {}
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(":")
            out[key.strip()] = [float(x) for x in rest.split()]
    return out


@pytest.fixture
def fixture_reader():
    return read_fixture

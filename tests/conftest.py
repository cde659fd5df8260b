import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 (sm_103a) GPU")
    config.addinivalue_line("markers", "slow: full-size parity case")


def read_golden(name):
    """Rows of a whitespace-separated fixture under tests/golden/, comments
    (#) and blank lines dropped; trailing words after the data columns are
    the row's derivation and are returned as one string."""
    path = os.path.join(ROOT, "tests", "golden", name)
    rows = []
    with open(path) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split(None, 2))
    return rows


@pytest.fixture(scope="session")
def golden():
    return read_golden

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
# The oracle mutation test (test_oracle_mutants.py) runs the pins again against
# a copy of the oracle package with one planted mistake; the copy's parent
# directory is named here and shadows the real package.
_MUTANT_DIR = os.environ.get("FA_ORACLE_MUTANT_DIR")
if _MUTANT_DIR:
    sys.path.insert(0, _MUTANT_DIR)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on the GB300 box)")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_lines(name):
    """Non-comment lines of a golden fixture, split on '|'."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            out.append([part.strip() for part in line.split("|")])
    return out


@pytest.fixture(scope="session")
def oracle_mod():
    from oracle import oracle
    oracle.lib()
    return oracle

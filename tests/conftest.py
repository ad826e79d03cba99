import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Rows of a ``|``-separated golden file, comments and blanks skipped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([field.strip() for field in line.split("|")])
    return rows


def parse_pow2_sum(text):
    """Parse values such as ``1+2^-12`` or ``2^-6`` or ``0`` exactly."""
    from fractions import Fraction

    total = Fraction(0)
    for term in text.replace(" ", "").split("+"):
        sign = 1
        if term.startswith("-"):
            sign, term = -1, term[1:]
        if term.startswith("2^"):
            total += sign * Fraction(2) ** int(term[2:])
        else:
            total += sign * Fraction(term)
    return total


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle

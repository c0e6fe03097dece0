import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def read_golden_table(name):
    """Rows of whitespace-separated numbers from a golden file (comments skipped)."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def read_golden_cases(name):
    """Parse 'case NAME ... end' blocks; each key maps to a list of rows
    (rows separated by '|'), each row a list of floats."""
    cases = {}
    cur = None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {}
                cases[rest.strip()] = cur
            elif key == "end":
                cur = None
            else:
                cur[key] = [[float(t) for t in part.split()] for part in rest.split("|")]
    return cases


@pytest.fixture(scope="session")
def golden_cases():
    return read_golden_cases("worked_example.txt")

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: CPU test that takes tens of seconds")


def read_table(name):
    """Integer rows of a golden file (comment lines start with '#')."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return rows


def read_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in (l.strip() for l in f) if ln and not ln.startswith("#")]

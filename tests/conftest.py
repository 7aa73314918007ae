import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (seconds to minutes)")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Rows of a golden fixture: list of lists of '|'-separated fields."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([f.strip() for f in line.split("|")])
    return rows


def pytest_sessionfinish(session, exitstatus):
    """Writes the near-tie counts the discrete checks allowed in this session
    (top-k rows against the oracle's own logits, selector paths within 1e-4
    of the oracle's best), one line per case, when any was recorded."""
    from tests.helpers import NEAR_TIES
    if not NEAR_TIES:
        return
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "near_tie_counts.txt")
    with open(path, "w") as fh:
        fh.write("# near-ties allowed by the discrete checks of the last GPU test session\n"
                 "# case | check | near-ties | total\n")
        for (case, kind), (n, t) in sorted(NEAR_TIES.items()):
            fh.write(f"{case} | {kind} | {n} | {t}\n")

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture
def golden():
    return load_golden


def pytest_terminal_summary(terminalreporter):
    """Report the flagged-draw counts of the sampler parity comparisons: draws
    within 1e-5 of a decision threshold, and how many of those sequences came
    out differently on the GPU (the exact check covers all the others)."""
    from tests.util import FLAG_LOG
    if not FLAG_LOG:
        return
    tot_f = sum(e[1] for e in FLAG_LOG)
    tot_n = sum(e[2] for e in FLAG_LOG)
    tot_d = sum(e[3] for e in FLAG_LOG)
    tr = terminalreporter
    tr.write_sep("-", f"flagged draws: {tot_f} of {tot_n} sequences flagged, {tot_d} of them "
                      f"differ, in {len(FLAG_LOG)} comparisons")
    by_test = {}
    for label, f, n, d in FLAG_LOG:
        a = by_test.setdefault(label, [0, 0, 0, 0])
        a[0] += f
        a[1] += n
        a[2] += d
        a[3] += 1
    for label, (f, n, d, c) in sorted(by_test.items()):
        if f:
            tr.write_line(f"  {label}: {f} flagged of {n}, {d} differ ({c} comparisons)")

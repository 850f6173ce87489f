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
    within 1e-5 of a decision threshold, which the bit-exact check skips."""
    from tests.util import FLAG_LOG
    if not FLAG_LOG:
        return
    tot_f = sum(f for _, f, _ in FLAG_LOG)
    tot_n = sum(n for _, _, n in FLAG_LOG)
    tr = terminalreporter
    tr.write_sep("-", f"flagged draws: {tot_f} of {tot_n} sequences in {len(FLAG_LOG)} comparisons")
    by_test = {}
    for label, f, n in FLAG_LOG:
        a = by_test.setdefault(label, [0, 0, 0])
        a[0] += f
        a[1] += n
        a[2] += 1
    for label, (f, n, c) in sorted(by_test.items()):
        if f:
            tr.write_line(f"  {label}: {f} flagged of {n} ({c} comparisons)")

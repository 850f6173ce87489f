"""The batched-serving workloads' drafter noise gives the acceptance rates the
configurations ask for (about 0.45 and 0.75 per draft position), measured with
the oracle's target distribution on rows of another seed than the one used to
calibrate (tests/calibrate_draft_noise.py)."""
import pytest

from speculative_decoding_verification_76_gb300 import workloads as wl
from tests.calibrate_draft_noise import mean_alpha


@pytest.mark.parametrize("name,target", [("batched_serving_a45", 0.45),
                                         ("batched_serving_a75", 0.75)])
def test_batched_alpha(name, target):
    spec = wl.SPECS[name]
    a = mean_alpha(spec, spec.draft_noise, B=4, seed=202)
    assert abs(a - target) < 0.03, a

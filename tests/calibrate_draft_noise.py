"""Calibrate the drafter noise sigma of the batched-serving workloads.

The batched-serving configurations ask for a draft whose acceptance rate is
about 0.45 and about 0.75.  For one draft position the acceptance rate is
alpha = sum_x min(p(x), q(x)) ("Speculative Decoding" (atlas), "Exact sampling:
account for every probability": the accepted mass of one proposal), with p the
target distribution as served (temperature 1, top-p 0.9, from the oracle) and
q the drafter's actual distribution (softmax(logits + N(0, sigma)), truncated
the same way, from the input generator).  Sigma is bisected on the mean alpha
over a sample of rows; the values found are written into workloads.py by hand
and pinned by tests/test_workload_alpha.py.

    python tests/calibrate_draft_noise.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import sampler as osm  # noqa: E402
from speculative_decoding_verification_76_gb300 import workloads as wl  # noqa: E402


def mean_alpha(spec: wl.Spec, sigma: float, B: int = 6, seed: int = 101) -> float:
    """Mean of sum_x min(p, q) over the draft rows of B sequences."""
    w = wl.make_sampler_inputs(spec.with_(B=B, draft_noise=float(sigma)), seed=seed)
    cfg = osm.SamplerCfg(temperature=spec.temperature, top_k=spec.top_k, top_p=spec.top_p)
    logits = w.logits.numpy()
    q = w.draft_probs.numpy().astype(np.float64)
    vals = []
    for b in range(B):
        for i in range(q.shape[1]):
            p, _ = osm.target_distribution(logits[b, i], cfg)
            vals.append(float(np.minimum(p, q[b, i]).sum()))
    return float(np.mean(vals))


def calibrate(spec: wl.Spec, target: float, lo=0.0, hi=6.0, iters=14) -> float:
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if mean_alpha(spec, mid) > target:
            lo = mid           # too easy to accept: more noise
        else:
            hi = mid
    return round(0.5 * (lo + hi), 3)


if __name__ == "__main__":
    base = wl.SPECS["batched_serving_a75"]
    for tgt in (0.45, 0.75):
        s = calibrate(base, tgt)
        print(f"alpha {tgt}: sigma {s} (mean alpha {mean_alpha(base, s):.4f})")

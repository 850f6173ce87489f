"""CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
shares no code with the CUDA library and never calls it.

Plain numpy in float64, written for a reader who checks it against the pages
by eye, with no blocking, fusion or reordering beyond the definitions:

  tree.py       ancestor masks, depth and position ids of a flattened draft
                tree ("Speculative Decoding" (atlas), "Chains, trees and
                visibility").
  attention.py  full-softmax multi-row attention with an explicit visibility
                set per row, read through the block table (the target's
                multi-position causal pass: "Drafters and Speculative
                Decoding", "From a proposed block to a causal target pass";
                split-K flash-decoding is exact up to rounding, so no split).
  sampler.py    target distribution (temperature, top-k, top-p), the
                left-to-right min(1, p/q) test on shifted rows, the residual
                norm(max(0, p - q)), the bonus token, greedy mode and the
                draft-tree rule ("Speculative Decoding" (atlas), "One round
                and shifted logits", "Exact sampling: account for every
                probability", "Greedy, sampling and the real sampler",
                "Implementation roadmap and tests"; "Drafters and Speculative
                Decoding", "Sampling needs a correction rule").
  commit.py     the next step's KV bookkeeping: the processed length after
                acceptance, the released pages, and a tree's accepted path
                compacted into the next logical prefix ("Speculative
                Decoding" (atlas), "Committed tokens versus cached states",
                "Chains, trees and visibility").
  append.py     the block's K/V rows written into the paged cache, keys
                rotated for their depth position ("Speculative Decoding"
                (atlas), "Chains, trees and visibility": position ids follow
                depth; the rotation itself is a reading, see the module).

Every function is pinned by a test in tests/test_oracle_*.py against worked
examples printed on the pages, closed forms or brute force.
"""
from . import append, attention, commit, sampler, tree  # noqa: F401

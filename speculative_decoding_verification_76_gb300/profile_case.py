"""One library call on a workload, for profilers (ncu -k ... -c ...).

    python -m speculative_decoding_verification_76_gb300.profile_case attn NAME B REPS
    python -m speculative_decoding_verification_76_gb300.profile_case sampler NAME B REPS

Builds the named synthetic workload with B sequences (same generator as the tests
and the bench) and makes REPS calls of the verify attention's partial pass or of
the acceptance sampler (no p returned), then synchronises.
"""
import sys

import torch

from . import api as sv
from . import workloads as wl


def main(argv):
    what, name, B = argv[0], argv[1], int(argv[2])
    reps = int(argv[3]) if len(argv) > 3 else 3
    spec = wl.SPECS[name].with_(B=B)
    if what == "attn":
        w = wl.make_attention_inputs(spec, device="cuda")
        # a chain needs no mask (the causal block), as in the verify step
        anc = sv.tree_prepare(w.parent, w.ctx_len)[0] if spec.is_tree else None
        call = sv.AttnCall(w.q, w.k_cache, w.v_cache, w.block_table, w.ctx_len, anc,
                           num_splits=spec.num_splits)
        for _ in range(reps):
            call.partials()
    elif what == "sampler":
        w = wl.make_sampler_inputs(spec, seed=spec.seed, device="cuda")
        cfg = sv.SamplerConfig(temperature=spec.temperature, top_k=spec.top_k, top_p=spec.top_p,
                               greedy=spec.greedy)
        for _ in range(reps):
            if spec.is_tree:
                sv.accept_sample_tree(w.logits, w.draft_probs, w.draft_tokens, w.parent,
                                      w.uniforms, cfg)
            else:
                sv.accept_sample(w.logits, w.draft_probs, w.draft_tokens, w.uniforms, cfg)
    else:
        raise SystemExit(f"unknown case {what!r}: attn or sampler")
    torch.cuda.synchronize()
    print("ok", what, name, B, reps)


if __name__ == "__main__":
    main(sys.argv[1:])

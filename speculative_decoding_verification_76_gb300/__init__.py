"""GB300-native verification step of speculative decoding.

The compute lives in libspecverify.so (hand-written CUDA for sm_103a, C ABI in
include/spec_verify.h); this package is its thin binding plus the seeded
workload generator used by the tests and the benchmark.
"""
from .api import (AttnCall, SamplerConfig, SpecError, accept_sample,  # noqa: F401
                  accept_sample_tree, append_block, attn_num_splits, attn_workspace_size,
                  kv_commit, load, logits_penalize, new_workspace, sample_workspace_size,
                  tree_prepare, verify_attn, workspace_error)

"""Bounded device waits: a wait that runs out ends the kernel with an error word.

spec_debug_attn_fault makes the copy warps of the attention partial passes
withhold one K/V stage and bounds every wait by 20 us, so the waits on that
stage run out on purpose.  The call must return, the workspace error word must
read SPEC_ERR_MBAR_TIMEOUT, and the next normal call on a fresh workspace must
agree with the oracle.  Covered: the warp-MMA pass (a chain), both tcgen05
passes (128 and 512 rows per KV head), and the allocation-free variant's error
reader.  No GPU fault is involved: every wait is bounded and every warp role
returns (tensor memory is freed after the last tensor-core operation).
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_76_gb300 as sv
from speculative_decoding_verification_76_gb300 import api
from speculative_decoding_verification_76_gb300 import workloads as wl
from tests.util import BF16_ATOL, np_u64, oracle_attention

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SPEC_ERR_MBAR_TIMEOUT = 0x100

SHAPES = [
    # name, spec: 20, 128 and 512 query rows per KV head
    ("warp_mma_chain", wl.Spec("wt_chain", B=2, Hq=32, Hkv=8, D=128, V=16, ctx=(1500, 2600),
                               gamma=4, shuffle_pages=True, seed=41)),
    ("tcgen05_one_tile", wl.Spec("wt_long", B=1, Hq=64, Hkv=8, D=128, V=16, ctx=(3000, 3000),
                                 gamma=15, seed=42)),
    ("tcgen05_two_tiles", wl.Spec("wt_tree", B=1, Hq=64, Hkv=8, D=128, V=16, ctx=(2500, 2500),
                                  tree_nodes=64, seed=43)),
]


def _fault(stage, ns):
    assert api.load().spec_debug_attn_fault(stage, ns) == api.SPEC_OK


@pytest.mark.parametrize("name,spec", SHAPES, ids=[s[0] for s in SHAPES])
def test_withheld_stage_times_out_then_recovers(name, spec):
    w = wl.make_attention_inputs(spec, device=DEV)
    anc, _, _ = sv.tree_prepare(w.parent, w.ctx_len)
    ws_bytes = sv.attn_workspace_size(spec.B, spec.R, spec.Hq, spec.Hkv, spec.D, spec.page_size,
                                      w.block_table.shape[1], 1)
    try:
        _fault(1, 20_000)                  # stage 1 never arrives; waits end after ~20 us
        ws = sv.new_workspace(ws_bytes, DEV)
        sv.verify_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.ctx_len, anc,
                       num_splits=1, workspace=ws)
        torch.cuda.synchronize()           # the kernels returned
        assert sv.workspace_error(ws) == SPEC_ERR_MBAR_TIMEOUT
    finally:
        _fault(-1, 0)
    # the context is usable and a normal call on a fresh workspace is correct
    ws = sv.new_workspace(ws_bytes, DEV)
    out, _ = sv.verify_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.ctx_len, anc,
                            num_splits=1, workspace=ws)
    torch.cuda.synchronize()
    assert sv.workspace_error(ws) == 0
    G = spec.Hq // spec.Hkv
    heads = [k * G + k % G for k in range(spec.Hkv)]
    ref, _ = oracle_attention(w, np_u64(anc), heads=heads)
    got = out.float().cpu().numpy()
    assert np.abs(got[:, :, heads] - ref[:, :, heads]).max() < BF16_ATOL


def test_noalloc_reports_a_timeout():
    spec = SHAPES[0][1]
    w = wl.make_attention_inputs(spec, device=DEV)
    anc, _, _ = sv.tree_prepare(w.parent, w.ctx_len)
    lib = api.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.empty_like(w.q)
    lse = torch.empty((spec.B, spec.R, spec.Hq), dtype=torch.float32, device=DEV)

    def call():
        npg, P, Hkv, D = w.k_cache.shape
        return lib.spec_verify_attn_noalloc(
            api._ptr(w.q), api._ptr(w.k_cache), api._ptr(w.v_cache), api.SPEC_BF16, P, npg,
            api._ptr(w.block_table), w.block_table.shape[1], api._ptr(w.ctx_len), api._ptr(anc),
            spec.B, spec.R, spec.Hq, Hkv, D, 0.0, 1, api._ptr(out), api._ptr(lse), stream)

    err = ctypes.c_int32(-1)
    try:
        _fault(1, 20_000)
        assert call() == api.SPEC_OK
        assert lib.spec_verify_attn_noalloc_error(ctypes.byref(err), stream) == api.SPEC_OK
        assert err.value == SPEC_ERR_MBAR_TIMEOUT
    finally:
        _fault(-1, 0)
    assert call() == api.SPEC_OK                 # each call clears the word first
    assert lib.spec_verify_attn_noalloc_error(ctypes.byref(err), stream) == api.SPEC_OK
    assert err.value == 0
    ref, _ = sv.verify_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.ctx_len, anc,
                            num_splits=1)
    torch.cuda.synchronize()
    np.testing.assert_allclose(out.float().cpu().numpy(), ref.float().cpu().numpy(), rtol=0,
                               atol=BF16_ATOL)

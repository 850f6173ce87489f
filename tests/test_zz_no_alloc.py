"""The allocation-free attention entry point, called through the C ABI.

spec_verify_attn_noalloc serves callers that cannot allocate device memory
(for example a plugin host that only passes its input/output buffers, or a
serving loop whose memory is fixed after start-up): its scratch is a fixed
array inside the library.  These tests check that it returns what the
workspace-based spec_verify_attn returns, on two calls in a row with
different problems (the shared array keeps the previous call's contents),
that the call's error word (read with spec_verify_attn_noalloc_error) stays
zero, and that a problem too big for the array is refused before any launch.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_76_gb300 as sv
from speculative_decoding_verification_76_gb300 import api
from speculative_decoding_verification_76_gb300 import workloads as wl
from tests.util import BF16_ATOL

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
P, I = ctypes.c_void_p, ctypes.c_int


def _fn():
    lib = sv.load()
    f = lib.spec_verify_attn_noalloc
    f.restype = I
    f.argtypes = [P, P, P, I, I, I, P, I, P, P, I, I, I, I, I, ctypes.c_float, I, P, P, P]
    return f


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call(f, w, anc, out, lse):
    B, R, Hq, D = w.q.shape
    npg, Pg, Hkv, _ = w.k_cache.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(_ptr(w.q), _ptr(w.k_cache), _ptr(w.v_cache), api.SPEC_BF16, Pg, npg,
             _ptr(w.block_table), w.block_table.shape[1], _ptr(w.ctx_len), _ptr(anc), B, R, Hq,
             Hkv, D, 0.0, 0, _ptr(out), _ptr(lse), stream)


def test_noalloc_matches_workspace_entry_point_twice():
    f = _fn()
    specs = [wl.Spec("na1", B=2, Hq=32, Hkv=8, D=128, V=16, ctx=(900, 3000), gamma=7,
                     shuffle_pages=True, seed=21),
             wl.Spec("na2", B=2, Hq=16, Hkv=2, D=128, V=16, ctx=(100, 700), tree_nodes=16,
                     shuffle_pages=True, seed=22)]
    for spec in specs:                       # two calls in a row, different problems
        w = wl.make_attention_inputs(spec, device=DEV)
        need = sv.attn_workspace_size(spec.B, spec.R, spec.Hq, spec.Hkv, spec.D, spec.page_size,
                                      w.block_table.shape[1])
        assert need <= (8 << 20)
        anc, _, _ = sv.tree_prepare(w.parent, w.ctx_len)
        ref_out, ref_lse = sv.verify_attn(w.q, w.k_cache, w.v_cache, w.block_table, w.ctx_len,
                                          anc)
        out = torch.full_like(w.q, float("nan"))
        lse = torch.full(ref_lse.shape, float("nan"), device=DEV)
        assert _call(f, w, anc, out, lse) == api.SPEC_OK
        # the call's error word, read without allocating: no bounded wait ran out
        err = ctypes.c_int32(-1)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        assert sv.load().spec_verify_attn_noalloc_error(ctypes.byref(err), stream) == api.SPEC_OK
        assert err.value == 0
        torch.cuda.synchronize()
        np.testing.assert_allclose(out.float().cpu().numpy(), ref_out.float().cpu().numpy(),
                                   rtol=0, atol=BF16_ATOL)
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), rtol=0, atol=1e-3)


def test_noalloc_refuses_problems_beyond_the_array():
    f = _fn()
    spec = wl.SPECS["long_context"]           # split-K scratch far above the fixed array
    R, B = spec.R, 1
    maxp = (spec.ctx[1] + R + 15) // 16
    need = sv.attn_workspace_size(B, R, spec.Hq, spec.Hkv, spec.D, 16, maxp, spec.num_splits)
    assert need > (8 << 20)
    null = ctypes.c_void_p(16)             # never dereferenced: refused on the host
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = f(null, null, null, api.SPEC_BF16, 16, maxp, null, maxp, null, null, B, R, spec.Hq,
           spec.Hkv, spec.D, 0.0, spec.num_splits, null, null, stream)
    assert rc == api.SPEC_EUNSUPPORTED

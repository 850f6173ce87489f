"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_76_gb300 as sv
from speculative_decoding_verification_76_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_76_gb300 import build
    build.build()
    return sv.load()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(spec_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(api.EXPORTS) <= set(names)


def test_status_strings(lib):
    for code in range(5):
        assert lib.spec_status_str(code).startswith(b"SPEC_")


def test_host_validation_rejects_bad_arguments(lib):
    null = None
    # tree_prepare: R out of range, missing outputs
    assert lib.spec_tree_prepare(null, ctypes.c_void_p(16), 1, 0, ctypes.c_void_p(16), null, null,
                                 null) == api.SPEC_EINVAL
    assert lib.spec_tree_prepare(null, ctypes.c_void_p(16), 1, 65, ctypes.c_void_p(16), null, null,
                                 null) == api.SPEC_EINVAL
    assert lib.spec_tree_prepare(null, null, 1, 4, ctypes.c_void_p(16), null, null,
                                 null) == api.SPEC_EINVAL
    # attention: null pointers, head-count mismatch, unsupported head_dim
    p = ctypes.c_void_p(4096)
    args = [p, p, p, api.SPEC_BF16, 16, 10, p, 4, p, p, 1, 4, 8, 2, 128, 0.0, 0, p, 1 << 20, p,
            null, null]
    # (args itself is never passed: only copies that the host must reject)
    bad = list(args)
    bad[0] = null
    assert lib.spec_verify_attn(*bad) == api.SPEC_EINVAL
    bad = list(args)
    bad[12] = 3                           # Hq % Hkv != 0
    assert lib.spec_verify_attn(*bad) == api.SPEC_EINVAL
    bad = list(args)
    bad[14] = 96                          # head_dim 96
    assert lib.spec_verify_attn(*bad) == api.SPEC_EUNSUPPORTED
    bad = list(args)
    bad[10] = 1
    bad[11] = 65                          # R > 64
    assert lib.spec_verify_attn(*bad) == api.SPEC_EUNSUPPORTED
    bad = list(args)
    bad[17] = ctypes.c_void_p(4096 + 8)   # workspace not 256-B aligned
    assert lib.spec_verify_attn(*bad) == api.SPEC_EINVAL
    bad = list(args)
    bad[18] = 16                          # workspace too small
    assert lib.spec_verify_attn(*bad) == api.SPEC_EINVAL


def test_sampler_config_validation(lib):
    p = ctypes.c_void_p(4096)
    ws = sv.sample_workspace_size(2, 5, 100)

    def call(cfg, B=2, R=5, V=100, wsb=ws, logits=p):
        c = cfg.c()
        return lib.spec_accept_sample(logits, p, p, p, B, R, V, ctypes.byref(c), p, wsb, p, p,
                                      None, None, None)

    assert call(api.SamplerConfig(temperature=0.0)) == api.SPEC_EINVAL
    assert call(api.SamplerConfig(temperature=-1.0)) == api.SPEC_EINVAL
    assert call(api.SamplerConfig(top_p=0.0)) == api.SPEC_EINVAL
    assert call(api.SamplerConfig(top_p=1.5)) == api.SPEC_EINVAL
    assert call(api.SamplerConfig(top_k=-2)) == api.SPEC_EINVAL
    assert call(api.SamplerConfig(), wsb=8) == api.SPEC_EINVAL
    assert call(api.SamplerConfig(), logits=None) == api.SPEC_EINVAL
    assert call(api.SamplerConfig(), R=65) == api.SPEC_EUNSUPPORTED
    assert call(api.SamplerConfig(), V=1 << 20) == api.SPEC_EUNSUPPORTED
    assert call(api.SamplerConfig(), B=0) == api.SPEC_OK     # empty batch: nothing to do
    c = api.SamplerConfig().c()
    assert lib.spec_accept_sample_tree(p, p, p, p, p, 2, 1, 100, ctypes.byref(c), p, ws, p, p, p,
                                       None, None, None) == api.SPEC_EINVAL


def test_workspace_sizes(lib):
    a = sv.attn_workspace_size(1, 8, 32, 8, 128, 16, 513)
    b = sv.attn_workspace_size(64, 5, 32, 8, 128, 16, 1026)
    assert 0 < a < b
    assert sv.attn_workspace_size(1, 8, 32, 8, 128, 16, 513, 0) % 256 == 0
    # explicit splits are honoured up to the 64-token stage granularity
    assert sv.attn_num_splits(1, 16, 64, 8, 128, 16, 8193, 128) >= 128
    assert sv.sample_workspace_size(4, 64, 128256) >= 256 + 4 * 64 * 16
    # the two-pass variant: few rows need nothing more; many rows room for the
    # pre-pass results (per row: 32 range records, 32 x 8 segments of 128 listed
    # ids and logits, their counts, the floor)
    few, mn = sv.sample_workspace_size(1, 8, 128256, True), sv.sample_workspace_size(1, 8, 128256)
    assert few == mn and mn % 256 == 0
    big, mn = sv.sample_workspace_size(64, 5, 152064, True), sv.sample_workspace_size(64, 5, 152064)
    assert big >= mn + 320 * (32 * 16 + 32 * 8 * 128 * 8 + 32 * 8 * 4 + 8)
    assert sv.sample_workspace_size(64, 5, 0) == 0          # no vocabulary: invalid
    assert sv.sample_workspace_size(64, 5, 0, True) == 0
    # the per-sequence counters have one place for every shape (65536 of them
    # after the 256-byte header); the rest grows with the rows
    one = sv.sample_workspace_size(1, 1, 100)
    assert one >= 256 + 65536 * 4
    assert sv.sample_workspace_size(64, 5, 100) - one < 64 * 5 * 16 + 256


def test_sampler_batch_limit_refused_on_host(lib):
    # more than 65536 sequences: refused before any launch (no device pointer
    # is touched, so dummy addresses do)
    p = ctypes.c_void_p(256)
    c = api.SamplerConfig().c()
    rc = lib.spec_accept_sample(p, p, p, p, 65537, 2, 100, ctypes.byref(c), p, 1 << 40, p, p,
                                None, None, None)
    assert rc == api.SPEC_EUNSUPPORTED


def test_kv_commit_host_validation(lib):
    # argument errors are refused on the host, before any launch
    buf = (ctypes.c_int32 * 128)()
    p = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)  # 16-byte aligned host memory
    assert lib.spec_kv_commit(None, None, 2, 1, 16, 1, 128, p, 1, p, p, None, None, 1, 8, p,
                              None, None, None) == api.SPEC_EINVAL
    assert lib.spec_kv_commit(p, p, 2, 1, 16, 1, 128, p, 1, p, p, None, None, 1, 65, p, None,
                              None, None) == api.SPEC_EINVAL
    assert lib.spec_kv_commit(p, p, 2, 1, 16, 1, 96, p, 1, p, p, None, None, 1, 8, p, None, None,
                              None) == api.SPEC_EUNSUPPORTED
    assert lib.spec_kv_commit(p, p, 3, 1, 16, 1, 128, p, 1, p, p, None, None, 1, 8, p, None, None,
                              None) == api.SPEC_EUNSUPPORTED
    # a parent array without a path has nothing to check
    assert lib.spec_kv_commit(p, p, 2, 1, 16, 1, 128, p, 1, p, p, None, p, 1, 8, p, None, None,
                              None) == api.SPEC_EINVAL
    assert lib.spec_kv_commit(p, p, 2, 1, 16, 1, 128, p, 1, p, p, None, None, 0, 8, p, None, None,
                              None) == api.SPEC_OK  # nothing to do


def test_split_plan_for_the_bench_shapes(lib):
    # few units: about one wave of CTAs (8B-shaped: 8 KV heads x 17 splits of 512 tokens);
    # units that fill the SMs: 4096-token chunks; explicit counts are honoured
    assert sv.attn_num_splits(1, 8, 32, 8, 128, 16, 513) == 17
    assert sv.attn_num_splits(64, 5, 32, 8, 128, 16, 1025) == 5  # 16400 tokens / 4096
    assert sv.attn_num_splits(1, 16, 64, 8, 128, 16, 8193) == 33  # 131088 tokens / 4096
    assert sv.attn_num_splits(1, 16, 64, 8, 128, 16, 8193, 128) >= 128


def test_noalloc_host_checks(lib):
    # a null output for the error reader, and sizes refused before any device work
    assert lib.spec_verify_attn_noalloc_error(None, None) == api.SPEC_EINVAL
    p = ctypes.c_void_p(4096)
    assert lib.spec_verify_attn_noalloc(p, p, p, api.SPEC_BF16, 16, 10, p, 4, p, p, -1, 4, 8, 2,
                                        128, 0.0, 0, p, None, None) == api.SPEC_EINVAL
    assert lib.spec_verify_attn_noalloc(p, p, p, api.SPEC_BF16, 16, 10, p, 4, p, p, 0, 4, 8, 2,
                                        128, 0.0, 0, p, None, None) == api.SPEC_OK


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(api, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        api.load(str(tmp_path / "missing.so"))


def test_debug_fault_setting_host_checks(lib):
    assert lib.spec_debug_attn_fault(-2, 0) == api.SPEC_EINVAL
    assert lib.spec_debug_attn_fault(3, 1000) == api.SPEC_OK
    assert lib.spec_debug_attn_fault(-1, 0) == api.SPEC_OK     # restored

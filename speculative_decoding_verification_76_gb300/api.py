"""Thin Python binding of libspecverify.so (argument marshalling only).

Every function here checks tensor placement, dtype and shape, allocates the
outputs and workspaces with PyTorch, and calls the C ABI declared in
include/spec_verify.h on the current CUDA stream.  All arithmetic of the
verify step runs in the library's kernels; there is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SPEC_OK, SPEC_EINVAL, SPEC_EUNSUPPORTED, SPEC_ECUDA, SPEC_ETIMEOUT = range(5)
SPEC_F32, SPEC_BF16 = 0, 1
SEQ_QZERO, SEQ_NONFINITE, SEQ_RESID_ZERO, SEQ_BAD_TREE = 1, 2, 4, 8

# every symbol include/spec_verify.h declares
EXPORTS = (
    "spec_status_str", "spec_tree_prepare", "spec_verify_attn_workspace_size",
    "spec_verify_attn_num_splits", "spec_verify_attn", "spec_verify_attn_partials",
    "spec_verify_attn_combine", "spec_accept_sample_workspace_size",
    "spec_accept_sample_workspace_size_two_pass",
    "spec_accept_sample", "spec_accept_sample_tree", "spec_workspace_error",
    "spec_kv_commit", "spec_verify_attn_noalloc", "spec_verify_attn_noalloc_error",
    "spec_append_block", "spec_logits_penalize", "spec_debug_attn_fault",
)


class SpecError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


class _Sampler(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32),
                ("top_p", ctypes.c_float), ("greedy", ctypes.c_int32),
                ("eos_id", ctypes.c_int32)]


@dataclass
class SamplerConfig:
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    greedy: bool = False
    eos_id: int = -1

    def c(self) -> _Sampler:
        return _Sampler(float(self.temperature), int(self.top_k), float(self.top_p),
                        1 if self.greedy else 0, int(self.eos_id))


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "(nvcc, sm_103a); there is no CPU fallback")
    lib = ctypes.CDLL(path)
    lib.spec_status_str.restype = ctypes.c_char_p
    lib.spec_status_str.argtypes = [_I]
    lib.spec_tree_prepare.restype = _I
    lib.spec_tree_prepare.argtypes = [_P, _P, _I, _I, _P, _P, _P, _P]
    lib.spec_verify_attn_workspace_size.restype = _SZ
    lib.spec_verify_attn_workspace_size.argtypes = [_I] * 8
    lib.spec_verify_attn_num_splits.restype = _I
    lib.spec_verify_attn_num_splits.argtypes = [_I] * 8
    lib.spec_verify_attn.restype = _I
    lib.spec_verify_attn.argtypes = [_P, _P, _P, _I, _I, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I,
                                     ctypes.c_float, _I, _P, _SZ, _P, _P, _P]
    common = [_P, _P, _P, _I, _I, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _I, _P,
              _SZ]
    lib.spec_verify_attn_partials.restype = _I
    lib.spec_verify_attn_partials.argtypes = common + [_P]
    lib.spec_verify_attn_combine.restype = _I
    lib.spec_verify_attn_combine.argtypes = common + [_P, _P, _P]
    lib.spec_accept_sample_workspace_size.restype = _SZ
    lib.spec_accept_sample_workspace_size.argtypes = [_I, _I, _I]
    lib.spec_accept_sample_workspace_size_two_pass.restype = _SZ
    lib.spec_accept_sample_workspace_size_two_pass.argtypes = [_I, _I, _I]
    lib.spec_accept_sample.restype = _I
    lib.spec_accept_sample.argtypes = [_P, _P, _P, _P, _I, _I, _I, ctypes.POINTER(_Sampler), _P,
                                       _SZ, _P, _P, _P, _P, _P]
    lib.spec_accept_sample_tree.restype = _I
    lib.spec_accept_sample_tree.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I,
                                            ctypes.POINTER(_Sampler), _P, _SZ, _P, _P, _P, _P, _P,
                                            _P]
    lib.spec_workspace_error.restype = _I
    lib.spec_workspace_error.argtypes = [_P, ctypes.POINTER(ctypes.c_int32), _P]
    lib.spec_kv_commit.restype = _I
    lib.spec_kv_commit.argtypes = [_P, _P, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P, _I, _I,
                                   _P, _P, _P, _P]
    lib.spec_verify_attn_noalloc.restype = _I
    lib.spec_verify_attn_noalloc.argtypes = [_P, _P, _P, _I, _I, _I, _P, _I, _P, _P, _I, _I, _I,
                                             _I, _I, ctypes.c_float, _I, _P, _P, _P]
    lib.spec_append_block.restype = _I
    lib.spec_append_block.argtypes = [_P, _P, _P, _I, _P, _P, _I, _I, _P, _I, _P, _P, _I, _I, _I,
                                      _I, _I, ctypes.c_float, _P, _P]
    lib.spec_logits_penalize.restype = _I
    lib.spec_logits_penalize.argtypes = [_P, _I, _I, _I, _P, _I, _P, _P, ctypes.c_float, _P, _I,
                                         _P]
    lib.spec_debug_attn_fault.restype = _I
    lib.spec_debug_attn_fault.argtypes = [_I, ctypes.c_ulonglong]
    lib.spec_verify_attn_noalloc_error.restype = _I
    lib.spec_verify_attn_noalloc_error.argtypes = [ctypes.POINTER(ctypes.c_int32), _P]
    _lib = lib
    return lib


def _check(fn: str, rc: int):
    if rc != SPEC_OK:
        raise SpecError(fn, rc, load().spec_status_str(rc).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """Zero-filled workspace (the library's counters start at zero)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def workspace_error(ws: torch.Tensor) -> int:
    v = ctypes.c_int32(0)
    _check("spec_workspace_error", load().spec_workspace_error(_ptr(ws), ctypes.byref(v),
                                                               _stream()))
    return int(v.value)


# ------------------------------------------------------------------ tree_prepare
def tree_prepare(parent: torch.Tensor | None, ctx_len: torch.Tensor, R: int | None = None,
                 anc_mask=None, pos_ids=None, status=None):
    """Ancestor mask [B,R] (int64 holding uint64 bits), position ids, per-seq status."""
    lib = load()
    _need(ctx_len, "ctx_len", torch.int32)
    B = ctx_len.shape[0]
    if parent is not None:
        _need(parent, "parent", torch.int32)
        R = parent.shape[1]
    dev = ctx_len.device
    anc_mask = torch.empty((B, R), dtype=torch.int64, device=dev) if anc_mask is None else anc_mask
    pos_ids = torch.empty((B, R), dtype=torch.int32, device=dev) if pos_ids is None else pos_ids
    status = torch.empty((B,), dtype=torch.int32, device=dev) if status is None else status
    _check("spec_tree_prepare", lib.spec_tree_prepare(_ptr(parent), _ptr(ctx_len), B, R,
                                                      _ptr(anc_mask), _ptr(pos_ids), _ptr(status),
                                                      _stream()))
    return anc_mask, pos_ids, status


def kv_commit(k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
              ctx_len: torch.Tensor, accepted_len: torch.Tensor, path=None, parent=None,
              R: int | None = None, new_len=None, keep_pages=None, status=None, stream=None):
    """Processed lengths after acceptance.  For a tree, path [B,R] int32 holds the
    accepted nodes (node 0 implied), as accept_sample_tree returns them; their K/V
    rows move in place to positions ctx + 1 .. ctx + accepted_len.  parent [B,R]
    (optional) lets the kernel check that the path follows the tree.
    Returns (new_len, keep_pages, status)."""
    lib = load()
    if k_cache.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("caches must be bf16 or fp32")
    npg, P, Hkv, D = k_cache.shape
    _need(k_cache, "k_cache", k_cache.dtype)
    _need(v_cache, "v_cache", k_cache.dtype, k_cache.shape)
    _need(block_table, "block_table", torch.int32)
    _need(ctx_len, "ctx_len", torch.int32)
    B = ctx_len.shape[0]
    _need(accepted_len, "accepted_len", torch.int32, (B,))
    if path is not None:
        _need(path, "path", torch.int32)
        R = path.shape[1]
    if parent is not None:
        _need(parent, "parent", torch.int32, (B, R))
    if R is None:
        raise ValueError("R (rows per sequence) is needed for a chain")
    dev = ctx_len.device
    new_len = torch.empty((B,), dtype=torch.int32, device=dev) if new_len is None else new_len
    keep_pages = (torch.empty((B,), dtype=torch.int32, device=dev) if keep_pages is None
                  else keep_pages)
    status = torch.empty((B,), dtype=torch.int32, device=dev) if status is None else status
    _check("spec_kv_commit",
           lib.spec_kv_commit(_ptr(k_cache), _ptr(v_cache), k_cache.element_size(), npg, P, Hkv,
                              D, _ptr(block_table), block_table.shape[1], _ptr(ctx_len),
                              _ptr(accepted_len), _ptr(path), _ptr(parent), B, R, _ptr(new_len),
                              _ptr(keep_pages), _ptr(status), _stream(stream)))
    return new_len, keep_pages, status


def append_block(k_new, v_new, k_cache, v_cache, block_table, ctx_len, pos_ids=None, q=None,
                 rope_base: float = 10000.0, status=None, stream=None):
    """Write the block's K/V rows (keys rotated at pos_ids; NULL: chain positions)
    into the paged cache at ctx + j, and rotate q [B,R,Hq,D] in place if given.
    Returns status [B]."""
    lib = load()
    dt = k_new.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("k_new must be bf16 or fp32")
    B, R, Hkv, D = k_new.shape
    npg, P = k_cache.shape[0], k_cache.shape[1]
    _need(k_new, "k_new", dt)
    _need(v_new, "v_new", dt, k_new.shape)
    _need(k_cache, "k_cache", dt)
    _need(v_cache, "v_cache", dt, k_cache.shape)
    if tuple(k_cache.shape[2:]) != (Hkv, D):
        raise ValueError("cache heads / head_dim differ from the block's")
    _need(block_table, "block_table", torch.int32)
    _need(ctx_len, "ctx_len", torch.int32, (B,))
    if pos_ids is not None:
        _need(pos_ids, "pos_ids", torch.int32, (B, R))
    Hq = 0
    if q is not None:
        _need(q, "q", dt)
        if q.shape[0] != B or q.shape[1] != R or q.shape[3] != D:
            raise ValueError("q must be [B, R, Hq, D]")
        Hq = q.shape[2]
    status = torch.empty((B,), dtype=torch.int32, device=k_new.device) if status is None \
        else status
    _check("spec_append_block",
           lib.spec_append_block(_ptr(k_new), _ptr(v_new), _ptr(q),
                                 SPEC_BF16 if dt == torch.bfloat16 else SPEC_F32, _ptr(k_cache),
                                 _ptr(v_cache), npg, P, _ptr(block_table), block_table.shape[1],
                                 _ptr(ctx_len), _ptr(pos_ids), B, R, Hq, Hkv, D,
                                 float(rope_base), _ptr(status), _stream(stream)))
    return status


def logits_penalize(logits, history=None, block_tokens=None, parent=None, penalty: float = 1.0,
                    banned=None, stream=None):
    """Repetition penalty over each row's prefix, then bans, on logits [B,R,V] in place."""
    lib = load()
    _need(logits, "logits", torch.float32)
    B, R, V = logits.shape
    H = 0
    if history is not None:
        _need(history, "history", torch.int32)
        H = history.shape[1]
    if block_tokens is not None:
        _need(block_tokens, "block_tokens", torch.int32)
    if parent is not None:
        _need(parent, "parent", torch.int32, (B, R))
    nb = 0
    if banned is not None:
        _need(banned, "banned", torch.int32)
        nb = banned.numel()
    _check("spec_logits_penalize",
           lib.spec_logits_penalize(_ptr(logits), B, R, V, _ptr(history), H, _ptr(block_tokens),
                                    _ptr(parent), float(penalty), _ptr(banned), nb,
                                    _stream(stream)))
    return logits


# ------------------------------------------------------------------ attention
def attn_workspace_size(B, R, Hq, Hkv, D, page_size, max_pages, num_splits=0) -> int:
    return int(load().spec_verify_attn_workspace_size(B, R, Hq, Hkv, D, page_size, max_pages,
                                                      num_splits))


def attn_num_splits(B, R, Hq, Hkv, D, page_size, max_pages, num_splits=0) -> int:
    return int(load().spec_verify_attn_num_splits(B, R, Hq, Hkv, D, page_size, max_pages,
                                                  num_splits))


def verify_attn(q, k_cache, v_cache, block_table, ctx_len, anc_mask, scale: float = 0.0,
                num_splits: int = 0, workspace=None, out=None, lse=None, stream=None):
    """Split-K verify attention.  q [B,R,Hq,D]; caches [pages,P,Hkv,D]; returns (out, lse)."""
    lib = load()
    dt = q.dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("q must be bf16 or fp32")
    B, R, Hq, D = q.shape
    npg, P, Hkv, D2 = k_cache.shape
    if D2 != D:
        raise ValueError("head_dim mismatch")
    _need(q, "q", dt)
    _need(k_cache, "k_cache", dt)
    _need(v_cache, "v_cache", dt, k_cache.shape)
    _need(block_table, "block_table", torch.int32)
    _need(ctx_len, "ctx_len", torch.int32, (B,))
    if anc_mask is not None:          # None: a chain (row i sees block rows 0 .. i)
        _need(anc_mask, "anc_mask", torch.int64, (B, R))
    maxp = block_table.shape[1]
    if workspace is None:
        workspace = new_workspace(attn_workspace_size(B, R, Hq, Hkv, D, P, maxp, num_splits),
                                  q.device)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, R, Hq), dtype=torch.float32, device=q.device)
    rc = lib.spec_verify_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                              SPEC_BF16 if dt == torch.bfloat16 else SPEC_F32, P, npg,
                              _ptr(block_table), maxp, _ptr(ctx_len), _ptr(anc_mask), B, R, Hq,
                              Hkv, D, float(scale), int(num_splits), _ptr(workspace),
                              workspace.numel(), _ptr(out), _ptr(lse), _stream(stream))
    _check("spec_verify_attn", rc)
    return out, lse


class AttnCall:
    """Pre-marshalled arguments of one verify-attention problem.

    Builds the argument list once (pointers, shapes, workspace) so repeated
    calls -- e.g. inside a timed loop or a CUDA-graph capture -- do no Python
    work beyond the foreign call.  partials() and combine() are the two
    phases; __call__ runs both."""

    def __init__(self, q, k_cache, v_cache, block_table, ctx_len, anc_mask, scale=0.0,
                 num_splits=0, workspace=None, out=None, lse=None):
        dt = q.dtype
        B, R, Hq, D = q.shape
        npg, P, Hkv, _ = k_cache.shape
        _need(q, "q", dt)
        _need(k_cache, "k_cache", dt)
        _need(v_cache, "v_cache", dt, k_cache.shape)
        _need(block_table, "block_table", torch.int32)
        _need(ctx_len, "ctx_len", torch.int32, (B,))
        if anc_mask is not None:      # None: a chain
            _need(anc_mask, "anc_mask", torch.int64, (B, R))
        maxp = block_table.shape[1]
        self.workspace = workspace if workspace is not None else new_workspace(
            attn_workspace_size(B, R, Hq, Hkv, D, P, maxp, num_splits), q.device)
        self.out = torch.empty_like(q) if out is None else out
        self.lse = torch.empty((B, R, Hq), dtype=torch.float32, device=q.device) \
            if lse is None else lse
        self._keep = (q, k_cache, v_cache, block_table, ctx_len, anc_mask)
        self.args = [_ptr(q), _ptr(k_cache), _ptr(v_cache),
                     SPEC_BF16 if dt == torch.bfloat16 else SPEC_F32, P, npg, _ptr(block_table),
                     maxp, _ptr(ctx_len), _ptr(anc_mask), B, R, Hq, Hkv, D, float(scale),
                     int(num_splits), _ptr(self.workspace), self.workspace.numel()]
        self.lib = load()

    def partials(self, stream=None):
        _check("spec_verify_attn_partials",
               self.lib.spec_verify_attn_partials(*self.args, _stream(stream)))

    def combine(self, stream=None):
        _check("spec_verify_attn_combine",
               self.lib.spec_verify_attn_combine(*self.args, _ptr(self.out), _ptr(self.lse),
                                                 _stream(stream)))

    def __call__(self, stream=None):
        _check("spec_verify_attn",
               self.lib.spec_verify_attn(*self.args, _ptr(self.out), _ptr(self.lse),
                                         _stream(stream)))
        return self.out, self.lse


# ------------------------------------------------------------------ sampler
def sample_workspace_size(B, R, V, two_pass: bool = False) -> int:
    """Bytes of sampler workspace; two_pass: room for the two-pass streaming
    variant (many truncated rows), which a workspace of that size selects."""
    if two_pass:
        return int(load().spec_accept_sample_workspace_size_two_pass(B, R, V))
    return int(load().spec_accept_sample_workspace_size(B, R, V))


def accept_sample(logits, draft_probs, draft_tokens, uniforms, cfg: SamplerConfig,
                  workspace=None, want_p: bool = False, out=None, stream=None):
    """Chain verification.  Returns dict(accepted_len, emitted, status[, p])."""
    lib = load()
    _need(logits, "target_logits", torch.float32)
    B, R, V = logits.shape
    if draft_probs is not None:
        _need(draft_probs, "draft_probs", torch.float32, (B, R - 1, V))
    if draft_tokens is not None:
        _need(draft_tokens, "draft_tokens", torch.int32, (B, R - 1))
    if uniforms is not None:
        _need(uniforms, "uniforms", torch.float32, (B, R))
    dev = logits.device
    if workspace is None:
        workspace = new_workspace(sample_workspace_size(B, R, V), dev)
    if out is None:
        out = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
                   emitted=torch.empty((B, R), dtype=torch.int32, device=dev),
                   status=torch.empty(B, dtype=torch.int32, device=dev))
        if want_p:
            out["p"] = torch.empty((B, R, V), dtype=torch.float32, device=dev)
    c = cfg.c()
    rc = lib.spec_accept_sample(_ptr(logits), _ptr(draft_probs), _ptr(draft_tokens),
                                _ptr(uniforms), B, R, V, ctypes.byref(c), _ptr(workspace),
                                workspace.numel(), _ptr(out["accepted_len"]), _ptr(out["emitted"]),
                                _ptr(out.get("p")), _ptr(out["status"]), _stream(stream))
    _check("spec_accept_sample", rc)
    return out


def accept_sample_tree(logits, draft_probs, node_tokens, parent, uniforms, cfg: SamplerConfig,
                       workspace=None, want_p: bool = False, out=None, stream=None):
    """Draft-tree verification.  Returns dict(accepted_len, path, emitted, status[, p])."""
    lib = load()
    _need(logits, "target_logits", torch.float32)
    B, N, V = logits.shape
    if draft_probs is not None:
        _need(draft_probs, "draft_probs", torch.float32, (B, N, V))
    _need(node_tokens, "node_tokens", torch.int32, (B, N))
    _need(parent, "parent", torch.int32, (B, N))
    if uniforms is not None:
        _need(uniforms, "uniforms", torch.float32, (B, N))
    dev = logits.device
    if workspace is None:
        workspace = new_workspace(sample_workspace_size(B, N, V), dev)
    if out is None:
        out = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
                   path=torch.empty((B, N), dtype=torch.int32, device=dev),
                   emitted=torch.empty((B, N), dtype=torch.int32, device=dev),
                   status=torch.empty(B, dtype=torch.int32, device=dev))
        if want_p:
            out["p"] = torch.empty((B, N, V), dtype=torch.float32, device=dev)
    c = cfg.c()
    rc = lib.spec_accept_sample_tree(_ptr(logits), _ptr(draft_probs), _ptr(node_tokens),
                                     _ptr(parent), _ptr(uniforms), B, N, V, ctypes.byref(c),
                                     _ptr(workspace), workspace.numel(), _ptr(out["accepted_len"]),
                                     _ptr(out["path"]), _ptr(out["emitted"]), _ptr(out.get("p")),
                                     _ptr(out["status"]), _stream(stream))
    _check("spec_accept_sample_tree", rc)
    return out

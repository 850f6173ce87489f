"""Seeded synthetic inputs for the speculative-decoding verify step.

This module is the one place that makes inputs. The CUDA path and the CPU
oracle both consume what it returns; it computes none of the verify method's
results (no attention, no acceptance test, no target distribution).

What it does build is the *drafter side* that the verify step takes as given:
a synthetic draft distribution q (a noisy, optionally truncated softmax of the
target logits), the draft tokens drawn from that q, and the uniforms.  The
pages require that q be the distribution that actually produced each draft
("Speculative Decoding" (atlas), section "Greedy, sampling and the real
sampler"), so drafts are drawn here from exactly the q tensor that is handed
to the verifier.

Shapes follow the verify-step contract:
  q            [B, R, Hq, D]          bf16 (fp32 for the tiny config)
  k/v_cache    [num_pages, P, Hkv, D] bf16 (fp32 for the tiny config)
  block_table  [B, max_pages] int32   (-1 where unused)
  ctx_len      [B] int32              committed tokens before the block
  parent       [B, R] int32           -1 for node 0 (the pending anchor)
  logits       [B, R, V] fp32         target logits, row i scores after row i
  draft_probs  chain: [B, R-1, V]; tree: [B, R, V] (row v = q at node v)
  draft_tokens chain: [B, R-1];   tree: node_tokens [B, R] (node 0 unused)
  uniforms     [B, R] fp32 on the 2^-24 grid
"""
from __future__ import annotations

import dataclasses
from collections import deque
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Spec:
    """One synthetic verify-step workload."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    V: int
    ctx: tuple            # (lo, hi) inclusive; lo == hi for a fixed context
    gamma: int = 4        # chain draft length (R = gamma + 1)
    tree_nodes: int = 0   # > 0: draft tree with this many nodes (node 0 = anchor)
    tree_depth: int = 6
    tree_branch: int = 4
    kv_dtype: str = "bf16"
    page_size: int = 16
    shuffle_pages: bool = False
    logit_sd: float = 3.0
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    draft_div: float = 1.0      # q = softmax(logits / draft_div + N(0, draft_noise))
    draft_noise: float = 1.0
    greedy: bool = False
    seed: int = 0
    num_splits: int = 0         # 0 = let the library choose

    @property
    def is_tree(self) -> bool:
        return self.tree_nodes > 0

    @property
    def R(self) -> int:
        return self.tree_nodes if self.is_tree else self.gamma + 1

    def with_(self, **kw) -> "Spec":
        return dataclasses.replace(self, **kw)


# Drafter noise of the batched-serving pair, bisected on the oracle's mean
# sum_x min(p, q) over sample rows (tests/calibrate_draft_noise.py) so that one
# draft position is accepted with probability about 0.45 and about 0.75.
SIGMA_ALPHA_045 = 1.442
SIGMA_ALPHA_075 = 0.607

# The five workloads: a tiny fp32 chain, a Llama-3-8B-shaped chain, a draft
# tree, a batched serving mix and a long-context reasoning chain.
SPECS = {
    "tiny_chain": Spec("tiny_chain", B=1, Hq=1, Hkv=1, D=64, V=32, ctx=(128, 128),
                       gamma=4, kv_dtype="f32", logit_sd=2.0, temperature=1.0,
                       draft_div=1.0, draft_noise=0.5, seed=0),
    "llama8b_chain": Spec("llama8b_chain", B=1, Hq=32, Hkv=8, D=128, V=128256,
                          ctx=(8192, 8192), gamma=7, logit_sd=3.0, temperature=0.8,
                          draft_div=0.8, draft_noise=1.0, seed=1),
    "draft_tree": Spec("draft_tree", B=4, Hq=64, Hkv=8, D=128, V=128256,
                       ctx=(32768, 32768), tree_nodes=64, logit_sd=3.0,
                       temperature=0.7, top_k=50, draft_div=0.7, draft_noise=1.0,
                       seed=2),
    "batched_serving_a45": Spec("batched_serving_a45", B=64, Hq=32, Hkv=8, D=128,
                                V=152064, ctx=(512, 16384), gamma=4,
                                shuffle_pages=True, logit_sd=3.0, temperature=1.0,
                                top_p=0.9, draft_div=1.0,
                                draft_noise=SIGMA_ALPHA_045, seed=3),
    "batched_serving_a75": Spec("batched_serving_a75", B=64, Hq=32, Hkv=8, D=128,
                                V=152064, ctx=(512, 16384), gamma=4,
                                shuffle_pages=True, logit_sd=3.0, temperature=1.0,
                                top_p=0.9, draft_div=1.0,
                                draft_noise=SIGMA_ALPHA_075, seed=3),
    "long_context": Spec("long_context", B=1, Hq=64, Hkv=8, D=128, V=128256,
                         ctx=(131072, 131072), gamma=15, logit_sd=3.0,
                         temperature=0.6, draft_div=0.6, draft_noise=1.0, seed=4,
                         num_splits=128),
}


@dataclass
class Workload:
    spec: Spec
    q: torch.Tensor = None
    k_cache: torch.Tensor = None
    v_cache: torch.Tensor = None
    block_table: torch.Tensor = None
    ctx_len: torch.Tensor = None
    parent: torch.Tensor = None
    logits: torch.Tensor = None
    draft_probs: torch.Tensor = None
    draft_tokens: torch.Tensor = None
    uniforms: torch.Tensor = None
    extra: dict = field(default_factory=dict)

    def to(self, device) -> "Workload":
        out = Workload(self.spec, extra=dict(self.extra))
        for f in ("q", "k_cache", "v_cache", "block_table", "ctx_len", "parent",
                  "logits", "draft_probs", "draft_tokens", "uniforms"):
            t = getattr(self, f)
            setattr(out, f, None if t is None else t.to(device))
        return out


def random_tree(n_nodes: int, max_depth: int, max_branch: int, rng: np.random.Generator):
    """Parent array of a random tree in BFS storage order (parent[i] < i).

    Node 0 is the anchor.  Each expanded node below ``max_depth`` gets
    U{1..max_branch} children; if the breadth-first frontier runs dry before
    ``n_nodes`` nodes exist, extra children go to the shallowest nodes above
    ``max_depth``.
    """
    parent = [-1]
    depth = [0]
    frontier = deque([0])
    while len(parent) < n_nodes and frontier:
        v = frontier.popleft()
        if depth[v] >= max_depth:
            continue
        for _ in range(int(rng.integers(1, max_branch + 1))):
            if len(parent) == n_nodes:
                break
            parent.append(v)
            depth.append(depth[v] + 1)
            frontier.append(len(parent) - 1)
    v = 0
    while len(parent) < n_nodes:
        # rare: top up breadth-first under the depth limit
        if depth[v] < max_depth:
            parent.append(v)
            depth.append(depth[v] + 1)
        v = (v + 1) % len(parent)
    # re-sort into BFS order so that children of a node keep storage order
    order = sorted(range(n_nodes), key=lambda i: (depth[i], i))
    pos = {old: new for new, old in enumerate(order)}
    par = [-1 if parent[o] < 0 else pos[parent[o]] for o in order]
    return np.asarray(par, dtype=np.int32)


def _truncate(probs: torch.Tensor, top_k: int, top_p: float) -> torch.Tensor:
    """The drafter's own truncation of its proposal distribution (top-k, then top-p)."""
    V = probs.shape[-1]
    if top_k and 0 < top_k < V:
        kth = torch.topk(probs, top_k, dim=-1).values[..., -1:]
        probs = torch.where(probs >= kth, probs, torch.zeros_like(probs))
        probs = probs / probs.sum(-1, keepdim=True)
    if 0.0 < top_p < 1.0:
        sp, si = torch.sort(probs, dim=-1, descending=True)
        cum = torch.cumsum(sp, dim=-1)
        keep_sorted = (cum - sp) < top_p          # keep up to and including the crossing one
        keep = torch.zeros_like(keep_sorted).scatter(-1, si, keep_sorted)
        probs = torch.where(keep, probs, torch.zeros_like(probs))
        probs = probs / probs.sum(-1, keepdim=True)
    return probs


def _uniform_grid(shape, gen, device) -> torch.Tensor:
    """u in [0, 1) on the 2^-24 grid (exact in fp32 and fp64)."""
    return torch.randint(0, 1 << 24, shape, generator=gen, device=device,
                         dtype=torch.int64).to(torch.float32) * (1.0 / (1 << 24))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_ctx_lens(spec: Spec, seed: int) -> np.ndarray:
    lo, hi = spec.ctx
    rng = np.random.default_rng(seed * 7919 + 1)
    if lo == hi:
        return np.full(spec.B, lo, dtype=np.int32)
    return rng.integers(lo, hi + 1, size=spec.B).astype(np.int32)


def make_parent(spec: Spec, seed: int) -> np.ndarray:
    B, R = spec.B, spec.R
    if not spec.is_tree:
        row = np.arange(-1, R - 1, dtype=np.int32)
        return np.tile(row, (B, 1))
    rng = np.random.default_rng(seed * 104729 + 3)
    return np.stack([random_tree(R, spec.tree_depth, spec.tree_branch, rng) for _ in range(B)])


def make_attention_inputs(spec: Spec, seed: int | None = None, device="cpu",
                          ctx_lens: np.ndarray | None = None) -> Workload:
    """Q, paged K/V cache and block table for one verify step."""
    seed = spec.seed if seed is None else seed
    dev = torch.device(device)
    g = _gen(seed, dev)
    B, R, P = spec.B, spec.R, spec.page_size
    ctx = make_ctx_lens(spec, seed) if ctx_lens is None else np.asarray(ctx_lens, np.int32)
    kv_len = ctx + R
    pages_per = (kv_len + P - 1) // P
    total_pages = int(pages_per.sum())
    max_pages = int(pages_per.max())
    ids = np.arange(total_pages, dtype=np.int32)
    if spec.shuffle_pages:
        np.random.default_rng(seed * 31 + 5).shuffle(ids)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        n = int(pages_per[b])
        bt[b, :n] = ids[off:off + n]
        off += n
    dt = torch.float32 if spec.kv_dtype == "f32" else torch.bfloat16
    w = Workload(spec)
    w.q = torch.randn((B, R, spec.Hq, spec.D), generator=g, device=dev, dtype=torch.float32).to(dt)
    w.k_cache = torch.randn((total_pages, P, spec.Hkv, spec.D), generator=g, device=dev,
                            dtype=torch.float32).to(dt)
    w.v_cache = torch.randn((total_pages, P, spec.Hkv, spec.D), generator=g, device=dev,
                            dtype=torch.float32).to(dt)
    w.block_table = torch.from_numpy(bt).to(dev)
    w.ctx_len = torch.from_numpy(ctx).to(dev)
    w.parent = torch.from_numpy(make_parent(spec, seed)).to(dev)
    return w


def make_sampler_inputs(spec: Spec, seed: int | None = None, device="cpu",
                        w: Workload | None = None) -> Workload:
    """Target logits, the drafter's actual q, draft tokens drawn from q, uniforms."""
    seed = spec.seed if seed is None else seed
    dev = torch.device(device)
    g = _gen(seed + 1000003, dev)
    B, R, V = spec.B, spec.R, spec.V
    w = Workload(spec) if w is None else w
    if w.parent is None:
        w.parent = torch.from_numpy(make_parent(spec, seed)).to(dev)
    logits = torch.randn((B, R, V), generator=g, device=dev, dtype=torch.float32) * spec.logit_sd
    nq = R if spec.is_tree else R - 1
    noise = torch.randn((B, nq, V), generator=g, device=dev, dtype=torch.float32) * spec.draft_noise
    q = torch.softmax(logits[:, :nq].double() / spec.draft_div + noise.double(), dim=-1)
    q = _truncate(q, spec.top_k, spec.top_p).to(torch.float32)
    # make every row sum to one in fp32 as served; drafts are drawn from this tensor
    q = q / q.sum(-1, keepdim=True)
    if spec.is_tree:
        par = w.parent.to(dev).long()
        src = par.clamp_min(0)                                   # node 0 has no proposal
        rows = torch.gather(q, 1, src[..., None].expand(B, R, V))
        tok = torch.multinomial(rows.reshape(-1, V), 1, generator=g).view(B, R)
        tok[:, 0] = -1
    else:
        tok = torch.multinomial(q.reshape(-1, V), 1, generator=g).view(B, nq)
    w.logits = logits
    w.draft_probs = q
    w.draft_tokens = tok.to(torch.int32)
    w.uniforms = _uniform_grid((B, R), g, dev)
    return w


def make_workload(spec: Spec, seed: int | None = None, device="cpu",
                  attention=True, sampler=True) -> Workload:
    w = make_attention_inputs(spec, seed, device) if attention else Workload(spec)
    if sampler:
        make_sampler_inputs(spec, seed, device, w)
    return w


def algorithmic_bytes(spec: Spec, ctx_lens: np.ndarray) -> dict:
    """Bytes the verify step must move at least once (see the design notes).

    attention: K and V of every visible position once, Q in, output out.
    sampler: every target-logit row once (all rows are needed when every draft
    survives), one draft-distribution row per sequence (a residual reads one
    row of q at most), and the small per-row vectors.
    step_all_q: the same step counting every draft-distribution row once
    (B * gamma * V * 4 for a chain, B * N * V * 4 for a tree) instead of one row
    per sequence -- the larger convention, which lowers the fraction.
    """
    el = 4 if spec.kv_dtype == "f32" else 2
    R = spec.R
    kv = int(np.sum(ctx_lens.astype(np.int64) + R)) * spec.Hkv * spec.D * el * 2
    qo = spec.B * R * spec.Hq * spec.D * el * 2
    logits = spec.B * R * spec.V * 4
    small = spec.B * R * 4 * 3
    qrow = spec.B * spec.V * 4 + small
    nq = R if spec.is_tree else R - 1
    qall = spec.B * nq * spec.V * 4 + small
    return {"attn": kv + qo, "kv": kv, "sampler": logits + qrow,
            "step": kv + qo + logits + qrow, "step_all_q": kv + qo + logits + qall}

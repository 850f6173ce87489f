"""Test plumbing: run the CUDA path and the oracle on the same seeded inputs."""
import numpy as np
import torch

import oracle
from oracle.sampler import SamplerCfg
from speculative_decoding_verification_76_gb300 import workloads as wl

BF16_ATOL = 2e-2     # attention, bf16 inputs, fp32 accumulation (stated tolerance)
F32_ATOL = 1e-5      # attention, fp32 tiny configuration (stated tolerance)
P_RTOL = 1e-6        # target distribution p, relative (stated tolerance)

# (test, flagged sequences, sequences, flagged sequences whose GPU outcome differs)
# of every sampler comparison in this session; printed at the end of the run by
# the conftest summary hook
FLAG_LOG = []


def record_flags(label: str, flagged: int, total: int, flagged_diff: int = 0):
    FLAG_LOG.append((label, int(flagged), int(total), int(flagged_diff)))


def np_u64(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint64)


def sub_sequence(w: wl.Workload, b: int):
    """One sequence as a self-contained problem: its pages only (numpy, fp64-ready)."""
    P = w.k_cache.shape[1]
    ctx = int(w.ctx_len[b])
    R = w.q.shape[1]
    npg = (ctx + R + P - 1) // P
    pages = w.block_table[b, :npg].long().cpu()
    k = w.k_cache.index_select(0, pages.to(w.k_cache.device)).float().cpu().numpy()
    v = w.v_cache.index_select(0, pages.to(w.v_cache.device)).float().cpu().numpy()
    q = w.q[b:b + 1].float().cpu().numpy()
    table = np.arange(npg)[None]
    return q, k, v, table, np.array([ctx])


def oracle_attention(w: wl.Workload, anc_mask: np.ndarray, batches=None, rows=None, heads=None,
                     scale=None):
    """Oracle output for selected sequences, computed one sequence at a time."""
    B, R, Hq, D = w.q.shape
    out = np.zeros((B, R, Hq, D))
    lse = np.zeros((B, R, Hq))
    for b in (range(B) if batches is None else batches):
        q, k, v, table, ctx = sub_sequence(w, b)
        o, l = oracle.attention.verify_attention(q, k, v, table, ctx, anc_mask[b:b + 1],
                                                 scale=scale, rows=rows, heads=heads)
        out[b] = o[0]
        lse[b] = l[0]
    return out, lse


def cfg_of(spec: wl.Spec, greedy=None, eos=-1) -> SamplerCfg:
    return SamplerCfg(temperature=spec.temperature, top_k=spec.top_k, top_p=spec.top_p,
                      greedy=spec.greedy if greedy is None else greedy, eos_id=eos)


def to_np(t):
    return None if t is None else t.detach().cpu().numpy()

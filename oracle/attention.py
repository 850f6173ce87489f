"""Oracle: multi-row verify attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it computes.  One target pass scores every row of the proposed block at
once, each row under its own mask ("Drafters and Speculative Decoding",
section "From a proposed block to a causal target pass"; "Speculative
Decoding" (atlas), "Turn guesses into parallel work": scoring a known block
resembles a small prefill under a causal mask).  For a draft tree a row sees
the accepted prefix, its ancestors and itself ("Speculative Decoding"
(atlas), "Chains, trees and visibility").  The dispatch "Speculative Token
Decoupling: Asynchronous Verification via Flash-Decoding" (section 03) runs
this with a split-K attention kernel; split-K with a log-sum-exp combine
reaches the plain full-softmax result up to rounding, so the oracle is that
plain result, with no split.

Readings (the pages are silent on these):
  * scale = 1/sqrt(D) unless given;
  * every committed context position [0, ctx_len) is visible to every row;
    block row j sits at cache position ctx_len + j;
  * grouped-query attention maps query head h to KV head h // (Hq / Hkv);
  * lse is the natural-log log-sum-exp of the scaled scores of the row.
"""
import math

import numpy as np


def gather_kv(cache, block_table_row, n_tokens: int):
    """Rows 0..n_tokens-1 of one sequence, read page by page: [n, Hkv, D]."""
    P = cache.shape[1]
    rows = []
    for t in range(n_tokens):
        page = int(block_table_row[t // P])
        rows.append(cache[page, t % P])
    return np.stack(rows) if rows else np.zeros((0,) + cache.shape[2:])


def visible_positions(ctx: int, mask_word) -> np.ndarray:
    """Cache positions one block row may attend to."""
    m = int(mask_word)
    block = [ctx + j for j in range(64) if (m >> j) & 1]
    return np.asarray(list(range(ctx)) + block, dtype=np.int64)


def verify_attention(q, k_cache, v_cache, block_table, ctx_len, anc_mask, scale=None,
                     batches=None, rows=None, heads=None):
    """Full-softmax attention of every (sequence, block row, query head).

    q [B,R,Hq,D]; k_cache, v_cache [pages, P, Hkv, D]; block_table [B, maxp];
    ctx_len [B]; anc_mask [B,R] (uint64 words).  Inputs are the values the GPU
    reads (bf16 inputs already widened); arithmetic is float64.
    Returns out [B,R,Hq,D] and lse [B,R,Hq].  batches / rows / heads restrict
    which outputs are computed (the others stay zero); the arithmetic of each
    computed output is unchanged.

    Row i's visible keys are the committed prefix [0, ctx) and the block
    positions ctx + j with bit j of its mask; the scores, the softmax and the
    weighted sum run over exactly that set (the query heads that share a KV
    head are scored together, one column each).
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    B, R, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, R, Hq, D))
    lse = np.zeros((B, R, Hq))
    hs = list(range(Hq) if heads is None else heads)
    for b in (range(B) if batches is None else batches):
        ctx = int(ctx_len[b])
        K = gather_kv(k_cache, block_table[b], ctx + R)
        Vv = gather_kv(v_cache, block_table[b], ctx + R)
        for i in (range(R) if rows is None else rows):
            vis = visible_positions(ctx, anc_mask[b][i])
            blk = vis[vis >= ctx]                      # the visible block positions
            for kvh in sorted({h // G for h in hs}):
                group = [h for h in hs if h // G == kvh]
                Qg = q[b, i, group, :]                 # [g, D]
                Kc, Vc = K[:ctx, kvh, :], Vv[:ctx, kvh, :]
                Kb, Vb = K[blk, kvh, :], Vv[blk, kvh, :]
                s = np.concatenate([Kc @ Qg.T, Kb @ Qg.T]) * scale   # [n_visible, g]
                smax = s.max(axis=0)
                e = np.exp(s - smax)
                z = e.sum(axis=0)
                o = e[:ctx].T @ Vc + e[ctx:].T @ Vb   # sum over the visible set
                out[b, i, group] = o / z[:, None]
                lse[b, i, group] = smax + np.log(z)
    return out, lse

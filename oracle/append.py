"""Oracle: rotary position at depth and the block's K/V append (next row f3).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it computes.  Before the verify attention, the target writes the K/V rows
of the proposed block into the paged cache: row j at position ctx_len + j (the
layout the verify attention reads).  Keys carry their position: "Speculative
Decoding" (atlas), "Chains, trees and visibility" -- position ids follow
depth, not flattened storage order -- so node j's key is rotated for position
ctx_len + depth(j) while it is stored at slot ctx_len + j.

Readings (the pages do not print the rotation):
  * the rotary embedding is the common split-half form: for pair index
    i < D/2, theta_i = base^(-2 i / D), the pair (x_i, x_{i + D/2}) at
    position t is rotated by the angle t * theta_i;
  * the same rotation applies to the block's queries (not stored);
  * values are stored unrotated.
"""
import numpy as np


def rope(x, pos, base: float = 10000.0):
    """x [..., D] rotated for integer positions pos (broadcast over x[..., 0])."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    if D % 2:
        raise ValueError("head_dim must be even")
    half = D // 2
    theta = base ** (-2.0 * np.arange(half) / D)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    if a.ndim > ang.ndim:  # heads between the position axes and D
        c = c[..., None, :]
        s = s[..., None, :]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def append_block(k_cache, v_cache, block_table, ctx_len, k_new, v_new, pos_ids, page_size: int,
                 base: float = 10000.0):
    """Copies of the caches with the block written in.

    k_new, v_new [B, R, Hkv, D] (keys before rotation); pos_ids [B, R] (ctx_len
    + depth).  Row j of sequence b goes to position ctx_len[b] + j; the key is
    rotated for pos_ids[b, j]."""
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    B, R = np.asarray(pos_ids).shape
    for b in range(B):
        for j in range(R):
            pos = int(ctx_len[b]) + j
            page, off = block_table[b][pos // page_size], pos % page_size
            kc[page, off] = rope(np.asarray(k_new)[b, j], int(pos_ids[b][j]), base)
            vc[page, off] = np.asarray(v_new)[b, j]
    return kc, vc

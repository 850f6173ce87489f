"""Oracle: visibility of a flattened draft tree.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "Speculative Decoding" (atlas), section "Chains, trees and
visibility": each flattened node may see the shared accepted prefix, its
ancestors and itself; position ids follow depth, not storage order; a parent
array plus an ancestor mask make this explicit.  A chain is the tree whose
node i has parent i - 1, and then the mask is the ordinary causal triangle
("Drafters and Speculative Decoding", "From a proposed block to a causal
target pass": each verification row sees only its own prefix).
"""
import numpy as np


def chain_parent(B: int, R: int) -> np.ndarray:
    return np.tile(np.arange(-1, R - 1, dtype=np.int64), (B, 1))


def ancestors(parent_row, i: int) -> list:
    """Node i and every node on the path from i up to the root."""
    out = []
    v = i
    while v >= 0:
        out.append(v)
        v = int(parent_row[v])
    return out


def tree_prepare(parent, ctx_len):
    """Return (anc_mask uint64 [B,R], depth int64 [B,R], pos int64 [B,R]).

    Bit j of anc_mask[b, i] is set iff node j is node i or one of its
    ancestors.  depth is the number of edges from node i to the root (the
    anchor has depth 0) and pos = ctx_len[b] + depth.
    """
    parent = np.asarray(parent, dtype=np.int64)
    ctx_len = np.asarray(ctx_len, dtype=np.int64)
    B, R = parent.shape
    if R > 64:
        raise ValueError("at most 64 nodes fit a 64-bit ancestor mask")
    mask = np.zeros((B, R), dtype=np.uint64)
    depth = np.zeros((B, R), dtype=np.int64)
    for b in range(B):
        for i in range(R):
            anc = ancestors(parent[b], i)
            m = 0
            for j in anc:
                m |= 1 << j
            mask[b, i] = np.uint64(m)
            depth[b, i] = len(anc) - 1
    pos = ctx_len[:, None] + depth
    return mask, depth, pos


def visible_block_nodes(mask_word) -> list:
    """Indices j with bit j set in one node's ancestor mask."""
    m = int(mask_word)
    return [j for j in range(64) if (m >> j) & 1]

"""Oracle: keeping the verified states after acceptance (KV commit).

TEST INFRASTRUCTURE ONLY (see the package docstring).

What it computes.  "Speculative Decoding" (atlas), section "Committed tokens
versus cached states": a sequence's committed tokens and its processed KV
length differ; verification writes states for the whole proposed block, the
states of accepted proposals are kept and the rejected suffix is removed; the
correction (or bonus) token is committed but its KV only comes with the next
pass.  Section "Chains, trees and visibility": after a tree's path is chosen,
its KV entries are compacted into the next logical prefix so that branch
states are no longer addressable ("Tree KV needs path compaction, not merely a
suffix length change").

Readings (the pages leave these open):
  * block row j (tree node j) was written at cache position ctx_len + j, as in
    the verify attention; row 0 is the pending anchor of the previous step,
    whose state this pass created, so it is kept with the accepted drafts;
  * after accepting a drafts the processed length is ctx_len + 1 + a and the
    correction / bonus token is the next pending anchor;
  * a tree's accepted path is node 0 followed by the accepted nodes in order;
    path node k moves to position ctx_len + k (its depth), so its position id
    from tree_prepare does not change;
  * positions at or beyond the new length are invalid; a page of the block
    table holding no valid position any more is released (its slot reported).
"""
import numpy as np


def committed_length(ctx_len, accepted_len):
    """New processed KV length per sequence: the context, the anchor, the accepted drafts."""
    ctx_len = np.asarray(ctx_len, dtype=np.int64)
    accepted_len = np.asarray(accepted_len, dtype=np.int64)
    if (accepted_len < 0).any():
        raise ValueError("accepted_len must be >= 0")
    return ctx_len + 1 + accepted_len


def released_slots(ctx_len, R: int, new_len, page_size: int):
    """Block-table slots, per sequence, whose pages the block touched and that
    hold no position below the new length any more (ascending)."""
    out = []
    for c, n in zip(np.asarray(ctx_len, dtype=np.int64), np.asarray(new_len, dtype=np.int64)):
        first = int(c) // page_size                 # first page the block wrote
        last = (int(c) + R - 1) // page_size        # last page the block wrote
        keep = (int(n) - 1) // page_size            # last page with a valid position
        out.append([s for s in range(first, last + 1) if s > keep])
    return out


def compact_path(cache, block_table, ctx_len, paths, page_size: int):
    """Copy of cache ([pages, page_size, Hkv, D]) with, for every sequence b and
    path index k, the row of node paths[b][k] (position ctx_len[b] + node)
    written at position ctx_len[b] + k.  All rows are read before any is
    written.  Rows outside the new prefix are left as they were."""
    out = np.array(cache, copy=True)
    src = np.asarray(cache)
    for b, path in enumerate(paths):
        c = int(ctx_len[b])
        rows = []
        for node in path:
            pos = c + int(node)
            rows.append(src[block_table[b][pos // page_size], pos % page_size].copy())
        for k, row in enumerate(rows):
            pos = c + k
            out[block_table[b][pos // page_size], pos % page_size] = row
    return out


def accepted_path(parent_row, node: int):
    """The path from node 0 (the anchor) down to node, as node ids."""
    path = []
    v = int(node)
    while v >= 0:
        path.append(v)
        v = int(parent_row[v])
    return path[::-1]

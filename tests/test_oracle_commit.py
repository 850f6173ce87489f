"""Pins for the oracle's KV commit and tree path compaction (CPU only)."""
import numpy as np
import pytest

from oracle import commit, tree as otree
from tests.conftest import load_golden


def test_committed_length_keeps_anchor_and_accepted_drafts():
    # every draft accepted: the whole block stays (ctx + R); none: the anchor only
    R = 8
    assert list(commit.committed_length([100, 7], [R - 1, 0])) == [100 + R, 8]
    with pytest.raises(ValueError):
        commit.committed_length([5], [-1])


def _released_brute(c, R, n, P):
    pages = sorted({pos // P for pos in range(c, c + R)})
    return [s for s in pages if all(pos >= n for pos in range(s * P, (s + 1) * P))]


def test_released_slots_hand_cases_and_brute_force():
    # positions 100..107 on page 6 (96..111): keeping 103 leaves the page in use
    assert commit.released_slots([100], 8, [103], 16) == [[]]
    # positions 110..117 cover pages 6 and 7; keeping 111 frees page 7 only
    assert commit.released_slots([110], 8, [111], 16) == [[7]]
    rng = np.random.default_rng(0)
    for _ in range(300):
        P = int(rng.choice([1, 4, 16]))
        c = int(rng.integers(0, 200))
        R = int(rng.integers(1, 65))
        a = int(rng.integers(0, R))
        n = int(commit.committed_length([c], [a])[0])
        assert commit.released_slots([c], R, [n], P) == [_released_brute(c, R, n, P)]


def _paged_cache(ctx, R, P, seed):
    """A cache whose row at position pos of sequence 0 holds the value pos in every
    entry, pages of the sequence scattered through a shuffled block table."""
    npos = ctx + R
    npages = (npos + P - 1) // P
    rng = np.random.default_rng(seed)
    table = rng.permutation(npages + 3)[:npages]
    cache = np.full((npages + 3, P, 2, 4), -1.0)
    for pos in range(npos):
        cache[table[pos // P], pos % P] = pos
    return cache, [list(table)]


def _row(cache, table, pos, P):
    return cache[table[0][pos // P], pos % P]


def test_chain_path_compaction_is_the_identity():
    # a chain keeps its accepted rows where they are: a length change is enough
    cache, table = _paged_cache(37, 8, 16, 1)
    for a in range(8):
        out = commit.compact_path(cache, table, [37], [list(range(a + 1))], 16)
        np.testing.assert_array_equal(out, cache)


def test_fox_tree_path_to_away():
    g = load_golden("fox_tree.json")
    names = g["flattened"]["nodes"]
    parent = np.array([g["flattened"]["parent"]])
    path = commit.accepted_path(parent[0], names.index("away"))
    assert [names[v] for v in path] == ["fox", "runs", "away"]
    assert commit.accepted_path(parent[0], names.index("over")) == [0, 1, 2]
    assert commit.accepted_path(parent[0], 0) == [0]
    ctx, P = 14, 16  # the block straddles a page boundary
    cache, table = _paged_cache(ctx, len(names), P, 2)
    out = commit.compact_path(cache, table, [ctx], [path], P)
    # path node k now sits at position ctx + k, which is its tree_prepare position
    _, depth, pos = otree.tree_prepare(parent, [ctx])
    for k, v in enumerate(path):
        assert depth[0, v] == k and pos[0, v] == ctx + k
        np.testing.assert_array_equal(_row(out, table, ctx + k, P), ctx + v)
    # no branch state is addressable inside the new prefix
    new_len = int(commit.committed_length([ctx], [len(path) - 1])[0])
    branch = {ctx + v for v in range(len(names)) if v not in path}
    for p_ in range(ctx, new_len):
        assert float(_row(out, table, p_, P)[0, 0]) not in branch
    # the context before the block is untouched
    for p_ in range(ctx):
        np.testing.assert_array_equal(_row(out, table, p_, P), p_)


def test_overlapping_moves_read_before_write():
    # path 0 -> 2 -> 3: node 2 moves to slot 1 while node 3 moves into node 2's slot
    cache, table = _paged_cache(5, 6, 4, 3)
    out = commit.compact_path(cache, table, [5], [[0, 2, 3]], 4)
    assert [float(_row(out, table, 5 + k, 4)[0, 0]) for k in range(3)] == [5.0, 7.0, 8.0]

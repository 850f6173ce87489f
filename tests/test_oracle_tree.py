"""Pins for the oracle's tree visibility (CPU only)."""
import numpy as np
import pytest

from oracle import tree as otree
from tests.conftest import load_golden


def test_fox_tree_masks_and_positions():
    g = load_golden("fox_tree.json")
    parent = np.array([g["flattened"]["parent"]])
    mask, depth, pos = otree.tree_prepare(parent, [100])
    assert [int(m) for m in mask[0]] == g["expected"]["anc_mask"]
    assert list(depth[0]) == g["expected"]["depth"]
    assert list(pos[0]) == [100 + d for d in g["expected"]["depth"]]
    names = g["flattened"]["nodes"]
    over = names.index("over")
    seen = {names[j] for j in otree.visible_block_nodes(mask[0, over])}
    assert set(g["printed"]["over_may_see"]) <= seen
    assert not (set(g["printed"]["over_must_not_see"]) & seen)


def test_chain_is_causal_triangle():
    g = load_golden("chain_bird.json")
    R = 5
    mask, depth, pos = otree.tree_prepare(otree.chain_parent(2, R), [7, 0])
    assert [int(m) for m in mask[0]] == g["expected"]["causal_mask_rows"]
    assert [int(m) for m in mask[0]] == [(1 << (i + 1)) - 1 for i in range(R)]
    assert list(pos[0]) == [7, 8, 9, 10, 11]
    assert list(pos[1]) == [0, 1, 2, 3, 4]


def test_triangular_mask_leaks_siblings():
    # the page warns that a triangular mask on flattened nodes leaks siblings:
    # for the fox tree the two masks must differ exactly on sibling/cousin bits
    parent = np.array([[-1, 0, 1, 1, 0, 4]])
    mask, _, _ = otree.tree_prepare(parent, [0])
    tri = [(1 << (i + 1)) - 1 for i in range(6)]
    assert int(mask[0, 3]) != tri[3]          # "high" must not see "over"
    assert not (int(mask[0, 3]) >> 2) & 1


def test_64_nodes_full_mask_bit63():
    parent = np.array([np.arange(-1, 63)])
    mask, depth, _ = otree.tree_prepare(parent, [0])
    assert int(mask[0, 63]) == (1 << 64) - 1
    assert depth[0, 63] == 63


def test_more_than_64_nodes_rejected():
    with pytest.raises(ValueError):
        otree.tree_prepare(np.array([np.arange(-1, 64)]), [0])

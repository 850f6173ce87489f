"""Pins for the oracle's rotary position at depth and block K/V append (CPU only)."""
import numpy as np
import pytest

from oracle import append, tree as otree
from tests.conftest import load_golden


def test_rope_closed_forms():
    t = 0.7
    # D = 2: a plain planar rotation by t (theta_0 = 1)
    np.testing.assert_allclose(append.rope([1.0, 0.0], t), [np.cos(t), np.sin(t)], atol=1e-15)
    # D = 4, base 10000: pairs (x0, x2) at theta 1 and (x1, x3) at theta 0.01
    np.testing.assert_allclose(append.rope([1.0, 0.0, 0.0, 0.0], t),
                               [np.cos(t), 0.0, np.sin(t), 0.0], atol=1e-15)
    np.testing.assert_allclose(append.rope([0.0, 1.0, 0.0, 0.0], t),
                               [0.0, np.cos(0.01 * t), 0.0, np.sin(0.01 * t)], atol=1e-15)
    with pytest.raises(ValueError):
        append.rope([1.0, 2.0, 3.0], 1)


def test_rope_invariants():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 64))
    pos = rng.integers(0, 5000, 5)
    y = append.rope(x, pos)
    # position 0 is the identity; norms are kept; rotations compose
    np.testing.assert_allclose(append.rope(x, np.zeros(5)), x, atol=0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    np.testing.assert_allclose(append.rope(y, pos + 3), append.rope(x, 2 * pos + 3), atol=1e-9)
    # a query-key score depends only on the position difference
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n in ((10, 3), (1000, 997), (7, 7)):
        s0 = append.rope(q, m) @ append.rope(k, n)
        for shift in (1, 50, 4096):
            np.testing.assert_allclose(append.rope(q, m + shift) @ append.rope(k, n + shift), s0,
                                       rtol=1e-9, atol=1e-9)


def test_append_fox_tree_rotates_at_depth_and_stores_in_slot_order():
    g = load_golden("fox_tree.json")
    parent = np.array([g["flattened"]["parent"]])
    R = parent.shape[1]
    ctx, P, Hkv, D = 14, 16, 2, 8  # the block straddles a page boundary
    _, depth, pos = otree.tree_prepare(parent, [ctx])
    rng = np.random.default_rng(1)
    npages = 4
    table = [[2, 0, 3]]
    kc = rng.standard_normal((npages, P, Hkv, D))
    vc = rng.standard_normal((npages, P, Hkv, D))
    k_new = rng.standard_normal((1, R, Hkv, D))
    v_new = rng.standard_normal((1, R, Hkv, D))
    ko, vo = append.append_block(kc, vc, table, [ctx], k_new, v_new, pos, P)
    for j in range(R):
        p_ = ctx + j
        slot = (table[0][p_ // P], p_ % P)
        np.testing.assert_allclose(ko[slot], append.rope(k_new[0, j], ctx + depth[0, j]),
                                   atol=1e-15)
        np.testing.assert_array_equal(vo[slot], v_new[0, j])
    # "away" (depth 2, slot 5) is rotated like a chain node two steps past the anchor
    np.testing.assert_allclose(ko[table[0][(ctx + 5) // P], (ctx + 5) % P],
                               append.rope(k_new[0, 5], ctx + 2), atol=1e-15)
    # positions before the block are untouched
    for p_ in range(ctx):
        np.testing.assert_array_equal(ko[table[0][p_ // P], p_ % P], kc[table[0][p_ // P], p_ % P])

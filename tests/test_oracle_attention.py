"""Pins for the oracle's verify attention (CPU only)."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oat
from oracle import tree as otree
from tests.conftest import load_golden


def _paged(contig, P, rng, shuffle=True):
    """Scatter a contiguous [B, T, Hkv, D] cache into pages; return cache, table."""
    B, T = contig.shape[:2]
    npg = (T + P - 1) // P
    ids = np.arange(B * npg)
    if shuffle:
        rng.shuffle(ids)
    cache = np.full((B * npg, P) + contig.shape[2:], np.nan)
    table = ids.reshape(B, npg)
    for b in range(B):
        for t in range(T):
            cache[table[b, t // P], t % P] = contig[b, t]
    return cache, table


def _brute(q, Kc, Vc, ctx, parent, scale):
    """Pure-Python loops; visibility by walking parent links (no masks)."""
    B, R, Hq, D = q.shape
    Hkv = Kc.shape[2]
    out = np.zeros_like(q)
    for b in range(B):
        for i in range(R):
            nodes = []
            v = i
            while v >= 0:
                nodes.append(v)
                v = parent[b][v]
            keys = list(range(ctx[b])) + [ctx[b] + j for j in sorted(nodes)]
            for h in range(Hq):
                kh = h // (Hq // Hkv)
                s = [sum(q[b, i, h, d] * Kc[b, t, kh, d] for d in range(D)) * scale for t in keys]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                z = sum(e)
                for d in range(D):
                    out[b, i, h, d] = sum(e[k] * Vc[b, t, kh, d] for k, t in enumerate(keys)) / z
    return out


@pytest.mark.parametrize("tree", [False, True])
def test_matches_bruteforce_paged_gqa(tree):
    rng = np.random.default_rng(10 + tree)
    B, R, Hq, Hkv, D, P = 2, 6, 4, 2, 8, 4
    ctx = np.array([5, 11])
    parent = ([[-1, 0, 1, 1, 0, 4]] * B) if tree else otree.chain_parent(B, R).tolist()
    T = int(ctx.max()) + R
    Kc = rng.normal(size=(B, T, Hkv, D))
    Vc = rng.normal(size=(B, T, Hkv, D))
    q = rng.normal(size=(B, R, Hq, D))
    kcache, table = _paged(Kc, P, rng)
    vcache = np.full_like(kcache, np.nan)
    for b in range(B):
        for t in range(T):
            vcache[table[b, t // P], t % P] = Vc[b, t]
    mask, _, _ = otree.tree_prepare(np.array(parent), ctx)
    out, lse = oat.verify_attention(q, kcache, vcache, table, ctx, mask, scale=0.3)
    ref = _brute(q, Kc, Vc, ctx, parent, 0.3)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    assert np.all(np.isfinite(lse))


def test_sdpa_chain_special_case():
    """A chain with a contiguous cache is textbook masked attention."""
    rng = np.random.default_rng(3)
    R, H, D, ctx = 5, 2, 16, 9
    T = ctx + R
    K = rng.normal(size=(1, T, H, D))
    V = rng.normal(size=(1, T, H, D))
    q = rng.normal(size=(1, R, H, D))
    table = np.arange(T)[None, :]                       # page size 1, identity
    mask, _, _ = otree.tree_prepare(otree.chain_parent(1, R), [ctx])
    out, _ = oat.verify_attention(q, K.reshape(T, 1, H, D), V.reshape(T, 1, H, D), table, [ctx],
                                  mask)
    allowed = torch.zeros(R, T, dtype=torch.bool)
    for i in range(R):
        allowed[i, :ctx + i + 1] = True
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q[0]).permute(1, 0, 2), torch.from_numpy(K[0]).permute(1, 0, 2),
        torch.from_numpy(V[0]).permute(1, 0, 2), attn_mask=allowed)
    np.testing.assert_allclose(out[0], ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(4)
    D = 8
    K = rng.normal(size=(1, 1, 1, D))
    V = rng.normal(size=(1, 1, 1, D))
    q = rng.normal(size=(1, 1, 1, D))
    out, lse = oat.verify_attention(q, K, V, np.array([[0]]), [0], np.array([[1]], np.uint64))
    np.testing.assert_array_equal(out[0, 0, 0], V[0, 0, 0])
    assert lse[0, 0, 0] == pytest.approx(float(q[0, 0, 0] @ K[0, 0, 0]) / math.sqrt(D))


def test_zero_query_is_mean_of_visible_values_and_lse_is_log_count():
    rng = np.random.default_rng(5)
    ctx, R, D, P = 7, 3, 4, 2
    T = ctx + R
    K = rng.normal(size=(T, 1, D))
    V = rng.normal(size=(T, 1, D))
    kc, table = _paged(K[None], P, rng)
    vc = np.full_like(kc, np.nan)
    for t in range(T):
        vc[table[0, t // P], t % P] = V[t]
    q = np.zeros((1, R, 1, D))
    mask, _, _ = otree.tree_prepare(otree.chain_parent(1, R), [ctx])
    out, lse = oat.verify_attention(q, kc, vc, table, [ctx], mask)
    for i in range(R):
        n = ctx + i + 1
        np.testing.assert_allclose(out[0, i, 0], V[:n, 0].mean(0), rtol=1e-12)
        assert lse[0, i, 0] == pytest.approx(math.log(n))


def test_fox_tree_hidden_nodes_do_not_matter():
    g = load_golden("fox_tree.json")
    parent = np.array([g["flattened"]["parent"]])
    names = g["flattened"]["nodes"]
    rng = np.random.default_rng(6)
    ctx, R, D = 4, 6, 8
    T = ctx + R
    K = rng.normal(size=(T, 1, 1, D))
    V = rng.normal(size=(T, 1, 1, D))
    q = rng.normal(size=(1, R, 1, D))
    mask, _, _ = otree.tree_prepare(parent, [ctx])
    table = np.arange(T)[None]
    out1, _ = oat.verify_attention(q, K, V, table, [ctx], mask)
    K2, V2 = K.copy(), V.copy()
    for nm in g["printed"]["over_must_not_see"]:
        K2[ctx + names.index(nm)] += 5.0
        V2[ctx + names.index(nm)] -= 3.0
    out2, _ = oat.verify_attention(q, K2, V2, table, [ctx], mask)
    over = names.index("over")
    np.testing.assert_array_equal(out1[0, over], out2[0, over])
    # ...while a node that does see 'runs' changes
    assert not np.allclose(out1[0, names.index("away")], out2[0, names.index("away")])
    # and a visible ancestor does change 'over'
    K3 = K.copy()
    K3[ctx + names.index("jumps")] += 5.0
    out3, _ = oat.verify_attention(q, K3, V, table, [ctx], mask)
    assert not np.allclose(out1[0, over], out3[0, over])


def test_page_order_is_irrelevant():
    rng = np.random.default_rng(8)
    B, R, H, D, P = 2, 4, 2, 8, 4
    ctx = np.array([13, 6])
    T = int(ctx.max()) + R
    K = rng.normal(size=(B, T, H, D))
    V = rng.normal(size=(B, T, H, D))
    q = rng.normal(size=(B, R, H, D))
    mask, _, _ = otree.tree_prepare(otree.chain_parent(B, R), ctx)
    res = []
    for shuffle in (False, True):
        r2 = np.random.default_rng(1)
        kc, table = _paged(K, P, r2, shuffle)
        r2 = np.random.default_rng(1)
        vc, _ = _paged(V, P, r2, shuffle)
        res.append(oat.verify_attention(q, kc, vc, table, ctx, mask)[0])
    np.testing.assert_array_equal(res[0], res[1])

"""GPU parity: KV commit after acceptance (processed lengths, tree path compaction)
against the oracle.  A copy: the caches must match bit for bit.

The path argument is the tree sampler's own output (the accepted nodes, node 0
implied); the oracle's compact_path takes the full root-to-node path, so the
tests prepend node 0 for it."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_76_gb300 as sv
from oracle import commit
from speculative_decoding_verification_76_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(B, R, Hkv, D, P, dtype, seed, tree):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(0, 40, B).astype(np.int32)
    max_pages = int((ctx.max() + R + P - 1) // P) + 1
    npages = B * max_pages + 3
    table = rng.permutation(npages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    k = torch.from_numpy(rng.standard_normal((npages, P, Hkv, D)).astype(np.float32)).to(dtype)
    v = torch.from_numpy(rng.standard_normal((npages, P, Hkv, D)).astype(np.float32)).to(dtype)
    paths, path, parent = None, None, None
    if tree:
        parent = np.full((B, R), -1, np.int32)
        paths = []
        path = np.full((B, R), -1, np.int32)
        acc = np.zeros(B, np.int32)
        for b in range(B):
            for i in range(1, R):
                parent[b, i] = rng.integers(0, i)
            pth = commit.accepted_path(parent[b], int(rng.integers(0, R)))
            paths.append(pth)
            path[b, :len(pth) - 1] = pth[1:]          # the sampler's form: node 0 implied
            acc[b] = len(pth) - 1
    else:
        acc = rng.integers(0, R, B).astype(np.int32)
    return ctx, table, k, v, acc, paths, path, parent


def _run(ctx, table, k, v, acc, path, R, parent=None):
    t = lambda a: None if a is None else torch.as_tensor(a).to(DEV).contiguous()  # noqa: E731
    kd, vd = k.to(DEV).contiguous(), v.to(DEV).contiguous()
    new_len, keep, status = sv.kv_commit(kd, vd, t(table), t(ctx), t(acc), t(path), t(parent),
                                         R=R)
    torch.cuda.synchronize()
    return kd.cpu(), vd.cpu(), new_len.cpu().numpy(), keep.cpu().numpy(), status.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D,P", [(128, 16), (64, 4)])
@pytest.mark.parametrize("with_parent", [False, True])
def test_tree_path_compaction_matches_oracle(dtype, D, P, with_parent):
    for seed in range(3):
        B, R, Hkv = 5, 16 if seed < 2 else 64, 2
        ctx, table, k, v, acc, paths, path, parent = _case(B, R, Hkv, D, P, dtype, seed, True)
        ko, vo, new_len, keep, status = _run(ctx, table, k, v, acc, path, R,
                                             parent if with_parent else None)
        for src, out in ((k, ko), (v, vo)):
            ref = commit.compact_path(src.float().numpy(), table, ctx, paths, P)
            np.testing.assert_array_equal(out.float().numpy(), ref)
        n = commit.committed_length(ctx, acc)
        np.testing.assert_array_equal(new_len, n)
        np.testing.assert_array_equal(keep, (n + P - 1) // P)
        assert (status == 0).all()


def test_chain_commit_moves_nothing():
    B, R = 6, 8
    ctx, table, k, v, acc, _, _, _ = _case(B, R, 2, 128, 16, torch.bfloat16, 7, False)
    ko, vo, new_len, keep, status = _run(ctx, table, k, v, acc, None, R)
    assert torch.equal(ko, k) and torch.equal(vo, v)
    np.testing.assert_array_equal(new_len, commit.committed_length(ctx, acc))
    assert (status == 0).all()


def test_bad_inputs_are_reported_and_left_untouched():
    """Every rejection branch of the kernel's check, one sequence each; the good
    sequences beside them move exactly as the oracle says."""
    B, R, P = 8, 8, 16
    ctx, table, k, v, acc, paths, path, parent = _case(B, R, 2, 128, P, torch.bfloat16, 9, True)
    acc, path, table = acc.copy(), path.copy(), table.copy()
    # the bad sequences need a path of length >= 2: give them a chain 0-1-2-3
    for b in range(6):
        parent[b] = np.arange(-1, R - 1)
        paths[b] = [0, 1, 2, 3]
        path[b] = -1
        path[b, :3] = [1, 2, 3]
        acc[b] = 3
    npages = k.shape[0]
    acc[0] = R                                   # more accepted drafts than the block holds
    path[1, :3] = [2, 2, 3]                      # not strictly increasing
    path[2, :3] = [1, 3, 2]                      # decreasing
    table[3, (ctx[3] + 2) // P] = -1             # a page the path reads is missing
    table[4, (ctx[4] + 1) // P] = npages + 5     # a page the path writes is out of range
    path[5, :3] = [2, 3, 4]                      # increasing, but 2 is not a child of 0
    ko, vo, new_len, _, status = _run(ctx, table, k, v, acc, path, R, parent)
    bad = [0, 1, 2, 3, 4, 5]
    for b in bad:
        assert status[b] == sv.api.SEQ_BAD_TREE, b
        assert new_len[b] == ctx[b], b
    assert (status[6:] == 0).all()
    full = [[] if b in bad else paths[b] for b in range(B)]   # bad ones: nothing moves
    for src, out in ((k, ko), (v, vo)):
        ref = commit.compact_path(src.float().numpy(), table, ctx, full, P)
        np.testing.assert_array_equal(out.float().numpy(), ref)
    # without the parent array only the order is checked: sequence 5 is then moved
    _, _, _, _, status2 = _run(ctx, table, k, v, acc, path, R, None)
    assert status2[5] == 0 and status2[1] == sv.api.SEQ_BAD_TREE


def test_tree_sampler_feeds_commit_on_device():
    """accept_sample_tree -> kv_commit with no host step between them: the
    sampler's accepted_len and path_nodes are the commit's inputs as they stand."""
    spec = wl.Spec("chain_to_commit", B=6, Hq=8, Hkv=2, D=128, V=500, ctx=(20, 90),
                   tree_nodes=24, tree_depth=5, shuffle_pages=True, temperature=0.9,
                   draft_div=0.9, draft_noise=0.3, seed=17)
    w = wl.make_workload(spec, device=DEV)
    k0, v0 = w.k_cache.clone(), w.v_cache.clone()
    cfg = sv.SamplerConfig(temperature=spec.temperature)
    res = sv.accept_sample_tree(w.logits, w.draft_probs, w.draft_tokens, w.parent, w.uniforms,
                                cfg)
    new_len, keep, status = sv.kv_commit(w.k_cache, w.v_cache, w.block_table, w.ctx_len,
                                         res["accepted_len"], res["path"], w.parent)
    torch.cuda.synchronize()
    acc = res["accepted_len"].cpu().numpy()
    pth = res["path"].cpu().numpy()
    assert (status.cpu().numpy() == 0).all()
    assert acc.max() > 0, "no path moved anything: the case does not test the chaining"
    ctx = w.ctx_len.cpu().numpy()
    table = w.block_table.cpu().numpy()
    full = [[0] + pth[b, :acc[b]].tolist() for b in range(spec.B)]
    for src, out in ((k0, w.k_cache), (v0, w.v_cache)):
        ref = commit.compact_path(src.float().cpu().numpy(), table, ctx, full, spec.page_size)
        np.testing.assert_array_equal(out.float().cpu().numpy(), ref)
    np.testing.assert_array_equal(new_len.cpu().numpy(), commit.committed_length(ctx, acc))

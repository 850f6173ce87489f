"""GPU parity: KV commit after acceptance (processed lengths, tree path compaction)
against the oracle.  A copy: the caches must match bit for bit."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_76_gb300 as sv
from oracle import commit

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
    paths, path = None, None
    if tree:
        parent = np.full((B, R), -1, np.int64)
        paths = []
        path = np.full((B, R), -1, np.int32)
        acc = np.zeros(B, np.int32)
        for b in range(B):
            for i in range(1, R):
                parent[b, i] = rng.integers(0, i)
            pth = commit.accepted_path(parent[b], int(rng.integers(0, R)))
            paths.append(pth)
            path[b, :len(pth)] = pth
            acc[b] = len(pth) - 1
    else:
        acc = rng.integers(0, R, B).astype(np.int32)
    return ctx, table, k, v, acc, paths, path


def _run(ctx, table, k, v, acc, path, R):
    t = lambda a: torch.as_tensor(a).to(DEV).contiguous()  # noqa: E731
    kd, vd = k.to(DEV).contiguous(), v.to(DEV).contiguous()
    new_len, keep, status = sv.kv_commit(kd, vd, t(table), t(ctx), t(acc),
                                         None if path is None else t(path), R=R)
    torch.cuda.synchronize()
    return kd.cpu(), vd.cpu(), new_len.cpu().numpy(), keep.cpu().numpy(), status.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D,P", [(128, 16), (64, 4)])
def test_tree_path_compaction_matches_oracle(dtype, D, P):
    for seed in range(3):
        B, R, Hkv = 5, 16 if seed < 2 else 64, 2
        ctx, table, k, v, acc, paths, path = _case(B, R, Hkv, D, P, dtype, seed, True)
        ko, vo, new_len, keep, status = _run(ctx, table, k, v, acc, path, R)
        for src, out in ((k, ko), (v, vo)):
            ref = commit.compact_path(src.float().numpy(), table, ctx, paths, P)
            np.testing.assert_array_equal(out.float().numpy(), ref)
        n = commit.committed_length(ctx, acc)
        np.testing.assert_array_equal(new_len, n)
        np.testing.assert_array_equal(keep, (n + P - 1) // P)
        assert (status == 0).all()


def test_chain_commit_moves_nothing():
    B, R = 6, 8
    ctx, table, k, v, acc, _, _ = _case(B, R, 2, 128, 16, torch.bfloat16, 7, False)
    ko, vo, new_len, keep, status = _run(ctx, table, k, v, acc, None, R)
    assert torch.equal(ko, k) and torch.equal(vo, v)
    np.testing.assert_array_equal(new_len, commit.committed_length(ctx, acc))
    assert (status == 0).all()


def test_bad_inputs_are_reported_and_left_untouched():
    B, R = 3, 8
    ctx, table, k, v, acc, paths, path = _case(B, R, 2, 128, 16, torch.bfloat16, 9, True)
    acc = acc.copy()
    path = path.copy()
    acc[0] = R                   # more accepted drafts than the block holds
    path[1, 0] = 1               # the path must start at node 0
    ko, vo, new_len, _, status = _run(ctx, table, k, v, acc, path, R)
    assert status[0] == sv.api.SEQ_BAD_TREE and status[1] == sv.api.SEQ_BAD_TREE
    assert new_len[0] == ctx[0] and new_len[1] == ctx[1]
    # the good sequence moved exactly as the oracle says; the bad ones not at all
    ref = commit.compact_path(k.float().numpy(), table, ctx, [[0], [0], paths[2]], 16)
    np.testing.assert_array_equal(ko.float().numpy(), ref)
    assert status[2] == 0

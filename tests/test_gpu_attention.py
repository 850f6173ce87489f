"""GPU parity: tree_prepare and split-K verify attention against the oracle.

Element-by-element at sizes the oracle finishes quickly (several 64-token
stages, ragged tails, shuffled pages, several split counts); sampled outputs
at the full workload sizes.  Tolerances: 2e-2 absolute for bf16 inputs,
1e-5 absolute for the fp32 tiny configuration.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_76_gb300 as sv
from speculative_decoding_verification_76_gb300 import workloads as wl
from tests.util import BF16_ATOL, F32_ATOL, np_u64, oracle_attention

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gpu(w):
    return w.to(DEV)


def _run(w, num_splits=0, parent_null=False):
    g = _gpu(w)
    anc, pos, st = sv.tree_prepare(None if parent_null else g.parent, g.ctx_len, R=w.q.shape[1])
    out, lse = sv.verify_attn(g.q, g.k_cache, g.v_cache, g.block_table, g.ctx_len, anc,
                              num_splits=num_splits)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), np_u64(anc), pos.cpu().numpy(), \
        st.cpu().numpy()


# ------------------------------------------------------------------ tree_prepare
@pytest.mark.parametrize("R", [1, 5, 33, 64])
def test_tree_prepare_matches_oracle(R):
    spec = wl.Spec("t", B=7, Hq=1, Hkv=1, D=64, V=8, ctx=(0, 999), tree_nodes=R if R > 1 else 0,
                   gamma=0 if R == 1 else 4, seed=R)
    parent = wl.make_parent(spec, R)
    ctx = wl.make_ctx_lens(spec, R)
    m_o, d_o, p_o = oracle.tree.tree_prepare(parent, ctx)
    anc, pos, st = sv.tree_prepare(torch.from_numpy(parent).to(DEV), torch.from_numpy(ctx).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(np_u64(anc), m_o)
    assert np.array_equal(pos.cpu().numpy(), p_o)
    assert not st.cpu().numpy().any()


def test_tree_prepare_fox_and_chain():
    fox = np.array([[-1, 0, 1, 1, 0, 4]], dtype=np.int32)
    anc, pos, _ = sv.tree_prepare(torch.from_numpy(fox).to(DEV),
                                  torch.tensor([10], dtype=torch.int32, device=DEV))
    assert [int(x) for x in np_u64(anc)[0]] == [1, 3, 7, 11, 17, 49]
    assert pos.cpu().tolist() == [[10, 11, 12, 12, 11, 12]]
    anc, pos, _ = sv.tree_prepare(None, torch.tensor([0, 5], dtype=torch.int32, device=DEV), R=64)
    m = np_u64(anc)
    assert int(m[1, 63]) == (1 << 64) - 1 and pos.cpu()[1, 63].item() == 68


def test_tree_prepare_rejects_bad_parent():
    bad = np.array([[-1, 0, 2, 1], [-1, 0, 1, 1], [0, 0, 1, 1]], dtype=np.int32)
    _, _, st = sv.tree_prepare(torch.from_numpy(bad).to(DEV),
                               torch.zeros(3, dtype=torch.int32, device=DEV))
    assert st.cpu().tolist() == [sv.api.SEQ_BAD_TREE, 0, sv.api.SEQ_BAD_TREE]


# ------------------------------------------------------------------ attention, small sizes
def test_tiny_chain_fp32_exact_config():
    spec = wl.SPECS["tiny_chain"]
    w = wl.make_attention_inputs(spec)
    for ns in (0, 1, 2, 3):
        out, lse, anc, _, _ = _run(w, ns)
        ref, lref = oracle_attention(w, anc)
        assert np.abs(out - ref).max() < F32_ATOL, ns
        assert np.abs(lse - lref).max() < 1e-4


CASES = [
    # name, B, Hq, Hkv, R (chain gamma+1 or tree nodes), tree, ctx range, page, splits
    ("gqa4_chain", 3, 8, 2, 5, False, (100, 700), 16, (0, 1, 3, 7)),
    ("gqa4_chain8", 2, 32, 8, 8, False, (300, 900), 16, (0, 2)),
    ("mha_chain", 2, 2, 2, 4, False, (33, 260), 32, (0, 1, 5)),
    ("gqa8_chain16", 1, 16, 2, 16, False, (1000, 1000), 16, (0, 4)),
    ("tree64_gqa8", 2, 16, 2, 64, True, (200, 450), 16, (0, 1, 3)),
    ("tree12_gqa4", 3, 8, 2, 12, True, (0, 130), 16, (0, 2)),
    ("ctx0", 2, 8, 2, 5, False, (0, 0), 16, (0,)),
    # tcgen05 passes with softmax warps that own no valid row: 96 rows (one tile,
    # a dead warp), 200 rows (two tiles, the second partly dead), 384 rows (the
    # last CTA's second tile entirely dead)
    ("tc1_96rows", 2, 16, 2, 12, True, (300, 900), 16, (0, 2)),
    ("tc2_200rows", 2, 16, 2, 25, True, (300, 900), 16, (0, 3)),
    ("tc2_384rows", 1, 16, 2, 48, True, (700, 700), 16, (0, 1)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_bf16_attention_small(case):
    name, B, Hq, Hkv, R, tree, ctx, P, splits = case
    spec = wl.Spec(name, B=B, Hq=Hq, Hkv=Hkv, D=128, V=16, ctx=ctx, page_size=P,
                   tree_nodes=R if tree else 0, gamma=R - 1, shuffle_pages=True, seed=sum(map(ord, name)) % 97)
    w = wl.make_attention_inputs(spec)
    ref = None
    outs = []
    for ns in splits:
        out, lse, anc, _, _ = _run(w, ns)
        if ref is None:
            ref, lref = oracle_attention(w, anc)
        err = np.abs(out - ref).max()
        assert err < BF16_ATOL, (ns, err)
        assert np.abs(lse - lref).max() < 1e-3, ns
        outs.append(out)
    # the LSE combine makes the split count irrelevant up to rounding
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() < 1e-2


def test_chain_parent_null_equals_explicit_chain():
    spec = wl.Spec("c", B=2, Hq=8, Hkv=2, D=128, V=16, ctx=(50, 300), gamma=6, seed=3)
    w = wl.make_attention_inputs(spec)
    a = _run(w, 0, parent_null=False)
    b = _run(w, 0, parent_null=True)
    assert np.array_equal(a[2], b[2])
    assert np.array_equal(a[0], b[0])


@pytest.mark.parametrize("Hq,Hkv,R", [(8, 2, 7), (64, 8, 16), (4, 1, 64)])
def test_attention_without_mask_is_the_chain(Hq, Hkv, R):
    """No ancestor mask = the causal chain: identical outputs to the explicit chain
    mask on every bf16 kernel (warp-MMA: 28 rows per KV head; tcgen05 one tile:
    128; two tiles: 256)."""
    spec = wl.Spec("c2", B=2, Hq=Hq, Hkv=Hkv, D=128, V=16, ctx=(150, 700), gamma=R - 1,
                   shuffle_pages=True, seed=R)
    g = wl.make_attention_inputs(spec, device=DEV)
    anc, _, _ = sv.tree_prepare(None, g.ctx_len, R=R)
    o1, l1 = sv.verify_attn(g.q, g.k_cache, g.v_cache, g.block_table, g.ctx_len, anc)
    o2, l2 = sv.verify_attn(g.q, g.k_cache, g.v_cache, g.block_table, g.ctx_len, None)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_invisible_nodes_and_stale_cache_do_not_leak():
    """Sibling nodes' K/V and cache slots past the sequence end must not matter."""
    spec = wl.Spec("fox", B=1, Hq=4, Hkv=1, D=128, V=16, ctx=(70, 70), tree_nodes=6, seed=5)
    w = wl.make_attention_inputs(spec)
    w.parent = torch.tensor([[-1, 0, 1, 1, 0, 4]], dtype=torch.int32)
    base, _, anc, _, _ = _run(w, 0)
    w2 = wl.Workload(spec, **{f: getattr(w, f).clone() for f in
                              ("q", "k_cache", "v_cache", "block_table", "ctx_len", "parent")})
    P = spec.page_size
    ctx = 70
    for node in (4, 5):                     # runs, away
        t = ctx + node
        pg = int(w.block_table[0, t // P])
        w2.k_cache[pg, t % P] += 3.0
        w2.v_cache[pg, t % P] -= 2.0
    # poison the unused slots of the last page with NaN
    last = ctx + 6
    pg = int(w.block_table[0, (last - 1) // P])
    w2.k_cache[pg, last % P:] = float("nan")
    w2.v_cache[pg, last % P:] = float("nan")
    out, _, _, _, _ = _run(w2, 0)
    for node in (0, 1, 2, 3):               # fox, jumps, over, high do not see runs/away
        assert np.array_equal(out[0, node], base[0, node])
    assert np.isfinite(out).all()
    assert not np.allclose(out[0, 5], base[0, 5])


# ------------------------------------------------------------------ attention, full sizes
FULL = ["llama8b_chain", "long_context", "batched_serving_a75", "draft_tree"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_outputs(name):
    """The bench's launch at full size: every sequence and every block row, for one
    query head of every KV head (a different one per sequence) plus the first and
    last query heads, compared element by element with the oracle."""
    spec = wl.SPECS[name]
    w = wl.make_attention_inputs(spec, device=DEV)
    g = w
    anc, _, _ = sv.tree_prepare(g.parent, g.ctx_len)
    out, lse = sv.verify_attn(g.q, g.k_cache, g.v_cache, g.block_table, g.ctx_len, anc,
                              num_splits=spec.num_splits)
    torch.cuda.synchronize()
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    anc_np = np_u64(anc)
    B, R, Hq, _ = w.q.shape
    G = Hq // spec.Hkv
    assert np.isfinite(out).all()
    worst = 0.0
    for b in range(B):
        heads = sorted({0, Hq - 1} | {k * G + (b + k) % G for k in range(spec.Hkv)})
        ref, lref = oracle_attention(w, anc_np, batches=[b], heads=heads)
        err = np.abs(out[b][:, heads] - ref[b][:, heads]).max()
        worst = max(worst, float(err))
        assert err < BF16_ATOL, (b, err)
        assert np.abs(lse[b][:, heads] - lref[b][:, heads]).max() < 1e-3, b
    print(f"{name}: {B} sequences x {R} rows, max abs error {worst:.2e}")

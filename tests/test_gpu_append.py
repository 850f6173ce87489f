"""GPU parity for the steps in front of the verify calls: the block's K/V append
with keys rotated at their depth position (against oracle/append.py) and the
served target logits, bans and repetition penalty (against the sampler
oracle's served_logits).

Tolerances: values are copied, so bit-exact; rotated rows are rounded once to
the cache dtype from an fp32 rotation with fp32 sine / cosine of an angle
reduced in double, so each element is within one rounding of the oracle's
float64 value (bf16: 2^-8 relative) plus 2e-6 relative for the fp32 steps.
Penalised logits are computed in fp32 on both sides: bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_76_gb300 as sv
from oracle import append as oapp
from oracle import sampler as osm
from oracle.sampler import SamplerCfg
from speculative_decoding_verification_76_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _rel_tol(dtype):
    return (2.0 ** -8 if dtype == torch.bfloat16 else 0.0) + 2e-6


def _append_case(spec, dtype, D, rotate_q, seed):
    w = wl.make_attention_inputs(spec.with_(D=D), seed=seed)
    B, R, Hq, Hkv = spec.B, spec.R, spec.Hq, spec.Hkv
    g = torch.Generator().manual_seed(seed)
    k_new = torch.randn((B, R, Hkv, D), generator=g).to(dtype)
    v_new = torch.randn((B, R, Hkv, D), generator=g).to(dtype)
    kc, vc = w.k_cache.to(dtype), w.v_cache.to(dtype)
    q = w.q.to(dtype)
    anc, depth, pos = oracle.tree.tree_prepare(w.parent.numpy(), w.ctx_len.numpy())
    return w, k_new, v_new, kc, vc, q, pos


def _check_rows(got, ref, dtype):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bad = err > _rel_tol(dtype) * np.abs(ref) + 1e-6
    assert not bad.any(), (np.argwhere(bad)[:5], err.max())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("tree", [False, True])
def test_append_block_matches_oracle(dtype, D, tree):
    spec = wl.Spec("app", B=5, Hq=8, Hkv=2, D=D, V=16, ctx=(3, 300),
                   tree_nodes=24 if tree else 0, gamma=6, shuffle_pages=True, seed=31)
    w, k_new, v_new, kc, vc, q, pos = _append_case(spec, dtype, D, True, 31 + D + tree)
    kd, vd, qd = kc.to(DEV), vc.to(DEV), q.to(DEV)
    pos_t = torch.from_numpy(pos.astype(np.int32)).to(DEV) if tree else None
    st = sv.append_block(k_new.to(DEV), v_new.to(DEV), kd, vd, w.block_table.to(DEV),
                         w.ctx_len.to(DEV), pos_ids=pos_t, q=qd)
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()
    kref, vref = oapp.append_block(kc.double().numpy(), vc.double().numpy(),
                                   w.block_table.numpy(), w.ctx_len.numpy(),
                                   k_new.double().numpy(), v_new.double().numpy(), pos, spec.page_size)
    # values: copied bit for bit; every position outside the block untouched
    np.testing.assert_array_equal(vd.cpu().double().numpy(), vref)
    kgot = kd.cpu().double().numpy()
    touched = np.zeros(kgot.shape[:2], dtype=bool)
    P = spec.page_size
    for b in range(spec.B):
        for j in range(spec.R):
            t = int(w.ctx_len[b]) + j
            touched[int(w.block_table[b, t // P]), t % P] = True
    np.testing.assert_array_equal(kgot[~touched], kref[~touched])
    _check_rows(kgot[touched], kref[touched], dtype)
    # queries: rotated in place at the same positions
    _check_rows(qd.cpu().double().numpy(), oapp.rope(q.double().numpy(), pos), dtype)


def test_append_block_long_positions_and_bad_rows():
    """Positions past 10^5 (the long-context shape) keep the angle exact; a
    sequence whose page is missing is reported and left untouched."""
    dtype = torch.bfloat16
    spec = wl.Spec("app_long", B=3, Hq=8, Hkv=2, D=128, V=16, ctx=(131000, 131072), gamma=15,
                   shuffle_pages=True, seed=5)
    w, k_new, v_new, kc, vc, q, pos = _append_case(spec, dtype, 128, False, 5)
    table = w.block_table.clone()
    P = spec.page_size
    bad_b = 1
    t_bad = int(w.ctx_len[bad_b]) + 3
    table[bad_b, t_bad // P] = -1
    kd, vd = kc.to(DEV), vc.to(DEV)
    st = sv.append_block(k_new.to(DEV), v_new.to(DEV), kd, vd, table.to(DEV), w.ctx_len.to(DEV))
    torch.cuda.synchronize()
    st = st.cpu().numpy()
    assert st[bad_b] == sv.api.SEQ_BAD_TREE and st[0] == 0 and st[2] == 0
    good = [0, 2]
    kref, vref = oapp.append_block(kc.double().numpy(), vc.double().numpy(),
                                   table.numpy()[good], w.ctx_len.numpy()[good],
                                   k_new.double().numpy()[good], v_new.double().numpy()[good],
                                   pos[good], P)
    kgot = kd.cpu().double().numpy()
    for b in good:
        for j in range(spec.R):
            t = int(w.ctx_len[b]) + j
            slot = (int(table[b, t // P]), t % P)
            _check_rows(kgot[slot], kref[slot], dtype)
    # the bad sequence's rows on valid pages were not written either
    for j in range(spec.R):
        t = int(w.ctx_len[bad_b]) + j
        pg = int(table[bad_b, t // P])
        if pg >= 0:
            np.testing.assert_array_equal(kgot[pg, t % P], kc[pg, t % P].double().numpy())


# ------------------------------------------------------------------ served logits
def _penalty_case(B, R, V, tree, seed, H=40, n_ban=30):
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 3, (B, R, V)).astype(np.float32)
    logits[0, 0, :5] = 0.0                              # zeros: multiplied, stay 0
    hist = rng.integers(0, V, (B, H)).astype(np.int32)
    hist[:, -5:] = -1                                   # padding
    hist[:, 0] = hist[:, 1]                             # a repeated token: penalised once
    parent = None
    if tree:
        parent = np.stack([wl.random_tree(R, 5, 3, rng) for _ in range(B)]).astype(np.int32)
        toks = rng.integers(0, V, (B, R)).astype(np.int32)
        toks[:, 0] = -1
    else:
        toks = rng.integers(0, V, (B, R - 1)).astype(np.int32)
        toks[:, 1] = toks[:, 0]                         # a draft repeated in the block
    banned = rng.choice(V, n_ban, replace=False).astype(np.int32)
    banned[0] = hist[0, 2]                              # banned and penalised
    return logits, hist, toks, parent, banned


@pytest.mark.parametrize("tree", [False, True])
@pytest.mark.parametrize("penalty", [1.3, 0.7, 1.0])
def test_logits_penalize_matches_oracle(tree, penalty):
    B, R, V = 6, 24 if tree else 8, 5003
    logits, hist, toks, parent, banned = _penalty_case(B, R, V, tree, int(penalty * 10) + tree)
    t = lambda a: None if a is None else torch.as_tensor(a).to(DEV).contiguous()  # noqa: E731
    lg = t(logits)
    sv.logits_penalize(lg, t(hist), t(toks), t(parent), penalty=penalty, banned=t(banned))
    torch.cuda.synchronize()
    ref = osm.served_logits_batch(logits, hist, toks, parent, penalty, banned)
    np.testing.assert_array_equal(lg.cpu().numpy(), ref)


def test_penalized_rows_feed_the_sampler():
    """Served logits through the whole chain: penalise then sample, against the
    oracle sampling the oracle's served logits (bit-exact on unflagged rows)."""
    spec = wl.SPECS["llama8b_chain"].with_(B=8, V=32000)
    w = wl.make_sampler_inputs(spec, seed=9)
    rng = np.random.default_rng(9)
    hist = rng.integers(0, spec.V, (spec.B, 64)).astype(np.int32)
    banned = rng.choice(spec.V, 200, replace=False).astype(np.int32)
    lg = w.logits.to(DEV).contiguous()
    sv.logits_penalize(lg, torch.from_numpy(hist).to(DEV), w.draft_tokens.to(DEV), None,
                       penalty=1.2, banned=torch.from_numpy(banned).to(DEV))
    cfg = SamplerCfg(temperature=spec.temperature)
    res = sv.accept_sample(lg, w.draft_probs.to(DEV), w.draft_tokens.to(DEV),
                           w.uniforms.to(DEV), sv.SamplerConfig(temperature=spec.temperature))
    torch.cuda.synchronize()
    served = osm.served_logits_batch(w.logits.numpy(), hist, w.draft_tokens.numpy(), None, 1.2,
                                     banned)
    ref = osm.accept_chain_batch(served, w.draft_probs.numpy(), w.draft_tokens.numpy(),
                                 w.uniforms.numpy(), cfg)
    ok = ~ref["flagged"]
    assert ok.sum() >= spec.B - 1
    np.testing.assert_array_equal(res["accepted_len"].cpu().numpy()[ok], ref["accepted_len"][ok])
    np.testing.assert_array_equal(res["emitted"].cpu().numpy()[ok], ref["emitted"][ok])
    # no banned token is ever emitted
    em = res["emitted"].cpu().numpy()
    assert not np.isin(em[em >= 0], banned).any()

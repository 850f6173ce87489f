"""Pins for the oracle's acceptance sampler (CPU only).

Each test checks the oracle against something fixed outside it: a worked
example printed on the pages (tests/golden), a closed form, a textbook
special case, or a statistical test of the lossless property.
"""
import math

import numpy as np
import pytest
from scipy import stats

from oracle import sampler as osm
from oracle.sampler import SamplerCfg
from tests.conftest import load_golden


def _walk1(p, q, x, u_test, u_final):
    """One draft position followed by the final draw (R = 2)."""
    return osm.chain_walk([p, p], [q], [x], [u_test, u_final])


# ---------------------------------------------------------------- worked examples

def test_three_token_residual_and_rejection_mass():
    g = load_golden("three_token.json")
    p = np.array(g["solved_from_printed"]["p"])
    q = np.array(g["solved_from_printed"]["q"])
    pr = g["printed"]
    res, mass = osm.residual(p, q)
    np.testing.assert_allclose(np.maximum(0, p - q), pr["positive_part_p_minus_q"], atol=1e-12)
    np.testing.assert_allclose(res, pr["residual"], atol=1e-12)
    # rejection probability = sum_x q(x) (1 - min(1, p/q))
    rej = sum(q[x] * (1 - min(1.0, p[x] / q[x])) for x in range(3))
    assert rej == pytest.approx(pr["rejection_probability"], abs=1e-12)
    # the mass of the positive part equals the rejection probability
    assert mass == pytest.approx(pr["rejection_probability"], abs=1e-12)


def test_three_token_final_distribution_by_enumeration():
    """Enumerate the proposal and both uniforms: the output law equals p."""
    g = load_golden("three_token.json")
    p = np.array(g["solved_from_printed"]["p"])
    q = np.array(g["solved_from_printed"]["q"])
    n = 200
    grid = (np.arange(n) + 0.5) / n
    out = np.zeros(3)
    for x in range(3):
        for ut in grid:
            for uf in grid[::4]:
                r = _walk1(p, q, x, ut, uf)
                out[r["emitted"][0]] += q[x] / (n * len(grid[::4]))
    np.testing.assert_allclose(out, p, atol=0.011)
    pr = g["printed"]
    assert out[1] == pytest.approx(pr["final_B"], abs=0.011)
    assert out[2] == pytest.approx(pr["final_C"], abs=0.011)


def test_three_token_accepted_part_of_B():
    g = load_golden("three_token.json")
    p = np.array(g["solved_from_printed"]["p"])
    q = np.array(g["solved_from_printed"]["q"])
    # B proposed and accepted: q_B * min(1, p_B/q_B) = printed accepted part
    n = 1000
    acc = np.mean([_walk1(p, q, 1, (k + 0.5) / n, 0.5)["accepted_len"] for k in range(n)])
    assert q[1] * acc == pytest.approx(g["printed"]["final_B_accepted_part"], abs=1e-12)


def test_alpha_08_instance():
    g = load_golden("alpha08.json")
    p = np.array(g["constructed_instance"]["p"])
    q = np.array(g["constructed_instance"]["q"])
    pr = g["printed"]
    assert np.minimum(p, q).sum() == pytest.approx(pr["alpha"], abs=1e-12)
    res, mass = osm.residual(p, q)
    assert mass == pytest.approx(pr["rejection_probability"], abs=1e-12)
    vocab = g["constructed_instance"]["vocab"]
    for name in pr["residual_tokens"]:
        assert res[vocab.index(name)] == pytest.approx(pr["residual_each"], abs=1e-12)
    assert res[vocab.index("other")] == 0.0
    # empirical acceptance rate over drafts ~ q and uniform u
    rng = np.random.default_rng(5)
    xs = rng.choice(3, size=40000, p=q)
    us = rng.random(40000)
    acc = np.mean([_walk1(p, q, int(x), u, 0.5)["accepted_len"] for x, u in zip(xs, us)])
    assert acc == pytest.approx(pr["alpha"], abs=4 * math.sqrt(0.16 / 40000))


def test_chain_bird_shifted_rows():
    g = load_golden("chain_bird.json")
    c = g["constructed_distributions"]
    p_rows = np.array(c["p_rows"])
    q_rows = np.array(c["q_rows"])
    for uu in ([0.0] * 5, [0.999] * 5, [0.3, 0.7, 0.1, 0.9, 0.42]):
        r = osm.chain_walk(p_rows, q_rows, c["drafts"], uu)
        assert r["accepted_len"] == g["expected"]["accepted_len"]
        assert r["emitted"] == g["expected"]["emitted"]
    # unshifted use (row i+1 checking draft i+1) would reject 'the' at once
    r_bad = osm.chain_walk(p_rows[1:].tolist() + [p_rows[-1]], q_rows, c["drafts"], [0.5] * 5)
    assert r_bad["accepted_len"] != g["expected"]["accepted_len"]


# ---------------------------------------------------------------- closed form

@pytest.mark.parametrize("alpha_src,gamma", [("alpha08", 4), ("alpha08", 7), ("three", 4)])
def test_expected_tokens_closed_form(alpha_src, gamma):
    if alpha_src == "alpha08":
        g = load_golden("alpha08.json")["constructed_instance"]
    else:
        g = load_golden("three_token.json")["solved_from_printed"]
    p, q = np.array(g["p"]), np.array(g["q"])
    alpha = np.minimum(p, q).sum()
    expect = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    rng = np.random.default_rng(11 + gamma)
    n = 20000
    counts = np.empty(n)
    P = [p] * (gamma + 1)
    Q = [q] * gamma
    for s in range(n):
        drafts = rng.choice(3, size=gamma, p=q)
        u = rng.random(gamma + 1)
        counts[s] = len(osm.chain_walk(P, Q, drafts, u)["emitted"])
    assert counts.min() >= 1 and counts.max() <= gamma + 1
    se = counts.std() / math.sqrt(n)
    assert abs(counts.mean() - expect) < 4 * se, (counts.mean(), expect)


# ---------------------------------------------------------------- lossless (chi-square)

def _chisq_ok(counts, probs, min_p=1e-3):
    keep = probs > 0
    assert counts[~keep].sum() == 0, "emitted a token with p = 0"
    exp = probs[keep] * counts.sum()
    return stats.chisquare(counts[keep], exp).pvalue > min_p


@pytest.mark.parametrize("V,top_k,top_p", [(3, 0, 1.0), (32, 0, 1.0), (32, 5, 1.0), (32, 0, 0.8),
                                           (32, 8, 0.9)])
def test_emitted_tokens_follow_p(V, top_k, top_p):
    rng = np.random.default_rng(100 + V + top_k)
    cfg = SamplerCfg(temperature=0.9, top_k=top_k, top_p=top_p)
    logits = rng.normal(0, 2, size=V).astype(np.float32)
    p, _ = osm.target_distribution(logits, cfg)
    # a draft law that misses some of p's support and adds mass elsewhere
    q = np.exp(rng.normal(0, 1.5, size=V))
    q[np.argsort(-p)[1]] = 0.0
    q /= q.sum()
    gamma = 3
    P, Q = [p] * (gamma + 1), [q] * gamma
    n = 20000
    first = np.zeros(V)
    second = np.zeros(V)
    for _ in range(n):
        d = rng.choice(V, size=gamma, p=q)
        r = osm.chain_walk(P, Q, d, rng.random(gamma + 1))
        first[r["emitted"][0]] += 1
        if len(r["emitted"]) > 1:
            second[r["emitted"][1]] += 1
    assert _chisq_ok(first, p)
    assert _chisq_ok(second, p)


def test_tree_rule_first_token_follows_p_root():
    rng = np.random.default_rng(7)
    V = 6
    p_root = np.array([0.35, 0.25, 0.2, 0.1, 0.1, 0.0])
    q_root = np.array([0.05, 0.4, 0.05, 0.3, 0.0, 0.2])
    N = 5                                   # anchor + 3 children; child 1 has one child
    parent = [-1, 0, 0, 0, 1]
    p_nodes = [p_root] + [rng.dirichlet(np.ones(V)) for _ in range(N - 1)]
    q_nodes = [q_root] + [rng.dirichlet(np.ones(V)) for _ in range(N - 1)]
    n = 30000
    first = np.zeros(V)
    for _ in range(n):
        toks = [-1] + list(rng.choice(V, size=3, p=q_root)) + [rng.choice(V, p=q_nodes[1])]
        r = osm.tree_walk(p_nodes, q_nodes, toks, parent, rng.random(N))
        first[r["emitted"][0]] += 1
    assert _chisq_ok(first, p_root)


def test_tree_rule_reduces_to_chain():
    rng = np.random.default_rng(3)
    V, R = 16, 6
    for _ in range(200):
        P = [rng.dirichlet(np.ones(V) * 0.5) for _ in range(R)]
        Q = [rng.dirichlet(np.ones(V) * 0.5) for _ in range(R - 1)]
        d = [int(rng.choice(V, p=Q[i])) for i in range(R - 1)]
        u = rng.random(R)
        a = osm.chain_walk(P, Q, d, u)
        t = osm.tree_walk(P, Q + [Q[-1]], [-1] + d, list(range(-1, R - 1)), u)
        assert a["accepted_len"] == t["accepted_len"]
        assert a["emitted"] == t["emitted"]


# ---------------------------------------------------------------- special cases (test list)

def test_p_equals_q_never_rejects():
    rng = np.random.default_rng(1)
    p = rng.dirichlet(np.ones(10))
    for _ in range(500):
        d = rng.choice(10, size=4, p=p)
        r = osm.chain_walk([p] * 5, [p] * 4, d, rng.random(5))
        assert r["accepted_len"] == 4


def test_p_zero_always_rejects_and_q_zero_reachable():
    p = np.array([0.0, 0.6, 0.4])
    q = np.array([0.5, 0.5, 0.0])
    for u in (0.0, 0.5, 0.999):
        assert _walk1(p, q, 0, u, 0.1)["accepted_len"] == 0
    # token 2 has q = 0 < p: only the residual can emit it
    res, _ = osm.residual(p, q)
    assert res[2] > 0
    hits = sum(_walk1(p, q, 0, 0.5, (k + 0.5) / 100)["emitted"][0] == 2 for k in range(100))
    assert hits > 0


def test_q_zero_proposal_is_reported():
    p = np.array([0.2, 0.8])
    q = np.array([1.0, 0.0])
    r = _walk1(p, q, 1, 0.9, 0.5)
    assert r["accepted_len"] == 1 and r["status"] & osm.ST_QZERO


def test_topk_ties_take_lower_ids():
    logits = np.array([1.0, 3.0, 3.0, 2.0, 3.0], dtype=np.float32)
    p, _ = osm.target_distribution(logits, SamplerCfg(top_k=2))
    assert list(np.nonzero(p)[0]) == [1, 2]
    p, _ = osm.target_distribution(logits, SamplerCfg(top_k=3))
    assert list(np.nonzero(p)[0]) == [1, 2, 4]
    p, _ = osm.target_distribution(logits, SamplerCfg(top_k=4))
    assert list(np.nonzero(p)[0]) == [1, 2, 3, 4]


def test_topp_minimal_prefix_includes_crossing_token():
    logits = np.log(np.array([0.4, 0.3, 0.2, 0.1])).astype(np.float32)
    p, fl = osm.target_distribution(logits, SamplerCfg(top_p=0.65))
    np.testing.assert_allclose(p, [4 / 7, 3 / 7, 0, 0], rtol=1e-6)
    assert not fl
    p, fl = osm.target_distribution(logits, SamplerCfg(top_p=0.75))
    np.testing.assert_allclose(p, [4 / 9, 3 / 9, 2 / 9, 0], rtol=1e-6)
    # a cutoff that lands on the boundary is ambiguous: without room for
    # alternatives it is flagged, with room the other cutoff is offered
    p, fl = osm.target_distribution(logits, SamplerCfg(top_p=0.7))
    assert fl
    alts = []
    p, fl = osm.target_distribution(logits, SamplerCfg(top_p=0.7), alts)
    assert not fl and len(alts) == 1
    assert {int((p > 0).sum()), alts[0]} == {2, 3}
    alt = osm.p_for_cutoff(logits, SamplerCfg(top_p=0.7), alts[0])
    assert int((alt > 0).sum()) == alts[0] and alt.sum() == pytest.approx(1.0)


def test_topp_ambiguity_flags_only_when_outcome_changes():
    # p over 4 tokens with a cutoff on the boundary between 2 and 3 kept
    logits = np.log(np.array([0.4, 0.3, 0.2, 0.1])).astype(np.float32)
    cfg = SamplerCfg(top_p=0.7)
    q = np.array([0.25, 0.25, 0.25, 0.25])
    # draft 0 accepted for any u (p/q > 1 either way), bonus drawn with u = 0.1
    # from a row whose cutoff is unambiguous -> outcome is robust
    rob = osm.accept_chain(np.stack([logits, np.log(np.array([.97, .01, .01, .01])).astype(np.float32)]),
                           [q], [0], [0.5, 0.1], cfg)
    assert not rob["flagged"]
    # draft 2 is kept only under the 3-token cutoff: the outcome depends on it
    amb = osm.accept_chain(np.stack([logits, logits]), [q], [2], [0.5, 0.1], cfg)
    assert amb["flagged"]


def test_topk_then_topp_and_temperature():
    logits = np.array([0.0, 1.0, 2.0, 3.0, 4.0], dtype=np.float32)
    cfg = SamplerCfg(temperature=0.5, top_k=3, top_p=0.9)
    p, _ = osm.target_distribution(logits, cfg)
    z = np.array([4.0, 3.0, 2.0]) / np.float64(np.float32(0.5))
    e = np.exp(z - z.max())
    pk = e / e.sum()                       # top-3 renormalised: ~[0.867, 0.117, 0.016]
    assert pk[0] < 0.9 <= pk[0] + pk[1]
    expect = np.zeros(5)
    expect[[4, 3]] = pk[:2] / pk[:2].sum()
    np.testing.assert_allclose(p, expect, rtol=1e-12)


def test_normalization_and_temperature_limit():
    rng = np.random.default_rng(2)
    logits = rng.normal(0, 3, size=1000).astype(np.float32)
    p, _ = osm.target_distribution(logits, SamplerCfg(temperature=1.0))
    assert p.sum() == pytest.approx(1.0, abs=1e-12)
    # textbook softmax via scipy at T = 1
    from scipy.special import softmax
    np.testing.assert_allclose(p, softmax(logits.astype(np.float64)), rtol=1e-12)
    # very low temperature concentrates on the argmax
    p, _ = osm.target_distribution(logits, SamplerCfg(temperature=1e-3))
    assert np.argmax(p) == np.argmax(logits) and p.max() > 0.99


def test_banned_token_minus_inf():
    logits = np.array([0.0, -np.inf, 1.0], dtype=np.float32)
    p, _ = osm.target_distribution(logits, SamplerCfg())
    assert p[1] == 0.0 and p.sum() == pytest.approx(1.0)


def test_greedy_reproduces_argmax_chain():
    rng = np.random.default_rng(4)
    logits = rng.normal(0, 1, size=(6, 20)).astype(np.float32)
    am = logits.argmax(-1)
    drafts = list(am[:3]) + [int((am[3] + 1) % 20), int(am[4])]
    r = osm.accept_chain(logits, None, drafts, np.zeros(6), SamplerCfg(greedy=True))
    assert r["accepted_len"] == 3
    assert r["emitted"] == list(am[:4])
    r = osm.accept_chain(logits, None, list(am[:5]), np.zeros(6), SamplerCfg(greedy=True))
    assert r["accepted_len"] == 5 and r["emitted"] == list(am[:6])


def test_greedy_ties_lowest_id():
    logits = np.array([[0.0, 2.0, 2.0], [5.0, 5.0, 1.0]], dtype=np.float32)
    r = osm.accept_chain(logits, None, [2], np.zeros(2), SamplerCfg(greedy=True))
    assert r["accepted_len"] == 0 and r["emitted"] == [1]


def test_eos_inside_block_stops_emission():
    p = np.full(8, 1 / 8)
    r = osm.chain_walk([p] * 4, [p] * 3, [5, 7, 3], [0.1] * 4, eos_id=7)
    assert r["accepted_len"] == 2 and r["emitted"] == [5, 7]
    # a correction that is EOS is emitted as the last token
    pe = np.zeros(8)
    pe[7] = 1.0
    qe = np.zeros(8)
    qe[2] = 1.0
    r = osm.chain_walk([pe, p], [qe], [2], [0.1, 0.3], eos_id=7)
    assert r["accepted_len"] == 0 and r["emitted"] == [7]


def test_inverse_cdf_edges_and_flags():
    w = np.array([0.0, 0.25, 0.0, 0.75])
    assert osm.inverse_cdf(w, 0.0)[0] == 1
    assert osm.inverse_cdf(w, 0.2499)[0] == 1
    assert osm.inverse_cdf(w, 0.25)[0] == 3          # running sum must exceed u*Z
    assert osm.inverse_cdf(w, 0.999999)[0] == 3
    assert osm.inverse_cdf(w, 0.25)[1]               # on an edge: flagged
    assert not osm.inverse_cdf(w, 0.6)[1]


def test_ratio_flag():
    p = np.array([0.5, 0.5])
    q = np.array([0.25, 0.75])
    r = _walk1(p, q, 1, 0.5 / 0.75, 0.3)
    assert r["flagged"]
    r = _walk1(p, q, 1, 0.2, 0.3)
    assert not r["flagged"]


# ---------------------------------------------------------------- tree rule: greedy, EOS, zero residual
# The fox tree as stored (tests/golden/fox_tree.json): fox (anchor) -> {jumps -> {over, high},
# runs -> {away}}.  Node tokens are arbitrary ids; every expectation below is derived by hand
# from the stated rules: greedy follows the first child (storage order) whose token is the
# argmax of the current node's row and emits the argmax at the first mismatch or after a leaf;
# emission stops after an EOS, whether accepted or emitted as the final token.
FOX_PARENT = [-1, 0, 1, 1, 0, 4]
FOX_TOKENS = [-1, 10, 20, 21, 11, 30]          # jumps=10 over=20 high=21 runs=11 away=30


def _greedy_rows(argmax_by_row, V=40, N=6):
    """Logit rows whose argmax is given per row (others: a fixed low pattern)."""
    logits = np.tile(np.linspace(-1.0, -2.0, V), (N, 1)).astype(np.float32)
    for r, a in argmax_by_row.items():
        logits[r, a] = 5.0
    return logits


def _fox_greedy(argmax_by_row, tokens=FOX_TOKENS, eos=-1):
    cfg = SamplerCfg(greedy=True, eos_id=eos)
    return osm.accept_tree(_greedy_rows(argmax_by_row), None, tokens, FOX_PARENT, np.zeros(6),
                           cfg)


def test_tree_greedy_walk_fox_by_hand():
    # fox: argmax 11 = runs (node 4); runs: argmax 30 = away (node 5, a leaf); away: 7
    r = _fox_greedy({0: 11, 4: 30, 5: 7, 1: 20, 2: 1, 3: 2})
    assert r["path"] == [4, 5] and r["emitted"] == [11, 30, 7] and r["accepted_len"] == 2
    # fox: 10 = jumps; jumps: 22 matches neither over (20) nor high (21): emit 22
    r = _fox_greedy({0: 10, 1: 22})
    assert r["path"] == [1] and r["emitted"] == [10, 22] and r["accepted_len"] == 1
    # jumps: 21 = high, the second child (node 3); high is a leaf: its argmax 5 is emitted
    r = _fox_greedy({0: 10, 1: 21, 3: 5, 2: 9})
    assert r["path"] == [1, 3] and r["emitted"] == [10, 21, 5]
    # fox: 12 matches no child: nothing accepted, 12 emitted
    r = _fox_greedy({0: 12, 1: 20, 4: 30})
    assert r["path"] == [] and r["emitted"] == [12] and r["accepted_len"] == 0


def test_tree_greedy_siblings_with_the_argmax_token():
    # jumps and runs both carry token 10: the first in storage order (jumps) is followed,
    # even though only runs' row would have continued the match
    toks = [-1, 10, 20, 21, 10, 30]
    r = _fox_greedy({0: 10, 1: 3, 4: 30, 5: 6}, tokens=toks)
    assert r["path"] == [1] and r["emitted"] == [10, 3]
    r = _fox_greedy({0: 10, 1: 20, 2: 4}, tokens=toks)
    assert r["path"] == [1, 2] and r["emitted"] == [10, 20, 4]


def test_tree_greedy_eos_on_the_path():
    # over (20) is EOS and accepted: emission stops there, no bonus after it
    r = _fox_greedy({0: 10, 1: 20, 2: 5}, eos=20)
    assert r["path"] == [1, 2] and r["emitted"] == [10, 20] and r["accepted_len"] == 2
    # the EOS is the correction (matches no child of jumps): emitted last, not accepted
    r = _fox_greedy({0: 10, 1: 22}, eos=22)
    assert r["path"] == [1] and r["emitted"] == [10, 22] and r["accepted_len"] == 1
    # EOS accepted at depth 1 ends the walk before jumps' children are looked at
    r = _fox_greedy({0: 10, 1: 20}, eos=10)
    assert r["path"] == [1] and r["emitted"] == [10]


def test_tree_walk_eos_stops_after_an_accepted_node():
    V = 8
    uni = np.full(V, 1.0 / V)
    P = [uni] * 6
    Q = [uni] * 6                         # p = q everywhere: every first child is accepted
    toks = [-1, 1, 2, 3, 4, 5]
    u = [0.9, 0.9, 0.9, 0.9, 0.9, 0.3]
    r = osm.tree_walk(P, Q, toks, FOX_PARENT, u)
    # fox -> jumps (first child) -> over (first child, a leaf) -> bonus floor(0.3 * 8) = 2
    assert r["path"] == [1, 2] and r["emitted"] == [1, 2, 2]
    r = osm.tree_walk(P, Q, toks, FOX_PARENT, u, eos_id=2)
    assert r["path"] == [1, 2] and r["emitted"] == [1, 2] and r["accepted_len"] == 2
    r = osm.tree_walk(P, Q, toks, FOX_PARENT, u, eos_id=1)
    assert r["path"] == [1] and r["emitted"] == [1]


def test_zero_residual_draws_from_p_chain_and_tree():
    # p = q and the proposal has p = q = 0: it is rejected (u * 0 < 0 is false) and the
    # positive part of p - q is empty, so the draw falls back to p (reported, flagged)
    p = np.array([0.5, 0.5, 0.0, 0.0])
    r = osm.chain_walk([p, p], [p], [2], [0.5, 0.3])
    assert r["accepted_len"] == 0 and r["emitted"] == [0]      # 0.3 * 1 < 0.5: token 0
    assert r["status"] & osm.ST_RESID_ZERO and r["status"] & osm.ST_QZERO and r["flagged"]
    r = osm.chain_walk([p, p], [p], [3], [0.5, 0.7])
    assert r["emitted"] == [1]
    # tree: both children of fox propose a zero-mass token; p' stays p_root throughout
    toks = [-1, 2, 20, 21, 3, 30]
    P = [p] * 6
    Q = [p] * 6
    r = osm.tree_walk(P, Q, toks, FOX_PARENT, [0.5, 0.5, 0.5, 0.5, 0.5, 0.7])
    assert r["path"] == [] and r["emitted"] == [1]
    assert r["status"] & osm.ST_RESID_ZERO and r["flagged"]


def test_tree_topp_ambiguity_flags_only_when_outcome_changes():
    # the anchor's row has a top-p cutoff on the boundary between 2 and 3 kept tokens
    logits_root = np.log(np.array([0.4, 0.3, 0.2, 0.1])).astype(np.float32)
    logits_leaf = np.log(np.array([0.97, 0.01, 0.01, 0.01])).astype(np.float32)
    cfg = SamplerCfg(top_p=0.7)
    q = np.full((2, 4), 0.25)
    parent = [-1, 0]
    logits = np.stack([logits_root, logits_leaf])
    # token 0 is accepted under either cutoff (p(0) >= 0.4 / 0.9 > q): robust
    rob = osm.accept_tree(logits, q, [-1, 0], parent, [0.5, 0.1], cfg)
    assert rob["path"] == [1] and not rob["flagged"]
    # token 2 is kept only by the 3-token cutoff: the walk depends on it
    amb = osm.accept_tree(logits, q, [-1, 2], parent, [0.5, 0.1], cfg)
    assert amb["flagged"]
    # the same rows without ambiguity (top_p clear of the boundary) are not flagged
    clear = osm.accept_tree(logits, q, [-1, 2], parent, [0.5, 0.1], SamplerCfg(top_p=0.85))
    assert not clear["flagged"] and clear["path"] == [1]


# ---------------------------------------------------------------- served logits (bans, penalties)
def test_served_logits_closed_forms():
    l = np.array([2.0, -1.5, 0.0, 3.0, -4.0], dtype=np.float32)
    out = osm.served_logits(l, [0, 1, 2, 0, 0, -1, 99], penalty=2.0)
    # positive logits are divided, non-positive ones multiplied, once per distinct id;
    # ids outside the vocabulary are ignored
    np.testing.assert_array_equal(out, np.array([1.0, -3.0, 0.0, 3.0, -4.0], np.float32))
    assert out.dtype == np.float32
    # penalty 1 and no bans: the identity
    np.testing.assert_array_equal(osm.served_logits(l, [0, 1, 3], 1.0), l)
    # bans: -inf whatever the penalty did, and p = 0 there
    out = osm.served_logits(l, [3], penalty=1.3, banned=[3, 4, 7])
    assert out[3] == -np.inf and out[4] == -np.inf and out[0] == l[0]
    p, _ = osm.target_distribution(out, SamplerCfg())
    assert p[3] == 0.0 and p[4] == 0.0 and p.sum() == pytest.approx(1.0)


def test_served_logits_penalty_lowers_seen_tokens():
    rng = np.random.default_rng(8)
    l = rng.normal(0, 3, 300).astype(np.float32)
    seen = rng.integers(0, 300, 40)
    p0, _ = osm.target_distribution(l, SamplerCfg())
    p1, _ = osm.target_distribution(osm.served_logits(l, seen, penalty=1.5), SamplerCfg())
    s = np.unique(seen)
    rest = np.setdiff1d(np.arange(300), s)
    # every seen token loses probability relative to every unseen one
    assert np.all(p1[s] / p0[s] < p1[rest[0]] / p0[rest[0]])
    np.testing.assert_allclose(p1[rest] / p0[rest], p1[rest[0]] / p0[rest[0]], rtol=1e-9)


def test_row_prefix_tokens_chain_and_fox_tree():
    drafts = [11, 12, 13]
    assert [osm.row_prefix_tokens(drafts, None, i) for i in range(4)] == \
        [[], [11], [11, 12], [11, 12, 13]]
    toks = [-1, 10, 20, 21, 11, 30]      # fox, jumps, over, high, runs, away
    pre = [osm.row_prefix_tokens(toks, FOX_PARENT, v) for v in range(6)]
    # "over" scores after fox jumps over; "away" after fox runs away; siblings never mix
    assert pre == [[], [10], [10, 20], [10, 21], [11], [11, 30]]

"""Oracle: the lossless acceptance sampler of the verify step.

TEST INFRASTRUCTURE ONLY (see the package docstring).  float64 throughout.

Sources, all restated here in plain steps:

* "Speculative Decoding" (atlas), section "One round and shifted logits":
  the drafter proposes gamma tokens with their actual proposal
  probabilities; the target scores the block, giving gamma distributions that
  check the proposals plus one distribution after the last proposal; checks
  run left to right; the first rejection commits a corrected token and drops
  every later proposal; if all survive a bonus target token is sampled.  Row
  i of the target (row 0 = the pending anchor) checks draft i + 1: comparing
  unshifted logits is an off-by-one error.
* Same page, "Exact sampling: account for every probability" and the
  one-position listing under "Implementation roadmap and tests": accept the
  proposal x with probability min(1, p(x)/q(x)); on rejection draw from the
  positive part of p - q, renormalised.
* "Drafters and Speculative Decoding", section "Sampling needs a correction
  rule" (three-token example) and "Greedy verification".
* "Speculative Decoding" (atlas), "Greedy, sampling and the real sampler":
  greedy accepts while the proposal equals the target argmax and emits the
  argmax at the first mismatch; p and q must include temperature and
  truncation as actually served.
* Same page, "Chains, trees and visibility": a tree needs its own
  proposal/sampling rule; the rule used here is described in tree_walk.

Readings where the pages are silent (each also listed in the design notes):
  * z = logits / T; top-k keeps the k largest z (ties: lower token id first);
    top-p then keeps the shortest prefix, in (probability desc, id asc) order
    of the top-k-renormalised distribution, whose mass reaches top_p,
    including the crossing token; p is the softmax over the kept set.
    T, top_p are taken at their fp32 values, as served.
  * The acceptance test for u in [0, 1) is u * q(x) < p(x): the same event as
    u < min(1, p/q), without a division.  q(x) = 0 < p(x) therefore accepts
    and is reported; p(x) = 0 always rejects.
  * A draw from a weight vector w takes the first token id t whose running
    sum in ascending id order exceeds u * sum(w).  One uniform, u_final (the
    last one of the sequence), serves the correction draw and the bonus draw.
  * If the residual has zero mass after a rejection (possible only through
    rounding), the draw uses p itself and the sequence is reported.
  * Greedy takes the lowest id among equal maxima.
  * With eos_id >= 0, emission stops after the first EOS token, whether it is
    an accepted draft or the correction/bonus token.

Decision flags: a sequence whose outcome depends on a decision taken within
FLAG_EPS of its threshold is reported as flagged; bit-exact comparison skips
flagged sequences.
  * ratio test: |u - p(x)/q(x)| < FLAG_EPS;
  * inverse-CDF draw: u * Z within FLAG_EPS * Z of the chosen token's edges;
  * top-p: every cutoff that running masses perturbed by up to FLAG_EPS could
    select is tried; the sequence is flagged if any of them changes the
    outcome (accepted length or emitted tokens) of the walk.
"""
from dataclasses import dataclass

import numpy as np

FLAG_EPS = 1e-5

# per-sequence report bits (match the library's status_per_seq bits)
ST_QZERO = 1        # a proposed token had q(x) = 0
ST_NONFINITE = 2    # NaN or +inf in a target logit row that was read
ST_RESID_ZERO = 4   # residual mass was zero after a rejection


@dataclass
class SamplerCfg:
    temperature: float = 1.0
    top_k: int = 0
    top_p: float = 1.0
    greedy: bool = False
    eos_id: int = -1


def _f32(x) -> float:
    return float(np.float32(x))


MAX_ALTERNATIVES = 64


def _p_from_kept(z, kept):
    p = np.zeros(z.shape[0])
    zk = z[kept]
    e = np.exp(zk - zk.max())
    p[kept] = e / e.sum()
    return p


def _ordered_kept(logits_row, cfg: SamplerCfg):
    """z = logits / T and the top-k kept ids in (z desc, id asc) order."""
    l = np.asarray(logits_row, dtype=np.float64)
    V = l.shape[0]
    if np.any(np.isnan(l)) or np.any(l == np.inf):
        raise ValueError("non-finite target logit")
    z = l / _f32(cfg.temperature)
    order = np.lexsort((np.arange(V), -z))          # z descending, then id ascending
    kept = order
    if 0 < cfg.top_k < V:
        kept = kept[:cfg.top_k]
    return z, kept


def p_for_cutoff(logits_row, cfg: SamplerCfg, m: int):
    """p when top-p keeps exactly the first m tokens of the top-k order."""
    z, kept = _ordered_kept(logits_row, cfg)
    return _p_from_kept(z, kept[:m])


def target_distribution(logits_row, cfg: SamplerCfg, alternatives=None):
    """p over the vocabulary for one target row.  Returns (p, flagged).

    If `alternatives` is a list, the sizes of the other top-p cutoffs within
    FLAG_EPS (see the module docstring) are appended to it; more than
    MAX_ALTERNATIVES of them set the flag instead."""
    z, kept = _ordered_kept(logits_row, cfg)
    top_p = _f32(cfg.top_p)
    flagged = False
    if 0.0 < top_p < 1.0:
        zk = z[kept]
        e = np.exp(zk - zk[0])
        c = np.cumsum(e / e.sum())
        reach = np.nonzero(c >= top_p)[0]
        n = int(reach[0]) + 1 if reach.size else len(kept)
        # prefix lengths m that are "first to reach top_p" for some running
        # masses within FLAG_EPS of the exact ones
        prev = np.concatenate([[-np.inf], c[:-1]])
        cand = np.nonzero((c >= top_p - FLAG_EPS) & (prev < top_p + FLAG_EPS))[0] + 1
        others = [int(m) for m in cand if m != n]
        if others:
            if alternatives is None or len(others) > MAX_ALTERNATIVES:
                flagged = True
            else:
                alternatives.extend(others)
        kept = kept[:n]
    return _p_from_kept(z, kept), flagged


def inverse_cdf(w, u):
    """First id t (ascending) whose running sum of w exceeds u * sum(w).

    Returns (t, flagged)."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    Z = c[-1]
    if not Z > 0:
        raise ValueError("draw from a zero-mass vector")
    target = float(u) * Z
    t = int(np.searchsorted(c, target, side="right"))
    lo = c[t - 1] if t > 0 else 0.0
    flagged = (target - lo) < FLAG_EPS * Z or (c[t] - target) < FLAG_EPS * Z
    return t, bool(flagged)


def residual(p, q):
    """norm(max(0, p - q)) and its mass before normalising."""
    w = np.maximum(0.0, np.asarray(p, np.float64) - np.asarray(q, np.float64))
    m = w.sum()
    return (w / m if m > 0 else w), m


def _ratio_flag(u, px, qx) -> bool:
    return qx > 0 and abs(float(u) - px / qx) < FLAG_EPS


def chain_walk(p_rows, q_rows, drafts, u, eos_id=-1):
    """Left-to-right verification of one chain, given the final distributions.

    p_rows [R, V]: target distribution after block row i (row 0 = anchor).
    q_rows [R-1, V]: q_rows[i] is the distribution that proposed drafts[i].
    drafts [R-1]; u [R]: u[i] tests drafts[i], u[R-1] is the final draw.
    Returns dict(accepted_len, emitted, flagged, status).
    """
    R = len(p_rows)
    gamma = R - 1
    emitted, flagged, status = [], False, 0
    u_final = u[gamma]
    for i in range(gamma):
        x = int(drafts[i])
        px, qx = float(p_rows[i][x]), float(q_rows[i][x])
        if qx == 0.0:
            status |= ST_QZERO
        flagged |= _ratio_flag(u[i], px, qx)
        if float(u[i]) * qx < px:                    # accept with prob min(1, p/q)
            emitted.append(x)
            if x == eos_id:
                return dict(accepted_len=i + 1, emitted=emitted, flagged=flagged, status=status)
            continue
        w, mass = residual(p_rows[i], q_rows[i])     # first rejection: correction
        if mass == 0.0:
            w = p_rows[i]
            status |= ST_RESID_ZERO
            flagged = True
        t, fl = inverse_cdf(w, u_final)
        emitted.append(t)
        return dict(accepted_len=i, emitted=emitted, flagged=flagged | fl, status=status)
    t, fl = inverse_cdf(p_rows[gamma], u_final)      # every draft survived: bonus
    emitted.append(t)
    return dict(accepted_len=gamma, emitted=emitted, flagged=flagged | fl, status=status)


def greedy_argmax(row) -> int:
    """Lowest id among the maxima of one logit row."""
    return int(np.argmax(np.asarray(row, np.float64)))


def greedy_walk(logits, drafts, eos_id=-1):
    R = len(logits)
    gamma = R - 1
    emitted = []
    for i in range(gamma):
        a = greedy_argmax(logits[i])
        x = int(drafts[i])
        if x == a:
            emitted.append(x)
            if x == eos_id:
                return dict(accepted_len=i + 1, emitted=emitted, flagged=False, status=0)
            continue
        emitted.append(a)
        return dict(accepted_len=i, emitted=emitted, flagged=False, status=0)
    emitted.append(greedy_argmax(logits[gamma]))
    return dict(accepted_len=gamma, emitted=emitted, flagged=False, status=0)


def accept_chain(logits, q_rows, drafts, u, cfg: SamplerCfg):
    """One sequence: logits [R,V] fp32 values, q_rows [R-1,V], drafts [R-1], u [R]."""
    logits = np.asarray(logits)
    if cfg.greedy or cfg.temperature == 0:
        res = greedy_walk(logits, drafts, cfg.eos_id)
        res["p"] = None
        return res
    p_rows, alts, pflag = [], [], False
    for i in range(len(logits)):
        a = []
        p, fl = target_distribution(logits[i], cfg, a)
        p_rows.append(p)
        alts.append(a)
        pflag |= fl
    res = chain_walk(p_rows, q_rows, drafts, u, cfg.eos_id)
    flagged = res["flagged"] or pflag
    # rows the walk read: 0 .. last row it used; a near-threshold top-p cutoff
    # there flags the sequence only if moving the cutoff changes the outcome
    last_row = min(res["accepted_len"], len(p_rows) - 1)
    for i in range(last_row + 1):
        for m in alts[i]:
            if flagged:
                break
            trial = list(p_rows)
            trial[i] = p_for_cutoff(logits[i], cfg, m)
            r2 = chain_walk(trial, q_rows, drafts, u, cfg.eos_id)
            if r2["accepted_len"] != res["accepted_len"] or r2["emitted"] != res["emitted"]:
                flagged = True
    res["flagged"] = flagged
    res["p"] = np.stack(p_rows)
    res["alt_sizes"] = alts
    return res


def tree_walk(p_nodes, q_nodes, tokens, parent, u, eos_id=-1):
    """Draft-tree acceptance.  [READING: the pages give no rule]

    The rule is the multi-candidate form of the classical one, for children
    drawn i.i.d. from q at their parent: start at the anchor (node 0) with
    p' = p_0.  Try the children of the current node v in storage order; child
    c (token t) is accepted iff u[c-1] * q_v(t) < p'(t), and then the walk
    moves to c with p' = p_c.  A rejected child replaces p' by
    norm(max(0, p' - q_v)) before the next child is tried.  When no child is
    accepted (or v is a leaf) the final token is drawn from p' with u[N-1].
    For a chain (one child per node) this is exactly chain_walk.

    p_nodes, q_nodes [N, V]; tokens [N] (node 0 unused); parent [N]; u [N].
    Returns dict(accepted_len, path, emitted, flagged, status).
    """
    N = len(p_nodes)
    v = 0
    pcur = np.asarray(p_nodes[0], np.float64)
    path, emitted, flagged, status = [], [], False, 0
    children = [[c for c in range(N) if int(parent[c]) == v_] for v_ in range(N)]
    while True:
        moved = False
        for c in children[v]:
            t = int(tokens[c])
            px, qx = float(pcur[t]), float(q_nodes[v][t])
            if qx == 0.0:
                status |= ST_QZERO
            flagged |= _ratio_flag(u[c - 1], px, qx)
            if float(u[c - 1]) * qx < px:
                path.append(c)
                emitted.append(t)
                v = c
                pcur = np.asarray(p_nodes[c], np.float64)
                moved = True
                break
            w, mass = residual(pcur, q_nodes[v])
            if mass == 0.0:
                status |= ST_RESID_ZERO
                flagged = True
            else:
                pcur = w
        if moved and emitted[-1] == eos_id:
            break
        if not moved:
            t, fl = inverse_cdf(pcur, u[N - 1])
            emitted.append(t)
            flagged |= fl
            break
    return dict(accepted_len=len(path), path=path, emitted=emitted, flagged=flagged,
                status=status)


def accept_tree(logits, q_nodes, tokens, parent, u, cfg: SamplerCfg):
    logits = np.asarray(logits)
    N = len(logits)
    if cfg.greedy or cfg.temperature == 0:
        # greedy on a tree: follow the first child equal to the target argmax
        v, path, emitted = 0, [], []
        while True:
            a = greedy_argmax(logits[v])
            nxt = [c for c in range(N) if int(parent[c]) == v and int(tokens[c]) == a]
            emitted.append(a)
            if not nxt or a == cfg.eos_id:
                if nxt:
                    path.append(nxt[0])
                break
            path.append(nxt[0])
            v = nxt[0]
        return dict(accepted_len=len(path), path=path, emitted=emitted, flagged=False,
                    status=0, p=None)
    p_nodes, alts, pflag = [], [], False
    for i in range(N):
        a = []
        p, fl = target_distribution(logits[i], cfg, a)
        p_nodes.append(p)
        alts.append(a)
        pflag |= fl
    res = tree_walk(p_nodes, q_nodes, tokens, parent, u, cfg.eos_id)
    flagged = res["flagged"] or pflag
    for v in [0] + list(res["path"]):              # nodes whose p the walk read
        for m in alts[v]:
            if flagged:
                break
            trial = list(p_nodes)
            trial[v] = p_for_cutoff(logits[v], cfg, m)
            r2 = tree_walk(trial, q_nodes, tokens, parent, u, cfg.eos_id)
            if r2["path"] != res["path"] or r2["emitted"] != res["emitted"]:
                flagged = True
    res["flagged"] = flagged
    res["p"] = np.stack(p_nodes)
    res["alt_sizes"] = alts
    return res


def _pad(rows, width):
    out = np.full((len(rows), width), -1, dtype=np.int64)
    for b, r in enumerate(rows):
        out[b, :len(r)] = r
    return out


def accept_chain_batch(logits, q, drafts, u, cfg: SamplerCfg, want_p=False):
    """Batch form: logits [B,R,V], q [B,R-1,V], drafts [B,R-1], u [B,R]."""
    B, R = logits.shape[0], logits.shape[1]
    res = [accept_chain(logits[b], None if q is None else q[b], drafts[b], u[b], cfg)
           for b in range(B)]
    out = dict(accepted_len=np.array([r["accepted_len"] for r in res]),
               emitted=_pad([r["emitted"] for r in res], R),
               flagged=np.array([r["flagged"] for r in res]),
               status=np.array([r["status"] for r in res]))
    if want_p and res and res[0]["p"] is not None:
        out["p"] = np.stack([r["p"] for r in res])
        out["alt_sizes"] = [r["alt_sizes"] for r in res]
    return out


def accept_tree_batch(logits, q, tokens, parent, u, cfg: SamplerCfg, want_p=False):
    """Batch form: logits, q [B,N,V]; tokens, parent [B,N]; u [B,N]."""
    B, N = logits.shape[0], logits.shape[1]
    res = [accept_tree(logits[b], None if q is None else q[b], tokens[b], parent[b], u[b], cfg)
           for b in range(B)]
    out = dict(accepted_len=np.array([r["accepted_len"] for r in res]),
               path=_pad([r["path"] for r in res], N),
               emitted=_pad([r["emitted"] for r in res], N),
               flagged=np.array([r["flagged"] for r in res]),
               status=np.array([r["status"] for r in res]))
    if want_p and res and res[0]["p"] is not None:
        out["p"] = np.stack([r["p"] for r in res])
        out["alt_sizes"] = [r["alt_sizes"] for r in res]
    return out


# ---------------------------------------------------------------- served logits: bans, penalties
def row_prefix_tokens(block_tokens, parent, i: int):
    """Block tokens already in front of block row i (the row scores after them).

    Chain (parent None): block_tokens [R-1] are the drafts; row i follows drafts
    0 .. i-1.  Tree: block_tokens [R] are the node tokens (node 0, the anchor,
    is not listed -- the anchor belongs to the history); row v follows the
    tokens of its ancestors below the anchor and its own."""
    if parent is None:
        return [int(t) for t in block_tokens[:i]]
    out, v = [], int(i)
    while v > 0:
        out.append(int(block_tokens[v]))
        v = int(parent[v])
    return out[::-1]


def served_logits(logits_row, seen, penalty: float = 1.0, banned=()):
    """One target row as served ("Speculative Decoding" (atlas), "Greedy,
    sampling and the real sampler": p must include token bans and repetition
    penalties).  [READING: the pages give no formula]  The common multiplicative
    repetition penalty: every distinct token id in `seen` (the history and the
    row's block prefix) has its logit l replaced by l / penalty if l > 0, else
    l * penalty -- once, however often it occurs; then every banned id gets -inf.
    Ids outside [0, V) are ignored.  Computed in fp32, the arithmetic of the
    served logits."""
    out = np.array(logits_row, dtype=np.float32, copy=True)
    V = out.shape[0]
    th = np.float32(penalty)
    for t in sorted({int(t) for t in seen if 0 <= int(t) < V}):
        out[t] = out[t] / th if out[t] > 0 else out[t] * th
    for t in banned:
        if 0 <= int(t) < V:
            out[int(t)] = -np.inf
    return out


def served_logits_batch(logits, history, block_tokens, parent, penalty, banned):
    """logits [B,R,V]; history [B,H] (-1 unused); block_tokens chain [B,R-1] or
    tree [B,R]; parent [B,R] or None (chain)."""
    logits = np.asarray(logits, dtype=np.float32)
    out = np.empty_like(logits)
    B, R, _ = logits.shape
    for b in range(B):
        hist = [int(t) for t in np.asarray(history[b]) if int(t) >= 0]
        for i in range(R):
            pre = row_prefix_tokens(block_tokens[b], None if parent is None else parent[b], i)
            out[b, i] = served_logits(logits[b, i], hist + pre, penalty, banned)
    return out

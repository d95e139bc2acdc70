"""Acceptance rules, longest accepted path and the bonus token (fp64).

Node c != 0 carries tokens[c]; it is verified against the target distribution computed at its
parent p (the hidden state at a position predicts the next token: [MTP] section "Medusa",
[GLOSS] operation flow, [GUIDE] section "並列検証").

Rules
* greedy (temperature 0, the regime of [GUIDE] section "結論・成果"): accept c iff
  tokens[c] == argmax_v z[p, v] (lowest index on ties).
* typical ([GLOSS] section "Medusa-1: 典型的採択"): accept when the target probability of the
  candidate reaches an entropy-dependent threshold.  The page gives no formula; the rule used is
  p_p(x) >= min(eps, delta * exp(-H(p_p))), H in nats, with ">=" following the page's wording
  ("以上").  p_p = softmax(z[p] / tau).
* rejection ([GUIDE] section "棄却サンプリング：出力品質を保証する"): accept with probability
  min(1, T[x] / D[x]); on rejection sample from norm(relu(T - D)).  On a tree the siblings of a
  node are tried in index order against one residual R that starts at T_e and is replaced by
  norm(relu(R - D_e)) after each rejected sibling (if that residual has zero mass R is kept).
  D_e is the draft distribution the children of e were drawn from, scattered into the target
  vocabulary through the draft-to-target id map (zero outside the map).  A ratio with
  D[x] = 0 counts as 1 when R[x] > 0 and 0 otherwise.

Path ([GUIDE] same section: every candidate after a rejection is discarded; [MTP] section
"ツリー検証": the path that passes acceptance furthest is adopted).  Greedy/typical: enumerate
every root-to-leaf path, walk it from the root until the first rejected node; the endpoint is
the deepest node reached over all paths, lowest node index on ties.  Rejection: the walk above.
accept_len = depth of the endpoint; path = root ... endpoint.

Bonus token: greedy/typical take argmax z[endpoint] (not stated on the pages; deterministic
reading).  Rejection samples by inverse CDF over R: the smallest j with
sum_{v <= j} R[v] > u' * sum_v R[v], u' = U(seed, b, endpoint, purpose 1).

Margins (decisions within MARGIN of their threshold; counted, and a request with one is not
compared bit for bit): greedy, top-1 minus top-2 logit < MARGIN; typical,
|ln p(x) - ln thr| < MARGIN; rejection, |u - min(1, R[x]/D[x])| < MARGIN.  The bonus sample is
flagged when u' * sum R lies within MARGIN * sum R of a cumulative boundary; ``bonus_window``
is then the range of indices whose interval meets that band.
"""

import numpy as np

from .lmhead import logits, row_stats
from .philox import uniforms
from .tree import children, depths, root_to_leaf_paths, validate_tree

MARGIN = 1e-4


def _path_to(parent, e):
    path = []
    while e >= 0:
        path.append(e)
        e = int(parent[e])
    return path[::-1]


def _residual(R, De):
    """relu(R - D_e), the unnormalised residual after a rejected sibling."""
    return np.maximum(R - De, 0.0)


def verify_request(parent, n, tokens, z, rule, tau, eps, delta, seed, b, draft_row=None,
                   u_fn=None):
    """Verify one request.

    parent, tokens: int arrays [>= n]; z: float64 [n][V] logits of the real nodes;
    draft_row(e) -> float64 [V] draft distribution of e's children in target vocabulary
    (rejection only); u_fn(node, purpose) -> uniform, defaulting to the Philox uniforms
    U(seed, b, node, purpose).  Returns a dict with accept_len, path, bonus, path_margins,
    bonus_margin, bonus_window.
    """
    if u_fn is None:
        def u_fn(node, purpose):
            return float(uniforms(seed, b, node, purpose))
    if not validate_tree(parent, n):
        raise ValueError("bad tree")
    stats = {}

    def st(i):
        if i not in stats:
            stats[i] = row_stats(z[i], tau if tau > 0 else 0.0)
        return stats[i]

    if rule in ("greedy", "typical"):
        decided = {}

        def decide(c):
            if c not in decided:
                s = st(int(parent[c]))
                x = int(tokens[c])
                if rule == "greedy":
                    decided[c] = (x == s["argmax"], s["gap"] < MARGIN)
                else:
                    px = s["p"][x]
                    thr = min(eps, delta * np.exp(-s["entropy"]))
                    acc = px >= thr
                    margin = thr > 0 and px > 0 and abs(np.log(px) - np.log(thr)) < MARGIN
                    decided[c] = (bool(acc), bool(margin))
            return decided[c]

        dep = depths(parent, n)
        best = 0
        for path in root_to_leaf_paths(parent, n):
            e = path[0]
            for c in path[1:]:
                acc, _ = decide(c)
                if not acc:
                    break
                e = c
            if dep[e] > dep[best] or (dep[e] == dep[best] and e < best):
                best = e
        path = _path_to(parent, best)
        sb = st(best)
        return dict(accept_len=len(path) - 1, path=path, bonus=sb["argmax"],
                    path_margins=sum(1 for a, m in decided.values() if m),
                    bonus_margin=bool(sb["gap"] < MARGIN), bonus_window=(sb["argmax"], sb["argmax"]))

    if rule != "rejection":
        raise ValueError(rule)
    e = 0
    R = st(0)["p"]
    path = [0]
    margins = 0
    while True:
        kids = children(parent, n, e)
        moved = False
        if kids:
            De = draft_row(e)
        for c in kids:
            x = int(tokens[c])
            u = u_fn(c, 0)
            if De[x] > 0:
                a = min(1.0, R[x] / De[x])
            else:
                a = 1.0 if R[x] > 0 else 0.0
            if abs(u - a) < MARGIN:
                margins += 1
            if u < a:
                e = c
                R = st(c)["p"]
                path.append(c)
                moved = True
                break
            res = _residual(R, De)
            s = res.sum()
            if s > 0:
                R = res / s
        if not moved:
            break
    u2 = u_fn(e, 1)
    C = np.cumsum(R)
    total = C[-1]
    target = u2 * total
    bonus = int(np.searchsorted(C, target, side="right"))
    band = MARGIN * total
    near = np.abs(C - target).min() < band or target < band
    lo = int(np.searchsorted(C, target - band, side="right"))
    hi = min(int(np.searchsorted(C, target + band, side="right")), len(C) - 1)
    return dict(accept_len=len(path) - 1, path=path, bonus=min(bonus, len(C) - 1),
                path_margins=margins, bonus_margin=bool(near), bonus_window=(lo, hi))


def draft_in_target_vocab(draft_row, draft_to_target, V):
    """The draft distribution of one node in the target vocabulary (float64 [V]).

    With a draft-to-target id map (EAGLE-3's smaller draft vocabulary), draft entry j lands on
    target id draft_to_target[j] and every target id outside the map has draft probability 0;
    without a map the row is already in the target vocabulary.
    """
    row = np.asarray(draft_row, dtype=np.float64)
    if draft_to_target is None:
        return row.copy()
    De = np.zeros(V)
    De[np.asarray(draft_to_target)] = row
    return De


def verify_accept(hidden, W, tokens, parent, n_nodes, rule, tau, eps, delta, seed,
                  draft_probs=None, draft_to_target=None, requests=None):
    """Verify a batch.  hidden [B][N][Hd], W [V][Hd] (float32 holding exact values, or float64).

    Returns a list of per-request dicts (see ``verify_request``); ``requests`` restricts the
    batch to some request indices (others are None).
    """
    B = tokens.shape[0]
    V = W.shape[0]
    todo = list(range(B)) if requests is None else list(requests)
    rows = [(b, i) for b in todo for i in range(int(n_nodes[b]))]
    z_all = logits(np.stack([hidden[b, i] for b, i in rows]), W) if rows else None
    out = [None] * B
    r0 = 0
    for b in todo:
        n = int(n_nodes[b])
        z = z_all[r0: r0 + n]
        r0 += n
        draft_row = None
        if rule == "rejection":
            def draft_row(e, b=b):
                return draft_in_target_vocab(draft_probs[b, e], draft_to_target, V)
        out[b] = verify_request(parent[b], n, tokens[b], z, rule, tau, eps, delta, seed, b, draft_row)
    return out

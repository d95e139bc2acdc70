"""Dynamic (context-aware) draft tree construction in the EAGLE-2 manner, layer by layer.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages say only that EAGLE-2 builds the draft tree dynamically, adapting its shape to how
confident the context is ([MTP] section "ツリー検証": EAGLE-2's dynamic tree balances accepted
length against verification cost; [GLOSS] section "EAGLE: Medusaの発展形": context-aware tree
construction selects the topology per input; [GUIDE] section "EAGLE-1/2からの進化": dynamic draft
tree).  Reading adopted (plainest form of "confidence-driven" expansion): a node's value is the
cumulative log-probability of its path under the draft model.
  * expand: every node of the current frontier proposes its top-k draft tokens; a candidate's
    score is its parent's score plus log p(token); the next frontier is the F' best candidates.
  * select: the tree is the root plus the N - 1 best candidates of all layers (a child never
    scores above its parent, since log p <= 0, so the kept set is closed under parents), numbered
    breadth-first (layer, then candidate index).
Ties: equal log-probabilities order by the lower token id; equal scores by the lower
(layer, candidate index).  Scores are float32 sums, as the drafter hands them over.
"""

import numpy as np


def expand_layer(logp, frontier_score, topk, next_k, frontier_valid=None, frontier_cand=None):
    """One expansion layer of one request.

    logp [F][Vd] float32 draft log-probabilities of the frontier nodes; frontier_score [F]
    float32.  Returns dict: token, score, parent [F*topk] (candidate f*topk + r is frontier node
    f's r-th best token; parent = frontier_cand[f], -1 for the root layer; invalid frontier rows
    give token -1, score -inf), next_index [next_k] (best candidates, -1 padded), next_score.
    """
    logp = np.asarray(logp, dtype=np.float32)
    F, Vd = logp.shape
    fs = np.asarray(frontier_score, dtype=np.float32)
    valid = np.ones(F, dtype=bool) if frontier_valid is None else np.asarray(frontier_valid) != 0
    fc = np.full(F, -1, dtype=np.int64) if frontier_cand is None else np.asarray(frontier_cand, dtype=np.int64)
    C = F * topk
    token = np.full(C, -1, dtype=np.int64)
    score = np.full(C, -np.inf, dtype=np.float32)
    parent = np.full(C, -1, dtype=np.int64)
    for f in range(F):
        if not valid[f]:
            continue
        order = np.lexsort((np.arange(Vd), -logp[f].astype(np.float64)))[:topk]
        for r, v in enumerate(order):
            c = f * topk + r
            token[c] = v
            score[c] = np.float32(fs[f] + logp[f, v])  # one float32 rounding, as on the device
            parent[c] = fc[f]
    ok = np.nonzero(score > -np.inf)[0]
    ranked = sorted(ok.tolist(), key=lambda c: (-float(score[c]), c))[:next_k]
    nxt = np.full(next_k, -1, dtype=np.int64)
    nxt[: len(ranked)] = ranked
    nscore = np.full(next_k, -np.inf, dtype=np.float32)
    nscore[: len(ranked)] = score[ranked]
    return dict(token=token, score=score, parent=parent, next_index=nxt, next_score=nscore)


def select_tree(score, token, parent, n_max, root_token=0, draft_to_target=None):
    """Tree of one request from all layers' candidates.

    score / token / parent [D][C] (parent: candidate index in the previous layer, ignored on
    layer 0; a candidate with score -inf, or a parent of -1 below layer 0, is absent).  Returns
    (tree_parent [N], tree_token [N], n_nodes, node_cand [N]) with node 0 the root; node_cand is
    layer * C + index (-1 for the root and for padding).
    """
    score = np.asarray(score, dtype=np.float32)
    D, C = score.shape
    present = np.zeros((D, C), dtype=bool)
    for l in range(D):
        for j in range(C):
            present[l, j] = score[l, j] > -np.inf and (l == 0 or parent[l][j] >= 0)
    cands = [(l, j) for l in range(D) for j in range(C) if present[l, j]]
    cands.sort(key=lambda lj: (-float(score[lj]), lj[0], lj[1]))
    kept = sorted(cands[: n_max - 1])  # breadth-first: (layer, index)
    node = {lj: i + 1 for i, lj in enumerate(kept)}
    tree_parent = np.full(n_max, -1, dtype=np.int64)
    tree_token = np.zeros(n_max, dtype=np.int64)
    node_cand = np.full(n_max, -1, dtype=np.int64)
    tree_token[0] = root_token
    for (l, j), i in node.items():
        tree_parent[i] = 0 if l == 0 else node[(l - 1, int(parent[l][j]))]  # KeyError = not closed
        t = int(token[l][j])
        tree_token[i] = t if draft_to_target is None else int(draft_to_target[t])
        node_cand[i] = l * C + j
    return tree_parent, tree_token, 1 + len(kept), node_cand

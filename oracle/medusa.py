"""Static Medusa tree expansion: per-head top-k candidates placed on a fixed tree topology.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[GLOSS] section "ツリー構造の候補構築": Medusa builds its candidate tree from combinations of the
top candidates of each head.  Head 0's top-3, head 1's top-3 and head 2's top-2 give at most
3 x 3 x 2 = 18 paths.  The tree follows a predefined topology ("Medusa Tree"); the standard
ones have 63, 127 or 255 nodes.

A node at depth d >= 1 is a tuple (r_0, ..., r_{d-1}) of ranks, r_j < k_j: the path takes the
r_j-th best token of head j at step j + 1.  Its own token is therefore the r_{d-1}-th best token
of head d - 1; its parent is the tuple without the last rank; the root is the empty tuple.

Readings (the pages leave these open): a head's "top candidates" are ordered by logit, ties to
the lower token id; a topology "pruned to N nodes" keeps the N - 1 tuples that come first in
the order (sum of ranks, depth, tuples compared element by element), which keeps every prefix
of a kept tuple (a prefix has a smaller or equal rank sum and a smaller depth); nodes are
numbered breadth-first (depth, then tuple), so siblings are contiguous and ordered by rank.
"""

import itertools

import numpy as np


def head_topk(x, k):
    """Indices of the k largest entries of x, best first; equal values go to the lower index."""
    x = np.asarray(x, dtype=np.float64)
    order = np.lexsort((np.arange(len(x)), -x))  # primary key -x, then the index
    return order[:k].astype(np.int64)


def cartesian_tuples(topk):
    """Every rank tuple of the full Cartesian tree for per-head candidate counts ``topk``."""
    out = []
    for d in range(1, len(topk) + 1):
        out.extend(itertools.product(*[range(int(k)) for k in topk[:d]]))
    return out


def pruned_topology(topk, n_nodes):
    """(parent, rank) arrays of the first n_nodes - 1 tuples in (rank sum, depth, tuple) order,
    numbered breadth-first (depth, then tuple) after the root; rank[i] is node i's rank in its
    head's list (0 at the root)."""
    tuples = cartesian_tuples(topk)
    if n_nodes < 1 or n_nodes - 1 > len(tuples):
        raise ValueError("topology size outside 1 .. 1 + product")
    tuples.sort(key=lambda t: (sum(t), len(t), t))
    kept = sorted(tuples[: n_nodes - 1], key=lambda t: (len(t), t))
    index = {(): 0}
    parent = [-1]
    rank = [0]
    for t in kept:
        index[t] = len(parent)
        parent.append(index[t[:-1]])
        rank.append(t[-1])
    return np.array(parent, dtype=np.int32), np.array(rank, dtype=np.int32)


def topology_depths(parent):
    d = np.zeros(len(parent), dtype=np.int64)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1
    return d


def medusa_expand(head_logits, parent, rank, topk, root_token=None):
    """Tokens of every node for every request.

    head_logits [B][K][V] (head j predicts the token j + 1 steps ahead); parent / rank: the
    topology; topk: candidates taken per head (rank < topk).  Returns (tokens [B][N] int32,
    topk_index [B][K][topk] int64).  tokens[b][0] = root_token[b] (0 when not given).
    """
    head_logits = np.asarray(head_logits, dtype=np.float64)
    B, K, _ = head_logits.shape
    N = len(parent)
    depth = topology_depths(parent)
    if parent[0] != -1 or any(not (0 <= parent[i] < i) for i in range(1, N)):
        raise ValueError("bad topology")
    if any(depth[i] > K or rank[i] >= topk or rank[i] < 0 for i in range(1, N)):
        raise ValueError("node beyond the heads or the candidate count")
    idx = np.zeros((B, K, topk), dtype=np.int64)
    for b in range(B):
        for j in range(K):
            idx[b, j] = head_topk(head_logits[b, j], topk)
    tokens = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        tokens[b, 0] = 0 if root_token is None else int(root_token[b])
        for i in range(1, N):
            tokens[b, i] = idx[b, depth[i] - 1, rank[i]]
    return tokens, idx

"""Draft-tree topologies as parent arrays.

Convention used everywhere in this repository: node 0 is the root (the last already-accepted
token), ``parent[0] == -1`` and ``0 <= parent[i] < i`` for every other node, so the node order
is topological; siblings are ordered by node index.

* Tree of the tiny fp32 case: root, 3 children, 2 children each (10 nodes).
* Static Medusa-style trees from per-depth top-k (jisaku glossary "Medusa", section on the tree
  candidate structure: top-3 x top-3 x top-2 gives up to 18 paths).  The named 63/127/255-node
  topologies are not given on the pages, so a prefix-closed subset of the Cartesian product is
  kept by sorting candidates by (sum of ranks, depth, lexicographic order).
* Random breadth-first trees with 1..4 children per node and a depth limit.
"""

import itertools
from collections import deque

import numpy as np


def tree_root_3x2():
    """Root with 3 children, each child with 2 children (10 nodes)."""
    return np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], dtype=np.int32)


def _tuples_to_parent(tuples):
    """Order rank tuples breadth-first (depth, then lexicographic) and return (parent, rank)."""
    order = [()] + sorted(tuples, key=lambda t: (len(t), t))
    index = {t: i for i, t in enumerate(order)}
    parent = np.full(len(order), -1, dtype=np.int32)
    rank = np.zeros(len(order), dtype=np.int32)
    for t, i in index.items():
        if t:
            parent[i] = index[t[:-1]]
            rank[i] = t[-1]
    return parent, rank


def cartesian_tree(topk):
    """Full prefix tree of the Cartesian product of per-depth top-k ranks.

    Returns (parent, sibling_rank).  Node tuple (r1, ..., rd) is the candidate taking rank r1
    at depth 1, ..., rank rd at depth d.
    """
    tuples = []
    for d in range(1, len(topk) + 1):
        tuples.extend(itertools.product(*[range(k) for k in topk[:d]]))
    return _tuples_to_parent(tuples)


def static_topk_tree(topk, n_nodes):
    """Prefix-closed subset of ``cartesian_tree(topk)`` with ``n_nodes`` nodes (root included).

    Candidates are ranked by (sum of ranks, depth, lexicographic); a prefix of a tuple always
    ranks before the tuple, so every leading subset of that order is a valid tree.
    """
    tuples = []
    for d in range(1, len(topk) + 1):
        tuples.extend(itertools.product(*[range(k) for k in topk[:d]]))
    tuples.sort(key=lambda t: (sum(t), len(t), t))
    if n_nodes - 1 > len(tuples):
        raise ValueError("tree larger than the Cartesian product")
    return _tuples_to_parent(tuples[: n_nodes - 1])


def random_bfs_tree(rng, n_nodes, max_depth, branch=(1, 4)):
    """Breadth-first random tree: each node above ``max_depth`` gets U{branch} children.

    Stops at ``n_nodes`` nodes, or earlier when every open node sits at ``max_depth``.
    Returns (parent, sibling_rank).
    """
    parent = [-1]
    rank = [0]
    depth = [0]
    queue = deque([0])
    while queue and len(parent) < n_nodes:
        p = queue.popleft()
        if depth[p] >= max_depth:
            continue
        nb = int(rng.integers(branch[0], branch[1] + 1))
        for r in range(nb):
            if len(parent) >= n_nodes:
                break
            parent.append(p)
            rank.append(r)
            depth.append(depth[p] + 1)
            queue.append(len(parent) - 1)
    return np.array(parent, dtype=np.int32), np.array(rank, dtype=np.int32)


def sibling_rank(parent):
    """Rank of each node among its siblings (0 for the first child), root gets 0."""
    parent = np.asarray(parent)
    rank = np.zeros(len(parent), dtype=np.int32)
    seen = {}
    for i in range(1, len(parent)):
        p = int(parent[i])
        rank[i] = seen.get(p, 0)
        seen[p] = rank[i] + 1
    return rank


def depths(parent):
    """Depth of every node (root = 0) for a topologically ordered parent array."""
    parent = np.asarray(parent)
    d = np.zeros(len(parent), dtype=np.int32)
    for i in range(1, len(parent)):
        d[i] = d[parent[i]] + 1
    return d


def chain_tree(n):
    """A single chain root -> 1 -> 2 -> ... (n nodes)."""
    return np.arange(-1, n - 1, dtype=np.int32)

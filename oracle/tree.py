"""Tree structure: validity, ancestors, the tree attention mask and root-to-leaf paths.

[MTP] section "ツリー検証：候補を「木」に束ねて1回で確かめる": every tree node (candidate token)
may attend only to its own ancestor nodes, which lets all candidate paths run as one batched
sequence in a single forward.  [GUIDE] section "Tree Attention：候補を木構造で探索する" draws the
same mask for a root with children t1a, t1b, t1c.  Each node also sees the KV-cache prefix
([GUIDE] section "並列検証"), and itself (its own key is the last position of its path).

Convention: node 0 is the root; parent[0] == -1 and 0 <= parent[i] < i.
"""

import numpy as np


def validate_tree(parent, n):
    """True iff parent[:n] is a topologically ordered tree rooted at node 0."""
    if n < 1 or n > len(parent):
        return False
    if int(parent[0]) != -1:
        return False
    for i in range(1, n):
        p = int(parent[i])
        if p < 0 or p >= i:
            return False
    return True


def ancestors_or_self(parent, i):
    """Set of nodes on the path from the root to node i (both included), by walking parents."""
    out = set()
    while i >= 0:
        out.add(i)
        i = int(parent[i])
    return out


def depths(parent, n):
    return np.array([len(ancestors_or_self(parent, i)) - 1 for i in range(n)], dtype=np.int64)


def tree_mask(parent, n, prefix_len):
    """Boolean [n][prefix_len + n]: row i sees the whole prefix and tree slots of anc(i) + {i}."""
    m = np.zeros((n, prefix_len + n), dtype=bool)
    m[:, :prefix_len] = True
    for i in range(n):
        for a in ancestors_or_self(parent, i):
            m[i, prefix_len + a] = True
    return m


def children(parent, n, e):
    """Children of node e in node-index order."""
    return [c for c in range(1, n) if int(parent[c]) == e]


def root_to_leaf_paths(parent, n):
    """Every root-to-leaf path as a list of node indices, root first, leaves in index order."""
    has_child = np.zeros(n, dtype=bool)
    for c in range(1, n):
        has_child[int(parent[c])] = True
    paths = []
    for leaf in range(n):
        if has_child[leaf]:
            continue
        path = []
        i = leaf
        while i >= 0:
            path.append(i)
            i = int(parent[i])
        paths.append(path[::-1])
    return paths

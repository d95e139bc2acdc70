"""Pins of the oracle's static Medusa tree expansion ([GLOSS] section "ツリー構造の候補構築")."""

import itertools

import numpy as np

import oracle
from gen import trees as T


def _leaves(parent):
    has_child = set(int(p) for p in parent[1:])
    return [i for i in range(len(parent)) if i not in has_child]


def test_pages_example_3x3x2_gives_18_paths():
    full = oracle.cartesian_tuples((3, 3, 2))
    parent, rank = oracle.pruned_topology((3, 3, 2), 1 + len(full))
    assert len(full) == 3 + 9 + 18
    assert len(_leaves(parent)) == 18  # every root-to-leaf path is one 3 x 3 x 2 combination


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(0)
    for _ in range(200):
        V = int(rng.integers(1, 9))
        x = rng.integers(-3, 4, size=V).astype(np.float64)  # many ties
        k = int(rng.integers(1, V + 1))
        best = max(itertools.permutations(range(V), k),
                   key=lambda p: tuple((x[i], -i) for i in p))
        assert oracle.head_topk(x, k).tolist() == list(best)
    assert oracle.head_topk([1.0, 3.0, 3.0, 2.0], 3).tolist() == [1, 2, 3]


def test_pruned_topology_is_a_prefix_closed_tree_in_the_stated_order():
    topk = (3, 3, 2, 2, 1)
    full = oracle.cartesian_tuples(topk)
    for n in (1, 2, 10, 63, 1 + len(full)):
        parent, rank = oracle.pruned_topology(topk, n)
        assert len(parent) == n and oracle.validate_tree(parent, n)
        # rebuild each node's tuple from the parent chain: kept tuples = first n-1 in order
        tup = [()]
        for i in range(1, n):
            tup.append(tup[parent[i]] + (int(rank[i]),))
        want = sorted(full, key=lambda t: (sum(t), len(t), t))[: n - 1]
        assert tup[1:] == sorted(want, key=lambda t: (len(t), t))


def test_topology_agrees_with_the_input_generator():
    """The input generator builds the config-2 topology with its own code."""
    for topk, n in (((3, 3, 2, 2, 1), 63), ((4, 4, 3, 2, 2), 127), ((6, 5, 4, 3, 3), 255)):
        p_o, r_o = oracle.pruned_topology(topk, n)
        p_g, r_g = T.static_topk_tree(topk, n)
        assert (p_o == p_g).all() and (r_o == r_g).all()


def test_expand_hand_example():
    # two heads over a 5-token vocabulary
    z = np.array([[[0.1, 0.9, 0.5, 0.9, -1.0],     # head 0 ranks: 1, 3, 2, 0, 4
                   [2.0, 0.0, 1.0, 3.0, 1.0]]])    # head 1 ranks: 3, 0, 2, 4, 1
    parent, rank = oracle.pruned_topology((2, 2), 7)
    tokens, idx = oracle.medusa_expand(z, parent, rank, topk=2, root_token=[42])
    assert idx[0].tolist() == [[1, 3], [3, 0]]
    depth = [0, 1, 1, 2, 2, 2, 2]
    for i in range(1, 7):
        assert tokens[0, i] == idx[0, depth[i] - 1, rank[i]]
    assert tokens[0, 0] == 42
    assert sorted(tokens[0, 1:3].tolist()) == [1, 3] and sorted(tokens[0, 3:].tolist()) == [0, 0, 3, 3]


def test_expand_rejects_nodes_beyond_the_heads():
    parent, rank = oracle.pruned_topology((2, 2, 2), 15)
    z = np.zeros((1, 2, 4))
    try:
        oracle.medusa_expand(z, parent, rank, topk=2)
    except ValueError:
        return
    raise AssertionError("depth 3 with two heads must fail")

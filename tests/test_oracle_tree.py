"""Pins for the oracle's tree handling (ancestor-only mask, paths, validation)."""

import json
import os

import networkx as nx
import numpy as np
import pytest

import oracle
from gen import trees as T

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_figure_guide.json")


def test_guide_figure_fixture():
    g = json.load(open(GOLDEN))
    parent = np.array(g["parent"])
    n = len(parent)
    assert oracle.validate_tree(parent, n)
    for i in range(n):
        assert oracle.ancestors_or_self(parent, i) == set(g["ancestors_or_self"][i])
    assert oracle.root_to_leaf_paths(parent, n) == g["root_to_leaf_paths"]
    assert list(oracle.depths(parent, n)) == g["depth"]
    # mask: prefix of 5 slots fully visible, tree part = ancestors-or-self
    m = oracle.tree_mask(parent, n, 5)
    assert m[:, :5].all()
    for i in range(n):
        assert set(np.nonzero(m[i, 5:])[0].tolist()) == set(g["ancestors_or_self"][i])


def _random_tree(rng, n):
    parent = np.full(n, -1)
    for i in range(1, n):
        parent[i] = rng.integers(0, i)
    return parent


@pytest.mark.parametrize("n", [1, 2, 7, 33, 255])
def test_mask_matches_graph_library_ancestors(n):
    rng = np.random.default_rng(n)
    parent = _random_tree(rng, n)
    G = nx.DiGraph()
    G.add_nodes_from(range(n))
    G.add_edges_from((int(parent[i]), i) for i in range(1, n))
    L = 3
    m = oracle.tree_mask(parent, n, L)
    for i in range(n):
        expect = nx.ancestors(G, i) | {i}
        assert set(np.nonzero(m[i, L:])[0].tolist()) == expect
        assert m[i, :L].all()
        # depth = shortest path length from the root
        assert oracle.depths(parent, n)[i] == nx.shortest_path_length(G, 0, i)


def test_paths_match_graph_library():
    rng = np.random.default_rng(7)
    parent, _ = T.random_bfs_tree(rng, 60, 5)
    n = len(parent)
    G = nx.DiGraph()
    G.add_edges_from((int(parent[i]), i) for i in range(1, n))
    leaves = sorted(v for v in G.nodes if G.out_degree(v) == 0)
    expect = [nx.shortest_path(G, 0, v) for v in leaves]
    assert oracle.root_to_leaf_paths(parent, n) == expect


def test_validate_rejects_bad_trees():
    assert not oracle.validate_tree(np.array([0, 0]), 2)          # root not -1
    assert not oracle.validate_tree(np.array([-1, 1]), 2)         # self parent
    assert not oracle.validate_tree(np.array([-1, 2, 0]), 3)      # parent after child
    assert not oracle.validate_tree(np.array([-1, -1]), 2)        # second root
    assert not oracle.validate_tree(np.array([-1, 0]), 0)         # empty
    assert oracle.validate_tree(np.array([-1, 0, 1, 1, -1]), 4)   # padding beyond n ignored


def test_children_in_index_order():
    parent = np.array([-1, 0, 0, 1, 0, 1])
    assert oracle.children(parent, 6, 0) == [1, 2, 4]
    assert oracle.children(parent, 6, 1) == [3, 5]
    assert oracle.children(parent, 6, 3) == []

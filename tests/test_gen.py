"""Checks of the synthetic input generator (tree shapes, determinism, layouts)."""

import numpy as np

import oracle
from gen import compact_draft, make_case, trees as T
from gen.bf16 import bf16_bits_to_f32, f32_to_bf16_bits


def test_cartesian_tree_has_18_paths():
    # jisaku glossary "Medusa", tree candidate section: top-3 x top-3 x top-2 -> up to 18 paths
    parent, _ = T.cartesian_tree((3, 3, 2))
    assert len(oracle.root_to_leaf_paths(parent, len(parent))) == 18
    assert len(parent) == 1 + 3 + 9 + 18


def test_static_63_tree_is_prefix_closed_with_expected_levels():
    parent, rank = T.static_topk_tree((3, 3, 2, 2, 1), 63)
    assert oracle.validate_tree(parent, 63)
    assert np.bincount(T.depths(parent)).tolist() == [1, 3, 8, 14, 23, 14]
    assert (rank[1:4] == [0, 1, 2]).all()
    assert (T.sibling_rank(parent) == rank).all()  # siblings are ordered by rank


def test_bfs_trees_valid_and_depth_limited():
    rng = np.random.default_rng(0)
    for n, dmax in ((127, 6), (255, 8), (10, 1)):
        parent, rank = T.random_bfs_tree(rng, n, dmax)
        assert oracle.validate_tree(parent, len(parent))
        assert T.depths(parent).max() <= dmax and len(parent) <= n
        assert (T.sibling_rank(parent) == rank).all()


def test_bf16_rounding_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 3.0e38], dtype=np.float32)
    back = bf16_bits_to_f32(f32_to_bf16_bits(x))
    assert back[0] == 1.0 and back[1] == 1.0            # tie -> even
    assert back[2] == np.float32(1.0 + 2 ** -7)         # above half -> up
    assert back[3] == -2.5 and np.isfinite(back[4])


def test_make_case_deterministic_and_shaped():
    kw = dict(dtype="bf16", Hq=4, Hkv=2, d=64, Hd=128, V=300, prefix_len=[7, 0],
              parents=[T.tree_root_3x2(), T.chain_tree(4)], rule="rejection", tau=0.7,
              tokens=("iid", 0.7, 0.5), seed=5)
    a, b = make_case(**kw), make_case(**kw)
    for name in ("q", "k_cache", "v_cache", "hidden", "W", "tokens", "draft_probs", "parent"):
        assert (getattr(a, name) == getattr(b, name)).all()
    assert a.q.shape == (2, 10, 4, 64) and a.k_cache.shape == (2, 2, a.L_cap, 64)
    assert a.L_cap == 17 and list(a.n_nodes) == [10, 4]
    assert (a.parent[1, 4:] == -1).all()
    assert a.draft_probs.shape == (2, 10, 300)
    # internal nodes have a draft row, tokens of their children lie in its support
    for bb in range(2):
        for c in range(1, a.n_nodes[bb]):
            assert a.draft_probs[bb, a.parent[bb, c], a.tokens[bb, c]] > 0


def test_compact_draft_keeps_exactly_the_expanded_rows():
    rng = np.random.default_rng(3)
    parents = [T.random_bfs_tree(rng, 20, 4)[0], T.chain_tree(5), np.array([-1], dtype=np.int32)]
    N, Vd = 20, 7
    parent = np.full((3, N), -1, dtype=np.int32)
    for b, p in enumerate(parents):
        parent[b, : len(p)] = p
    n_nodes = np.array([len(p) for p in parents])
    full = rng.random((3, N, Vd)).astype(np.float32)
    rows, index = compact_draft(full, parent, n_nodes, rng=rng)
    expanded = {(b, int(parent[b, c])) for b in range(3) for c in range(1, n_nodes[b])}
    assert rows.shape == (len(expanded), Vd)
    assert sorted(index[index >= 0].tolist()) == list(range(len(expanded)))
    for b in range(3):
        for e in range(N):
            if (b, e) in expanded:
                assert (rows[index[b, e]] == full[b, e]).all()
            else:
                assert index[b, e] == -1

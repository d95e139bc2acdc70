"""Pins for the oracle's tree attention.

* a single chain is ordinary causal decoding over prefix + chain (library scaled-dot-product
  attention in float64 with a causal mask offset by the prefix);
* a single node is plain decoding over prefix + itself;
* a node's output does not depend on the K/V of non-ancestor nodes;
* GQA: query heads of one group read the same KV head (library attention with repeated K/V);
* LSE against a library logsumexp.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle
from gen import trees as T


def _inputs(rng, B, N, Hq, Hkv, d, L):
    q = rng.standard_normal((B, N, Hq, d))
    k = rng.standard_normal((B, Hkv, L + N, d))
    v = rng.standard_normal((B, Hkv, L + N, d))
    return q, k, v


def _sdpa(q, k, v, mask):
    """Library attention: q [H][n][d], k/v [H][m][d], mask bool [n][m]."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=t(mask)).numpy()


@pytest.mark.parametrize("L,n", [(0, 5), (1, 1), (17, 9), (64, 33)])
def test_chain_equals_causal_attention(L, n):
    rng = np.random.default_rng(L * 100 + n)
    Hq, Hkv, d = 4, 2, 16
    q, k, v = _inputs(rng, 1, n, Hq, Hkv, d, L)
    parent = T.chain_tree(n)[None, :]
    O, LSE = oracle.tree_attention(q, k, v, np.array([L]), np.array([n]), parent)
    causal = np.tril(np.ones((n, L + n), dtype=bool), k=L)
    G = Hq // Hkv
    kk = np.repeat(k[0], G, axis=0)  # [Hq][L+n][d]
    vv = np.repeat(v[0], G, axis=0)
    ref = _sdpa(q[0].transpose(1, 0, 2), kk, vv, causal)  # [Hq][n][d]
    np.testing.assert_allclose(O[0].transpose(1, 0, 2), ref, rtol=1e-12, atol=1e-12)
    for h in range(Hq):
        S = (q[0, :, h] @ kk[h].T) / np.sqrt(d)
        for i in range(n):
            assert abs(LSE[0, i, h] - logsumexp(S[i, : L + i + 1])) < 1e-12


def test_single_node_is_plain_decoding():
    rng = np.random.default_rng(3)
    L, d = 40, 32
    q, k, v = _inputs(rng, 1, 1, 2, 1, d, L)
    O, LSE = oracle.tree_attention(q, k, v, np.array([L]), np.array([1]), np.array([[-1]]))
    ref = _sdpa(q[0].transpose(1, 0, 2), np.repeat(k[0], 2, 0), np.repeat(v[0], 2, 0),
                np.ones((1, L + 1), dtype=bool))
    np.testing.assert_allclose(O[0].transpose(1, 0, 2), ref, rtol=1e-12, atol=1e-12)


def test_non_ancestors_do_not_leak():
    rng = np.random.default_rng(5)
    parent, _ = T.random_bfs_tree(rng, 30, 4)
    n, L, d = len(parent), 11, 8
    q, k, v = _inputs(rng, 1, n, 2, 1, d, L)
    O, _ = oracle.tree_attention(q, k, v, np.array([L]), np.array([n]), parent[None])
    for i in range(n):
        anc = oracle.ancestors_or_self(parent, i)
        k2, v2 = k.copy(), v.copy()
        others = [L + j for j in range(n) if j not in anc]
        k2[0, :, others] += 3.0
        v2[0, :, others] -= 5.0
        O2, _ = oracle.tree_attention(q, k2, v2, np.array([L]), np.array([n]), parent[None])
        np.testing.assert_allclose(O2[0, i], O[0, i], rtol=0, atol=1e-13)
        if others:  # and the mask is not vacuous: an ancestor perturbation does change it
            k3 = k.copy()
            k3[0, :, L + i] += 3.0
            O3, _ = oracle.tree_attention(q, k3, v, np.array([L]), np.array([n]), parent[None])
            assert np.abs(O3[0, i] - O[0, i]).max() > 1e-6


def test_tree_matches_library_attention_with_tree_mask():
    """General tree vs library attention given the graph-built mask; padded nodes are zero."""
    rng = np.random.default_rng(11)
    parents = [T.random_bfs_tree(rng, 20, 4)[0], T.random_bfs_tree(rng, 13, 3)[0]]
    N = 20
    B, Hq, Hkv, d = 2, 8, 2, 16
    Ls = [37, 5]
    L_cap = max(Ls) + N
    q = rng.standard_normal((B, N, Hq, d))
    k = rng.standard_normal((B, Hkv, L_cap, d))
    v = rng.standard_normal((B, Hkv, L_cap, d))
    parent = np.full((B, N), -1)
    for b, p in enumerate(parents):
        parent[b, : len(p)] = p
    nn = np.array([len(p) for p in parents])
    O, LSE = oracle.tree_attention(q, k, v, np.array(Ls), nn, parent, scale=0.3)
    for b in range(B):
        n, L = nn[b], Ls[b]
        mask = np.zeros((n, L + n), dtype=bool)
        mask[:, :L] = True
        for i in range(n):
            j = i
            while j >= 0:
                mask[i, L + j] = True
                j = parent[b, j]
        G = Hq // Hkv
        kk = np.repeat(k[b, :, : L + n], G, 0)
        vv = np.repeat(v[b, :, : L + n], G, 0)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
        ref = F.scaled_dot_product_attention(t(q[b, :n].transpose(1, 0, 2)), t(kk), t(vv),
                                             attn_mask=t(mask), scale=0.3).numpy()
        np.testing.assert_allclose(O[b, :n].transpose(1, 0, 2), ref, rtol=1e-12, atol=1e-12)
        assert (O[b, n:] == 0).all() and (LSE[b, n:] == 0).all()


def test_rows_variant_matches_full():
    rng = np.random.default_rng(2)
    parent = np.array([[-1, 0, 0, 1, 1, 2]])
    q, k, v = _inputs(rng, 1, 6, 4, 2, 8, 9)
    O, LSE = oracle.tree_attention(q, k, v, np.array([9]), np.array([6]), parent)
    rows = [(0, 3, 1), (0, 5, 3), (0, 0, 0)]
    o, l = oracle.tree_attention_rows(q, k, v, np.array([9]), np.array([6]), parent, rows)
    for r, (b, i, h) in enumerate(rows):
        np.testing.assert_allclose(o[r], O[b, i, h], rtol=1e-13, atol=1e-13)
        assert abs(l[r] - LSE[b, i, h]) < 1e-13

"""Tree attention over a KV-cache prefix plus the ancestors of each node (fp64).

[GUIDE] section "並列検証" (parallel verification): the target model scores all candidates in
one forward pass, using the KV cache for the prefix.  [MTP] section "ツリー検証" and [GUIDE]
section "Tree Attention": each node attends only to its ancestors (and itself) within the tree.

For request b, query head h (KV head g = h // (Hq / Hkv), contiguous GQA groups), node i:
    S_j  = scale * <q[b, i, h], k[b, g, j]>   for visible key slots j,
    O    = sum_j softmax(S)_j * v[b, g, j],   LSE = log sum_j exp(S_j)  (natural log),
visible = prefix slots [0, L_b) and tree slots {L_b + a : a in anc(i) + {i}}; scale defaults to
1/sqrt(d).  Padded nodes (i >= n_b) produce zeros.
"""

import numpy as np

from .tree import tree_mask


def _attend(Q, K, Vv, mask, scale):
    """Masked softmax attention for query rows Q [r][d] over keys K/V [n_k][d]; mask [r][n_k]."""
    S = scale * (Q @ K.T)
    S = np.where(mask, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    ell = P.sum(axis=1, keepdims=True)
    O = (P @ Vv) / ell
    lse = (m + np.log(ell))[:, 0]
    return O, lse


def _scale(d, scale):
    return 1.0 / np.sqrt(d) if scale is None or scale <= 0 else float(scale)


def tree_attention(q, k_cache, v_cache, prefix_len, n_nodes, parent, scale=None):
    """Full tree attention.  q [B][N][Hq][d], caches [B][Hkv][L_cap][d] (float64).

    Returns O [B][N][Hq][d] and LSE [B][N][Hq] (float64).
    """
    B, N, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    s = _scale(d, scale)
    O = np.zeros((B, N, Hq, d))
    LSE = np.zeros((B, N, Hq))
    for b in range(B):
        L, n = int(prefix_len[b]), int(n_nodes[b])
        mask = tree_mask(parent[b], n, L)
        for g in range(Hkv):
            K = k_cache[b, g, : L + n]
            Vv = v_cache[b, g, : L + n]
            for h in range(g * G, (g + 1) * G):
                O[b, :n, h], LSE[b, :n, h] = _attend(q[b, :n, h], K, Vv, mask, s)
    return O, LSE


def tree_attention_rows(q, k_cache, v_cache, prefix_len, n_nodes, parent, rows, scale=None):
    """Tree attention for selected (b, i, h) rows only; same definition as ``tree_attention``.

    ``q`` may be any array-like indexable as q[b, i, h]; caches are float64 (or float32 holding
    exact bf16 values, widened here).  Returns (O [r][d], LSE [r]).
    """
    out_o, out_l = [], []
    for b, i, h in rows:
        L, n = int(prefix_len[b]), int(n_nodes[b])
        Hq = q.shape[2]
        Hkv = k_cache.shape[1]
        g = h // (Hq // Hkv)
        d = q.shape[3]
        if i >= n:
            out_o.append(np.zeros(d))
            out_l.append(0.0)
            continue
        mask = tree_mask(parent[b], n, L)[i: i + 1]
        K = np.asarray(k_cache[b, g, : L + n], dtype=np.float64)
        Vv = np.asarray(v_cache[b, g, : L + n], dtype=np.float64)
        Q = np.asarray(q[b, i, h], dtype=np.float64)[None, :]
        o, lse = _attend(Q, K, Vv, mask, _scale(d, scale))
        out_o.append(o[0])
        out_l.append(lse[0])
    return np.array(out_o), np.array(out_l)

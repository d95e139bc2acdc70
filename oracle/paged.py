"""Paged KV-cache layout: a request's logical cache slots scattered over fixed-size blocks of a
shared pool through a per-request block table.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[GLOSS] section "デプロイと運用上の考慮事項": batching requests whose trees differ needs padding
and mask management, and integration with continuous batching.  A paged cache is the plainest
layout for that: pool [num_blocks][Hkv][block_size][d]; request b's logical slot s is row
s % block_size of pool block table[b][s // block_size].  These two functions are the layout's
definition written out; tree attention and compaction on a paged cache are the contiguous
oracle functions applied to the gathered view.
"""

import numpy as np


def gather_paged(pool, table, block_size, L_cap):
    """Contiguous [B][Hkv][L_cap][d] view of every request's logical slots."""
    B = table.shape[0]
    _, Hkv, bs, d = pool.shape
    assert bs == block_size and L_cap <= table.shape[1] * bs
    out = np.zeros((B, Hkv, L_cap, d), dtype=pool.dtype)
    for b in range(B):
        for s in range(L_cap):
            out[b, :, s, :] = pool[table[b, s // bs], :, s % bs, :]
    return out


def scatter_paged(cache, pool, table, block_size):
    """Write a contiguous [B][Hkv][L][d] cache into the pool blocks its table names (in place)."""
    B, Hkv, L, d = cache.shape
    for b in range(B):
        for s in range(L):
            pool[table[b, s // block_size], :, s % block_size, :] = cache[b, :, s, :]
    return pool

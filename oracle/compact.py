"""KV compaction after acceptance.

[GUIDE] section "棄却サンプリング" (caution box): every candidate after a rejected one is
discarded; the accepted prefix stays.  [MTP] opening section: decoding re-reads the KV cache
from HBM every step, so the accepted tree entries must end up contiguous after the prefix.  The
pages do not name this step; compaction is the plain reading of "keep the accepted part".

For request b with prefix length L and accepted path (root first, accept_len + 1 nodes):
    new slot L + j receives the K/V of old slot L + path[j], for j = 0 .. accept_len,
    src_slot[j] = L + path[j],  new_len = L + 1 + accept_len.
All reads come from the cache as it was before the call (the move is a gather).  Works on raw
element arrays of any dtype, so bf16 bit patterns are compared bit for bit.
"""

import numpy as np


def compact_kv(k_cache, v_cache, prefix_len, paths, accept_len, path_cap):
    """Returns (k_new, v_new, src_slot [B][path_cap] (-1 padded), new_len [B])."""
    k_new = k_cache.copy()
    v_new = v_cache.copy()
    B = k_cache.shape[0]
    src = np.full((B, path_cap), -1, dtype=np.int64)
    new_len = np.zeros(B, dtype=np.int64)
    for b in range(B):
        L = int(prefix_len[b])
        n = int(accept_len[b]) + 1
        for j in range(n):
            s = L + int(paths[b][j])
            src[b, j] = s
            k_new[b, :, L + j] = k_cache[b, :, s]
            v_new[b, :, L + j] = v_cache[b, :, s]
        new_len[b] = L + n
    return k_new, v_new, src, new_len

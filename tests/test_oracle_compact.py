"""Pins for the oracle's KV compaction (exact index identity, in-place overlap)."""

import numpy as np

from oracle import compact_kv


def test_compaction_moves_path_rows():
    B, H, L_cap, d = 2, 3, 20, 4
    k = np.arange(B * H * L_cap * d, dtype=np.uint16).reshape(B, H, L_cap, d)
    v = (k + 7).astype(np.uint16)
    prefix = np.array([5, 9])
    paths = [[0, 2, 3, 6], [0]]
    alen = np.array([3, 0])
    k2, v2, src, new_len = compact_kv(k, v, prefix, paths, alen, path_cap=6)
    assert list(new_len) == [9, 10]
    assert src[0].tolist() == [5, 7, 8, 11, -1, -1] and src[1].tolist() == [9, -1, -1, -1, -1, -1]
    for j, p in enumerate(paths[0]):
        assert (k2[0, :, 5 + j] == k[0, :, 5 + p]).all() and (v2[0, :, 5 + j] == v[0, :, 5 + p]).all()
    # slots outside the compacted range are untouched (the overlapping reads use old contents)
    untouched = [s for s in range(L_cap) if not 5 <= s < 9]
    assert (k2[0][:, untouched] == k[0][:, untouched]).all()
    assert (k2[1] == k[1]).all()


def test_full_chain_is_identity():
    k = np.random.default_rng(0).integers(0, 60000, (1, 2, 12, 8)).astype(np.uint16)
    k2, _, _, new_len = compact_kv(k, k, np.array([4]), [[0, 1, 2, 3]], np.array([3]), 5)
    assert (k2 == k).all() and new_len[0] == 8

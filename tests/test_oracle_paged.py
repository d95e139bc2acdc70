"""Pins of the paged-cache layout helpers (the definition of the layout, written out)."""

import numpy as np

import oracle


def test_hand_example():
    # two requests, blocks of 2 slots, pool of 5 blocks, one KV head, d = 1
    pool = np.arange(5 * 1 * 2 * 1, dtype=np.float64).reshape(5, 1, 2, 1)  # block k holds 2k, 2k+1
    table = np.array([[3, 0], [1, 4]], dtype=np.int32)
    got = oracle.gather_paged(pool, table, 2, 4)
    assert got[0, 0, :, 0].tolist() == [6, 7, 0, 1]
    assert got[1, 0, :, 0].tolist() == [2, 3, 8, 9]


def test_round_trip_and_untouched_blocks():
    rng = np.random.default_rng(0)
    B, Hkv, bs, d, mb = 3, 2, 4, 8, 5
    nb = B * mb + 3
    table = rng.permutation(nb)[: B * mb].reshape(B, mb).astype(np.int32)
    cache = rng.standard_normal((B, Hkv, mb * bs, d))
    pool = np.full((nb, Hkv, bs, d), 7.0)
    oracle.scatter_paged(cache, pool, table, bs)
    assert (oracle.gather_paged(pool, table, bs, mb * bs) == cache).all()
    unused = sorted(set(range(nb)) - set(table.ravel().tolist()))
    assert (pool[unused] == 7.0).all()

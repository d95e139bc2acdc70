"""GPU parity of tree attention (through the C ABI) against the fp64 oracle."""

import numpy as np
import pytest

import oracle
from gen import make_case, make_config_case, trees as T
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def test_tiny_fp32_config():
    d = H.dev()
    case = H.config_case(1, 0)
    t = H.to_device(case, d)
    o, l, status = H.gpu_attention(case, t)
    assert status == 0
    H.check_attention(case, o, l)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [
    # (tree sizes, prefixes, Hq, Hkv, d)
    ([1], [0], 4, 1, 64),          # single root, empty prefix: plain decoding of one token
    ([2], [1], 8, 8, 128),         # G = 1
    ([33], [127], 8, 2, 64),       # ragged tile edges
    ([255], [129], 4, 1, 128),     # maximum tree, 1020 rows per KV head
    ([10, 63, 1], [200, 0, 65], 16, 2, 128),  # ragged batch, padded nodes
    ([40, 7], [70, 300], 12, 4, 128),  # G = 3: Q rows staged through registers (3 does not divide 128)
    ([5], [100], 128, 1, 64),      # G = 128: one node per 128-row group
])
def test_small_shapes(dtype, shape):
    d = H.dev()
    sizes, prefixes, Hq, Hkv, hd = shape
    rng = np.random.default_rng(sum(sizes) + hd)
    parents = [T.random_bfs_tree(rng, n, 8)[0] if n > 1 else np.array([-1]) for n in sizes]
    case = make_case(dtype=dtype, Hq=Hq, Hkv=Hkv, d=hd, Hd=64, V=16, prefix_len=prefixes, parents=parents,
                     tokens=("given", np.zeros((len(sizes), max(sizes)), dtype=np.int32)), seed=3)
    t = H.to_device(case, d)
    o, l, status = H.gpu_attention(case, t)
    assert status == 0
    H.check_attention(case, o, l)


def test_chain_tree_bf16():
    d = H.dev()
    case = make_case(dtype="bf16", Hq=32, Hkv=8, d=128, Hd=64, V=16, prefix_len=[1000],
                     parents=[T.chain_tree(70)], tokens=("given", np.zeros((1, 70), dtype=np.int32)), seed=5)
    t = H.to_device(case, d)
    o, l, status = H.gpu_attention(case, t)
    assert status == 0
    H.check_attention(case, o, l)


def test_llama8b_b1_l2048_medusa63_full():
    d = H.dev()
    case = H.config_case(2, 0)
    t = H.to_device(case, d)
    o, l, status = H.gpu_attention(case, t)
    assert status == 0
    H.check_attention(case, o, l)


def test_llama8b_b8_ragged_bfs127_full():
    d = H.dev()
    case = H.config_case(3, 1)
    t = H.to_device(case, d)
    o, l, status = H.gpu_attention(case, t)
    assert status == 0
    H.check_attention(case, o, l)


def _sample_rows(case, k, seed):
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(k):
        b = int(rng.integers(0, case.B))
        i = int(rng.integers(0, case.n_nodes[b]))
        h = int(rng.integers(0, case.Hq))
        rows.append((b, i, h))
    # always include the deepest node of each request and a padded row if any
    for b in range(case.B):
        rows.append((b, int(case.n_nodes[b]) - 1, case.Hq - 1))
    return rows


def test_eagle3_b32_l4096_sampled():
    d = H.dev()
    case = H.config_case(4, 2)
    t = H.to_device(case, d)
    o, l, status = H.gpu_attention(case, t)
    assert status == 0
    H.check_attention(case, o, l, rows=_sample_rows(case, 96, 4))


def test_llama70b_b4_long_context_sampled():
    d = H.dev()
    case = H.config_case(5, 3)
    t = H.to_device(case, d)
    o, l, status = H.gpu_attention(case, t)
    assert status == 0
    H.check_attention(case, o, l, rows=_sample_rows(case, 24, 5))
    # every row of the longest request (131072 prefix keys, 255 nodes) on KV head 0: its 8 query
    # heads x 255 nodes against the oracle on that slice of the problem
    b = int(np.argmax(case.prefix_len))
    L, n, G = int(case.prefix_len[b]), int(case.n_nodes[b]), case.Hq // case.Hkv
    q = case.f64("q")[b: b + 1, :, :G]
    kf = np.asarray(case.f32("k_cache")[b: b + 1, :1, : L + n], dtype=np.float64)
    vf = np.asarray(case.f32("v_cache")[b: b + 1, :1, : L + n], dtype=np.float64)
    O, LSE = oracle.tree_attention(q, kf, vf, case.prefix_len[b: b + 1], case.n_nodes[b: b + 1],
                                   case.parent[b: b + 1])
    err = np.abs(o[b: b + 1, :n, :G] - O[:, :n]).max()
    lerr = (np.abs(l[b: b + 1, :n, :G] - LSE[:, :n]) / np.maximum(np.abs(LSE[:, :n]), 1e-6)).max()
    assert L == 131072 and err < H.ATTN_TOL["bf16"] and lerr < H.LSE_RTOL, (err, lerr)
    # padded rows are exactly zero
    for b in range(case.B):
        n = int(case.n_nodes[b])
        if n < case.N:
            assert (o[b, n:] == 0).all() and (l[b, n:] == 0).all()

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


# ---- the persistent stream-K schedule ----------------------------------------------------------

def _align(x):
    return (x + 255) // 256 * 256


def _stream_k_workspace(B, N, Hq, Hkv, d, sms):
    """Workspace bytes of the stream-K path: tree scratch, arrival counters per 256-row block and
    group, and two partial slots of 256 rows per CTA."""
    G = Hq // Hkv
    W = (N + 31) // 32
    blocks = (N * G + 255) // 256
    return (_align(B * N * 4) + _align(B * N * W * 4) + 2 * _align(B * 4) + _align(B * Hkv * blocks * 2 * 4)
            + _align(sms * 2 * 256 * 8) + _align(sms * 2 * 256 * d * 4))


def _run_stream_k(case, d):
    import ctypes
    import torch
    import tree_speculative_decoding_split_gb300 as st
    t = H.to_device(case, d)
    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"],
                                schedule="stream_k")
    sms = torch.cuda.get_device_properties(d).multi_processor_count
    need = st.lib().spec_tree_attention_workspace(ctypes.byref(aa))
    assert need == _stream_k_workspace(case.B, case.N, case.Hq, case.Hkv, case.d, sms), "not the stream-K path"
    status = torch.zeros(1, dtype=torch.int32, device=d)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device=d)  # counters start as garbage
    code = st.lib().spec_tree_attention(ctypes.byref(aa), ctypes.c_void_p(ws.data_ptr()), need,
                                        ctypes.c_void_p(status.data_ptr()),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    return (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            int(status.item()))


@pytest.mark.parametrize("hd,Hq,Hkv", [(128, 8, 2), (64, 4, 4), (128, 16, 2)])
def test_stream_k_few_tiles_in_a_long_cache(hd, Hq, Hkv):
    """Stream-K with short prefixes in a 40000-slot cache: fewer tiles than SMs, so segments split
    into many one-tile pieces that the last arrival merges, including a piece of tree keys only;
    ragged trees with padded nodes, an empty prefix and G = 1 / 4 / 8."""
    d = H.dev()
    rng = np.random.default_rng(hd + Hq)
    parents = [T.random_bfs_tree(rng, n, 6)[0] for n in (37, 5, 60, 1)]
    case = make_case(dtype="bf16", Hq=Hq, Hkv=Hkv, d=hd, Hd=64, V=16, prefix_len=[700, 0, 1300, 64],
                     parents=parents, tokens=("given", np.zeros((4, 60), dtype=np.int32)), seed=13,
                     L_cap=40000)
    o, l, status = _run_stream_k(case, d)
    assert status == 0
    H.check_attention(case, o, l)
    for b in range(case.B):
        assert (o[b, case.n_nodes[b]:] == 0).all() and (l[b, case.n_nodes[b]:] == 0).all()


def test_stream_k_bad_tree_and_capacity_zero_their_rows():
    d = H.dev()
    rng = np.random.default_rng(5)
    good = T.random_bfs_tree(rng, 30, 5)[0]
    bad = good.copy()
    bad[9] = 20  # parent after its child
    case = make_case(dtype="bf16", Hq=8, Hkv=2, d=128, Hd=64, V=16, prefix_len=[3000, 2500, 4000],
                     parents=[good, bad, good], tokens=("given", np.zeros((3, 30), dtype=np.int32)), seed=4,
                     L_cap=30000)
    case.prefix_len[2] = 30000 - 10  # prefix + tree beyond the cache: a capacity error
    o, l, status = _run_stream_k(case, d)
    assert status in (4, 7)  # first error wins: SPEC_ERR_BAD_TREE or SPEC_ERR_CAPACITY
    assert (o[1] == 0).all() and (l[1] == 0).all() and (o[2] == 0).all() and (l[2] == 0).all()
    rows = [(0, i, h) for i in range(30) for h in (0, 3, 7)]
    H.check_attention(case, o, l, rows=rows)


@pytest.mark.parametrize("cfg", [3, 4])
def test_stream_k_on_the_8b_workloads(cfg):
    """The B8 ragged-prefix and B32 workloads under the stream-K schedule, against the oracle
    (all rows at B8, sampled rows at B32)."""
    d = H.dev()
    case = H.config_case(cfg, 1 if cfg == 3 else 2)
    o, l, status = _run_stream_k(case, d)
    assert status == 0
    H.check_attention(case, o, l, rows=None if cfg == 3 else _sample_rows(case, 96, 4))

"""GPU parity of the static Medusa tree expansion (spec_medusa_expand) with the oracle, bit for
bit: every head's top-k (ties to the lower id), every node's token, and the shared topology."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_split_gb300 as st
from gen import bf16 as BF, make_case
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _logits(rng, B, K, V, dtype, ties):
    x = rng.standard_normal((B, K, V)).astype(np.float32)
    if ties:
        x = np.round(x * 4) / 4  # many equal logits
    if dtype == "bf16":
        return BF.f32_to_bf16_bits(x)  # bit patterns (uint16)
    return x


def _run(x, dtype, parent, rank, topk, root=None):
    d = H.dev()
    t = H.tensor(x, d, dtype == "bf16")
    tp = torch.from_numpy(parent).to(d)
    tr = torch.from_numpy(rank).to(d)
    rt = None if root is None else torch.from_numpy(np.asarray(root, dtype=np.int32)).to(d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    out = st.medusa_expand(t, tp, tr, topk, root_token=rt, dev_status=status)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["status"] = int(status.item())
    return res


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V,topk_heads,n", [(128256, (3, 3, 2, 2, 1), 63), (30011, (4, 4, 3, 2, 2), 127),
                                             (1000, (10, 8, 6, 4, 2), 255), (50, (32, 2), 40)])
def test_expand_matches_oracle(dtype, V, topk_heads, n):
    rng = np.random.default_rng(V + n)
    B, K = 3, len(topk_heads)
    k = max(topk_heads)
    x = _logits(rng, B, K, V, dtype, ties=(V < 40000))
    parent, rank = st.medusa_topology(topk_heads, n)
    root = rng.integers(0, V, size=B)
    got = _run(x, dtype, parent, rank, k, root)
    assert got["status"] == 0
    xf = BF.bf16_bits_to_f64(x) if dtype == "bf16" else x.astype(np.float64)
    tokens, idx = oracle.medusa_expand(xf, parent, rank, k, root_token=root)
    assert (got["topk_index"] == idx).all()
    assert (got["tokens"] == tokens).all()
    assert (got["parent"] == np.tile(parent, (B, 1))).all() and (got["n_nodes"] == n).all()


def test_special_values_order():
    """-0 equals +0 (lower id first), NaN ranks below -inf, +inf on top."""
    x = np.zeros((1, 1, 8), dtype=np.float32)
    x[0, 0] = [-0.0, np.nan, 0.0, -np.inf, np.inf, 1.0, np.nan, -np.inf]
    parent, rank = st.medusa_topology((8,), 9)
    got = _run(x, "f32", parent, rank, 8)
    assert got["status"] == 0
    assert got["topk_index"][0, 0].tolist() == [4, 5, 0, 2, 3, 7, 1, 6]


def test_bad_topology_sets_status_and_zeroes_tokens():
    rng = np.random.default_rng(3)
    x = _logits(rng, 2, 2, 100, "f32", False)
    parent, rank = st.medusa_topology((3, 3, 2), 20)  # depth 3 with only two heads
    got = _run(x, "f32", parent, rank, 3)
    assert got["status"] == 4 and (got["tokens"] == 0).all()
    parent, rank = st.medusa_topology((3, 3), 8)
    rank = rank.copy()
    rank[4] = 3  # rank beyond topk
    got = _run(x, "f32", parent, rank, 3)
    assert got["status"] == 4


def test_expanded_tree_feeds_typical_acceptance():
    """Medusa drafting end to end: the expanded tree goes straight into spec_verify_accept."""
    d = H.dev()
    rng = np.random.default_rng(11)
    V, Hd = 4096, 256
    parent, rank = st.medusa_topology((3, 3, 2, 2, 1), 63)
    case = make_case(dtype="bf16", Hq=4, Hkv=1, d=64, Hd=Hd, V=V, prefix_len=[8] * 2, parents=[parent, parent],
                     rule="typical", tau=1.0, eps=0.09, delta=0.3, seed=7, tokens=("rank", 0.9), rng=rng)
    heads = _logits(rng, 2, 5, V, "bf16", False)
    got = _run(heads, "bf16", parent, rank, 3)
    assert got["status"] == 0
    case.tokens[:] = got["tokens"]
    out = H.gpu_verify(case, H.to_device(case, d))
    assert out["status"] == 0
    ref = H.oracle_verify(case)
    c = H.check_verify(case, out, ref)
    assert c.exact + c.excluded == 2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("topk_heads", [(12, 8, 3), (8, 5, 3)])
def test_plateaus_and_constant_rows(dtype, topk_heads):
    """Rows whose top values tie over hundreds of entries: a constant head (every chunk takes the
    per-warp register path, since more keys reach the threshold than shared memory gathers), a
    head with a 700-entry plateau at its maximum, and a random head; k above 8 (threshold from
    the threads' maxima) and k = 8 (from the warps' maxima)."""
    rng = np.random.default_rng(11)
    B, V = 2, 128256
    k = max(topk_heads)
    x = rng.standard_normal((B, 3, V)).astype(np.float32)
    x[:, 0] = 0.5
    x[:, 1, 4000:4700] = 9.0
    x[1, 1, 70001:70301] = 9.0
    xs = BF.f32_to_bf16_bits(x) if dtype == "bf16" else x
    parent, rank = st.medusa_topology(topk_heads, 60)
    got = _run(xs, dtype, parent, rank, k)
    assert got["status"] == 0
    xf = BF.bf16_bits_to_f64(xs) if dtype == "bf16" else xs.astype(np.float64)
    tokens, idx = oracle.medusa_expand(xf, parent, rank, k)
    assert (got["topk_index"] == idx).all()
    assert (got["tokens"] == tokens).all()
    assert idx[0, 0].tolist() == list(range(k))  # a constant row: the lowest ids


def test_expansion_captured_in_a_graph():
    """The expansion's merge launches as a programmatic dependent of the chunk kernel; captured
    into a CUDA graph and replayed (twice, the logits refilled in between) it gives what direct
    calls give."""
    d = H.dev()
    rng = np.random.default_rng(99)
    topk_heads = (3, 3, 2, 2, 1)
    parent, rank = st.medusa_topology(topk_heads, 63)
    x1, x2 = (BF.f32_to_bf16_bits(rng.standard_normal((2, 5, 128256)).astype(np.float32)) for _ in range(2))
    logits = H.tensor(x1, d, True)
    tp, tr = torch.from_numpy(parent).to(d), torch.from_numpy(rank).to(d)
    ma, outs = st.medusa_args(logits, tp, tr, 3)
    L = st.lib()
    need = L.spec_medusa_expand_workspace(ctypes.byref(ma))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        code = L.spec_medusa_expand(ctypes.byref(ma), ctypes.c_void_p(ws.data_ptr()), need,
                                    ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(s.cuda_stream))
    assert code == 0
    for x in (x1, x2):
        logits.copy_(H.tensor(x, d, True))
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.clone() for k, v in outs.items()}
        ref = st.medusa_expand(H.tensor(x, d, True), tp, tr, 3)
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(got[k], ref[k]), k
    assert int(status.item()) == 0

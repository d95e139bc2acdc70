"""GPU parity of KV compaction (bit-exact) and of the device-side error paths."""

import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_split_gb300 as st
from gen import make_case, trees as T
import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,hd", [("bf16", 128), ("f32", 64), ("bf16", 64)])
def test_compaction_bit_exact(dtype, hd):
    d = H.dev()
    rng = np.random.default_rng(hd)
    B, Hkv, path_cap = 6, 3, 12
    parents = [T.random_bfs_tree(rng, int(n), 9)[0] for n in rng.integers(1, 60, B)]
    case = make_case(dtype=dtype, Hq=Hkv, Hkv=Hkv, d=hd, Hd=64, V=16, prefix_len=rng.integers(0, 300, B),
                     parents=parents, tokens=("given", np.zeros((B, 60), dtype=np.int32)), N=60, seed=1)
    paths = []
    for b in range(B):
        n = int(case.n_nodes[b])
        e = int(rng.integers(0, n))
        p = [e]
        while p[-1] != 0:
            p.append(int(case.parent[b, p[-1]]))
        paths.append(p[::-1][:path_cap])
    alen = np.array([len(p) - 1 for p in paths], dtype=np.int32)
    path_arr = np.full((B, path_cap), -1, dtype=np.int32)
    for b, p in enumerate(paths):
        path_arr[b, : len(p)] = p
    kr, vr, src, new_len = oracle.compact_kv(case.k_cache, case.v_cache, case.prefix_len, paths, alen, path_cap)
    t = H.to_device(case, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    s_slot, n_len = st.compact_kv(t["k"], t["v"], t["prefix_len"], H.tensor(path_arr, d), H.tensor(alen, d),
                                  dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    view = np.int16 if dtype == "bf16" else np.float32
    kg = t["k"].view(torch.int16).cpu().numpy() if dtype == "bf16" else t["k"].cpu().numpy()
    vg = t["v"].view(torch.int16).cpu().numpy() if dtype == "bf16" else t["v"].cpu().numpy()
    assert (kg == kr.view(view)).all() and (vg == vr.view(view)).all()
    assert (s_slot.cpu().numpy() == src).all() and (n_len.cpu().numpy() == new_len).all()


def test_bad_trees_and_capacity_set_status_and_zero_outputs():
    d = H.dev()
    rng = np.random.default_rng(0)
    good = T.random_bfs_tree(rng, 12, 4)[0]
    bad = good.copy()
    bad[5] = 7  # parent after child
    case = make_case(dtype="bf16", Hq=4, Hkv=1, d=64, Hd=64, V=100, prefix_len=[10, 10], parents=[good, bad],
                     rule="greedy", tau=0.0, seed=2, tokens=("rank", 0.7))
    t = H.to_device(case, d)
    o, l, status = H.gpu_attention(case, t)
    assert status == 4  # SPEC_ERR_BAD_TREE
    assert (o[1] == 0).all() and (l[1] == 0).all()
    H.check_attention(case.__class__(**{**case.__dict__, "B": 1, "q": case.q[:1], "k_cache": case.k_cache[:1],
                                        "v_cache": case.v_cache[:1], "prefix_len": case.prefix_len[:1],
                                        "n_nodes": case.n_nodes[:1], "parent": case.parent[:1]}), o[:1], l[:1])
    got = H.gpu_verify(case, t)
    assert got["status"] == 4
    assert got["accept_len"][1] == 0 and got["bonus_token"][1] == -1 and got["path"][1, 0] == 0
    assert (got["path"][1, 1:] == -1).all()
    # capacity: prefix + nodes beyond L_cap (request 1 repaired first: one error per call)
    t["parent"][1] = t["parent"][0]
    t["prefix_len"][0] = case.L_cap
    _, _, status = H.gpu_attention(case, t)
    assert status == 7  # SPEC_ERR_CAPACITY
    # token outside the vocabulary
    t = H.to_device(case, d)
    t["parent"][1] = t["parent"][0]
    t["tokens"][0, 3] = 100
    got = H.gpu_verify(case, t)
    assert got["status"] == 6  # SPEC_ERR_BAD_TOKEN
    assert got["bonus_token"][0] == -1
    # a path longer than path_cap
    t = H.to_device(case, d)
    t["parent"][1] = t["parent"][0]
    chain = make_case(dtype="bf16", Hq=4, Hkv=1, d=64, Hd=64, V=100, prefix_len=[1], parents=[T.chain_tree(9)],
                      rule="typical", tau=1.0, eps=0.0, delta=0.0, seed=2, tokens=("rank", 0.7))
    got = H.gpu_verify(chain, H.to_device(chain, d), path_cap=4)  # thr 0 accepts all 8 levels
    assert got["status"] == 7 and got["accept_len"][0] == 0


def test_host_errors_raise():
    d = H.dev()
    case = make_case(dtype="bf16", Hq=4, Hkv=1, d=64, Hd=64, V=100, prefix_len=[10], parents=[T.chain_tree(3)],
                     rule="greedy", tau=0.0, seed=2, tokens=("rank", 0.7))
    t = H.to_device(case, d)
    with pytest.raises(st.SpecError) as e:
        st.verify_accept(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], "typical", 0.0)
    assert e.value.code == 1
    import ctypes
    a, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    L = st.lib()
    need = L.spec_tree_attention_workspace(ctypes.byref(a))
    ws = torch.empty(need, dtype=torch.uint8, device=d)
    code = L.spec_tree_attention(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), need - 1, None, None)
    assert code == 3  # SPEC_ERR_WORKSPACE_TOO_SMALL, returned before any launch

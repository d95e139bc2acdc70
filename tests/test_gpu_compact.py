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


def _fused_vs_separate(case, d, block_table=None):
    """spec_verify_accept_compact against spec_verify_accept followed by spec_compact_kv, on two
    copies of the same inputs: every output and both caches bit for bit."""
    t1, t2 = H.to_device(case, d), H.to_device(case, d)
    s1 = torch.zeros(1, dtype=torch.int32, device=d)
    s2 = torch.zeros(1, dtype=torch.int32, device=d)
    r1 = st.verify_accept(t1["hidden"], t1["W"], t1["tokens"], t1["parent"], t1["n_nodes"], case.rule, case.tau,
                          case.eps, case.delta, case.seed, draft_probs=t1["draft"], draft_to_target=t1["map"],
                          path_cap=case.N, dev_status=s1)
    src1, nl1 = st.compact_kv(t1["k"], t1["v"], t1["prefix_len"], r1["path"], r1["accept_len"], dev_status=s1)
    r2 = st.verify_accept_compact(t2["hidden"], t2["W"], t2["tokens"], t2["parent"], t2["n_nodes"], case.rule,
                                  t2["k"], t2["v"], t2["prefix_len"], case.tau, case.eps, case.delta, case.seed,
                                  draft_probs=t2["draft"], draft_to_target=t2["map"], path_cap=case.N, dev_status=s2)
    torch.cuda.synchronize()
    assert int(s1.item()) == int(s2.item())
    for key in ("accept_len", "path", "bonus_token", "margin_count", "bonus_margin"):
        assert torch.equal(r1[key], r2[key]), key
    assert torch.equal(src1, r2["src_slot"]) and torch.equal(nl1, r2["new_len"])
    for name in ("k", "v"):
        a, b = t1[name], t2[name]
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), name
    return r2, int(s2.item())


@pytest.mark.parametrize("rule,dtype,V", [("greedy", "bf16", 3000), ("typical", "f32", 2000),
                                          ("rejection", "bf16", 5000), ("rejection", "bf16", 300001),
                                          ("typical", "bf16", 30011)])
def test_verify_with_folded_compaction_matches_separate_calls(rule, dtype, V):
    """Greedy / typical fold the compaction into the last row block of each request, rejection into
    the end of the walk (clusters of CTAs at V = 5000, one CTA per request at V = 300001); the
    oracle pins the separate calls (test_compaction_bit_exact and the verify tests)."""
    d = H.dev()
    rng = np.random.default_rng(V)
    parents = [T.random_bfs_tree(rng, 40, 6)[0], T.chain_tree(12), T.random_bfs_tree(rng, 25, 3)[0]]
    case = make_case(dtype=dtype, Hq=4, Hkv=3, d=64 if dtype == "f32" else 128, Hd=128, V=V,
                     prefix_len=[17, 300, 0], parents=parents, rule=rule, tau=0.0 if rule == "greedy" else 0.9,
                     eps=0.09, delta=0.3, seed=V + 3,
                     tokens=("iid", 0.8, 0.4) if rule == "rejection" else ("rank", 0.9), rng=rng)
    r, status = _fused_vs_separate(case, d)
    assert status == 0
    ref = H.oracle_verify(case)
    H.check_verify(case, {k: v.cpu().numpy() for k, v in r.items()}, ref)


def test_folded_compaction_on_a_bad_tree_and_a_short_path_capacity():
    d = H.dev()
    rng = np.random.default_rng(3)
    good = T.random_bfs_tree(rng, 20, 4)[0]
    bad = good.copy()
    bad[7] = 15
    case = make_case(dtype="bf16", Hq=4, Hkv=2, d=128, Hd=128, V=1000, prefix_len=[9, 9], parents=[good, bad],
                     rule="greedy", tau=0.0, seed=1, tokens=("rank", 0.9), rng=rng)
    r, status = _fused_vs_separate(case, d)
    assert status == 4  # SPEC_ERR_BAD_TREE
    assert int(r["accept_len"][1]) == 0 and int(r["new_len"][1]) == 10

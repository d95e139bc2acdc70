"""Paged KV cache (block tables): tree attention against the oracle on the gathered logical view,
and KV compaction bit for bit, for every supported block size, with shared prefix blocks, a bad
table entry, and a context long enough that a CTA reads its table entries from global memory."""

import math

import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_split_gb300 as st
from gen import make_case, trees as T
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _pool(case, bs, rng, extra=7, share=0):
    """Scatter the case's contiguous caches into shuffled pool blocks; the first ``share`` blocks
    of request 1 are request 0's blocks (their contents must then be equal)."""
    B, Hkv, L_cap, d = case.k_cache.shape
    mb = math.ceil(L_cap / bs)
    nb = B * mb + extra
    table = rng.permutation(nb)[: B * mb].reshape(B, mb).astype(np.int32)
    if share:
        table[1, :share] = table[0, :share]
    kc = np.zeros((B, Hkv, mb * bs, d), dtype=case.k_cache.dtype)
    vc = np.zeros_like(kc)
    kc[:, :, :L_cap] = case.k_cache
    vc[:, :, :L_cap] = case.v_cache
    pk = np.zeros((nb, Hkv, bs, d), dtype=kc.dtype)
    pv = np.zeros_like(pk)
    oracle.scatter_paged(kc, pk, table, bs)
    oracle.scatter_paged(vc, pv, table, bs)
    return table, pk, pv


def _attend(case, table, pk, pv, d):
    t = H.to_device(case, d)
    bf = case.dtype == "bf16"
    status = torch.zeros(1, dtype=torch.int32, device=d)
    out, lse = st.tree_attention(t["q"], H.tensor(pk, d, bf), H.tensor(pv, d, bf), t["prefix_len"], t["n_nodes"],
                                 t["parent"], dev_status=status, block_table=H.tensor(table, d))
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), int(status.item())


def _case(rng, B, prefix, n_tree, G=4, Hkv=2, dd=128):
    parents = [T.random_bfs_tree(rng, n_tree, 6)[0] for _ in range(B)]
    return make_case(dtype="bf16", Hq=G * Hkv, Hkv=Hkv, d=dd, Hd=64, V=16, prefix_len=prefix, parents=parents,
                     tokens=("given", np.zeros((B, n_tree), dtype=np.int32)), N=n_tree, seed=int(rng.integers(1 << 30)),
                     rng=rng)


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
def test_paged_attention_matches_oracle(bs):
    d = H.dev()
    rng = np.random.default_rng(bs)
    case = _case(rng, 3, [777, 3, 2100], 40)
    table, pk, pv = _pool(case, bs, rng)
    o, l, status = _attend(case, table, pk, pv, d)
    assert status == 0
    H.check_attention(case, o, l)


def test_shared_prefix_blocks():
    d = H.dev()
    rng = np.random.default_rng(5)
    case = _case(rng, 2, [640, 640], 30, dd=64)
    case.k_cache[1, :, :640] = case.k_cache[0, :, :640]  # identical prefixes, one copy in the pool
    case.v_cache[1, :, :640] = case.v_cache[0, :, :640]
    table, pk, pv = _pool(case, 64, rng, share=10)
    o, l, status = _attend(case, table, pk, pv, d)
    assert status == 0
    H.check_attention(case, o, l)


@pytest.mark.parametrize("prefix", [[300, 500, 100], [100, 150, 50]])
def test_bad_table_entry_zeroes_that_request(prefix):
    """Long prefixes run several key splits (the merge zeroes the request); prefixes this short
    fit one split, where the attention kernel writes, and zeroes, the final rows itself."""
    d = H.dev()
    rng = np.random.default_rng(6)
    case = _case(rng, 3, prefix, 20)
    table, pk, pv = _pool(case, 32, rng)
    table[1, 3] = pk.shape[0] + 100
    o, l, status = _attend(case, table, pk, pv, d)
    assert status == 7  # SPEC_ERR_CAPACITY
    assert (o[1] == 0).all() and (l[1] == 0).all()
    keep = [0, 2]
    sub = case.__class__(**{**case.__dict__, "B": 2, "q": case.q[keep], "k_cache": case.k_cache[keep],
                            "v_cache": case.v_cache[keep], "prefix_len": case.prefix_len[keep],
                            "n_nodes": case.n_nodes[keep], "parent": case.parent[keep]})
    H.check_attention(sub, o[keep], l[keep])


def test_long_context_reads_the_table_from_global_memory():
    """600K slots in blocks of 16: each prefix split spans more table entries than a CTA stages."""
    d = H.dev()
    rng = np.random.default_rng(7)
    parents = [T.chain_tree(8)]
    case = make_case(dtype="bf16", Hq=4, Hkv=1, d=128, Hd=64, V=16, prefix_len=[600000], parents=parents,
                     tokens=("given", np.zeros((1, 8), dtype=np.int32)), seed=3, rng=rng)
    table, pk, pv = _pool(case, 16, rng, extra=3)
    o, l, status = _attend(case, table, pk, pv, d)
    assert status == 0
    rows = [(0, i, h) for i in range(8) for h in range(4)]
    H.check_attention(case, o, l, rows=rows)


@pytest.mark.parametrize("dtype,bs", [("bf16", 16), ("f32", 64), ("bf16", 256)])
def test_paged_compaction_bit_exact(dtype, bs):
    d = H.dev()
    rng = np.random.default_rng(bs + len(dtype))
    B, Hkv, path_cap = 4, 2, 12
    parents = [T.random_bfs_tree(rng, int(n), 9)[0] for n in rng.integers(2, 60, B)]
    case = make_case(dtype=dtype, Hq=Hkv, Hkv=Hkv, d=64, Hd=64, V=16, prefix_len=rng.integers(0, 300, B),
                     parents=parents, tokens=("given", np.zeros((B, 60), dtype=np.int32)), N=60, seed=1)
    paths = []
    for b in range(B):
        e = int(rng.integers(0, int(case.n_nodes[b])))
        p = [e]
        while p[-1] != 0:
            p.append(int(case.parent[b, p[-1]]))
        paths.append(p[::-1][:path_cap])
    alen = np.array([len(p) - 1 for p in paths], dtype=np.int32)
    path_arr = np.full((B, path_cap), -1, dtype=np.int32)
    for b, p in enumerate(paths):
        path_arr[b, : len(p)] = p
    kr, vr, src, new_len = oracle.compact_kv(case.k_cache, case.v_cache, case.prefix_len, paths, alen, path_cap)
    table, pk, pv = _pool(case, bs, rng)
    pk0 = pk.copy()
    bf = dtype == "bf16"
    tk, tv = H.tensor(pk, d, bf), H.tensor(pv, d, bf)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    s_slot, n_len = st.compact_kv(tk, tv, H.tensor(case.prefix_len.astype(np.int32), d), H.tensor(path_arr, d),
                                  H.tensor(alen, d), dev_status=status, block_table=H.tensor(table, d))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    view = np.int16 if bf else np.float32
    gk = tk.view(torch.int16).cpu().numpy() if bf else tk.cpu().numpy()
    gv = tv.view(torch.int16).cpu().numpy() if bf else tv.cpu().numpy()
    L_cap = case.k_cache.shape[2]
    assert (oracle.gather_paged(gk, table, bs, L_cap) == kr.view(view)).all()
    assert (oracle.gather_paged(gv, table, bs, L_cap) == vr.view(view)).all()
    unused = sorted(set(range(pk.shape[0])) - set(table.ravel().tolist()))
    assert (gk[unused] == pk0[unused].view(view)).all()
    assert (s_slot.cpu().numpy() == src).all() and (n_len.cpu().numpy() == new_len).all()
    # an entry out of range among the touched blocks: CAPACITY, nothing moved for that request
    table2 = table.copy()
    L0 = int(case.prefix_len[0])
    table2[0, L0 // bs] = -3
    before = tk.clone()
    status.zero_()
    st.compact_kv(tk, tv, H.tensor(case.prefix_len.astype(np.int32), d), H.tensor(path_arr, d), H.tensor(alen, d),
                  dev_status=status, block_table=H.tensor(table2, d))
    torch.cuda.synchronize()
    assert int(status.item()) == 7
    after = tk.view(torch.int16).cpu().numpy() if bf else tk.cpu().numpy()
    was = before.view(torch.int16).cpu().numpy() if bf else before.cpu().numpy()
    assert (oracle.gather_paged(after, table[:1], bs, L_cap) == oracle.gather_paged(was, table[:1], bs, L_cap)).all()


def test_paged_round_matches_direct_calls():
    """The captured round on a paged pool -- tree attention and verification as parallel branches,
    compaction after both -- gives the three direct calls' outputs and pool, bit for bit (the
    compaction rewrites pool rows the attention reads, so it must not overtake it)."""
    d = H.dev()
    rng = np.random.default_rng(5)
    parents = [T.random_bfs_tree(rng, 40, 6)[0] for _ in range(3)]
    case = make_case(dtype="bf16", Hq=8, Hkv=2, d=128, Hd=64, V=16, prefix_len=[500, 7, 1300], parents=parents,
                     tokens=("rank", 0.95), N=40, seed=11, rng=rng)  # drafts close to the target: paths accepted
    table, pk, pv = _pool(case, 32, rng)

    def fresh():
        t = H.to_device(case, d)
        return t, H.tensor(pk, d, True), H.tensor(pv, d, True), H.tensor(table, d)

    # the direct calls
    t, tk, tv, tab = fresh()
    out, lse = st.tree_attention(t["q"], tk, tv, t["prefix_len"], t["n_nodes"], t["parent"], block_table=tab)
    outs = st.verify_accept(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], "greedy", path_cap=case.N)
    src, nl = st.compact_kv(tk, tv, t["prefix_len"], outs["path"], outs["accept_len"], block_table=tab)
    torch.cuda.synchronize()
    ref = {"out": out.clone(), "lse": lse.clone(), "src": src.clone(), "nl": nl.clone(), "k": tk.clone(),
           "v": tv.clone(), **{k: v.clone() for k, v in outs.items()}}
    # the round on a fresh copy of everything
    t, tk, tv, tab = fresh()
    aa, out, lse = st.attn_args(t["q"], tk, tv, t["prefix_len"], t["n_nodes"], t["parent"], block_table=tab)
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], "greedy",
                              path_cap=case.N)
    ca, src, nl = st.compact_args(tk, tv, t["prefix_len"], outs["path"], outs["accept_len"], block_table=tab)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    r = st.Round(aa, va, ca, dev_status=status)
    r.launch()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = {"out": out, "lse": lse, "src": src, "nl": nl, "k": tk, "v": tv, **outs}
    for k, v in ref.items():
        a, b = got[k], v
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), k
    assert int(ref["accept_len"].max().item()) >= 1, "no request accepted a node: the compaction was not exercised"
    r.close()


def test_paged_matches_contiguous_at_70b_shapes():
    """70B-shaped attention (Hq 64, Hkv 8, d 128, 255-node BFS trees) at batch 4 with 8192-slot
    prefixes, from a shuffled pool of 16-slot blocks (V rows arriving one box per block) and from
    the contiguous caches: the same outputs within the bf16 tolerance and LSE within 1e-3."""
    d = H.dev()
    rng = np.random.default_rng(3)
    B, n = 4, 255
    parents = [T.random_bfs_tree(rng, n, 8)[0] for _ in range(B)]
    case = make_case(dtype="bf16", Hq=64, Hkv=8, d=128, Hd=64, V=16, prefix_len=[8192] * B, parents=parents,
                     tokens=("given", np.zeros((B, n), dtype=np.int32)), N=n, seed=4, rng=rng)
    t = H.to_device(case, d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    out_c, lse_c = st.tree_attention(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"],
                                     dev_status=status)
    table, pk, pv = _pool(case, 16, rng)
    out_p, lse_p = st.tree_attention(t["q"], H.tensor(pk, d, True), H.tensor(pv, d, True), t["prefix_len"],
                                     t["n_nodes"], t["parent"], dev_status=status, block_table=H.tensor(table, d))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert (out_c.float() - out_p.float()).abs().max().item() < 2e-2
    assert ((lse_c - lse_p).abs() / lse_c.abs().clamp_min(1.0)).max().item() < 1e-3

"""The CUDA-graph verification round (spec_round_create / spec_round_launch) against the three
direct calls: the same kernels run, so every output must match bit for bit, also after the
inputs are refilled in place and the round is launched again."""

import numpy as np
import pytest
import torch

import tree_speculative_decoding_split_gb300 as st
from gen import compact_draft, make_case, trees as T
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _case(rule, seed):
    rng = np.random.default_rng(seed)
    parents = [T.random_bfs_tree(rng, 30, 4)[0], T.chain_tree(9)]
    return make_case(dtype="bf16", Hq=8, Hkv=2, d=128, Hd=256, V=20000, prefix_len=[300, 41], parents=parents,
                     rule=rule, tau=0.0 if rule == "greedy" else 0.8, eps=0.09, delta=0.3, seed=seed,
                     tokens=("iid", 0.8, 0.5) if rule == "rejection" else ("rank", 0.9), rng=rng)


def _direct(case, t):
    status = torch.zeros(1, dtype=torch.int32, device=t["q"].device)
    out, lse = st.tree_attention(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"], dev_status=status)
    res = st.verify_accept(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                           case.eps, case.delta, case.seed, draft_probs=t["draft"], draft_to_target=t["map"],
                           path_cap=case.N, hooks=True, dev_status=status)
    src, nl = st.compact_kv(t["k"], t["v"], t["prefix_len"], res["path"], res["accept_len"], dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return {"out": out, "lse": lse, **res, "src_slot": src, "new_len": nl, "k": t["k"], "v": t["v"]}


def _same(a, b):
    for key in ("out", "lse", "accept_len", "path", "bonus_token", "row_max", "row_lse", "row_entropy",
                "row_argmax", "src_slot", "new_len", "k", "v"):
        x, y = a[key], b[key]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), key


@pytest.mark.parametrize("rule", ["typical", "rejection"])
def test_round_matches_direct_calls_and_follows_refilled_inputs(rule):
    d = H.dev()
    c1, c2 = _case(rule, 3), _case(rule, 4)
    c2.seed = c1.seed  # scalars (seed, tau, eps, delta) are frozen into the round; buffers are not
    # the round's own buffers, filled with the first input set
    t = H.to_device(c1, d)
    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], c1.rule, c1.tau, c1.eps,
                              c1.delta, c1.seed, t["draft"], t["map"], path_cap=c1.N, hooks=True)
    ca, src, nl = st.compact_args(t["k"], t["v"], t["prefix_len"], outs["path"], outs["accept_len"])
    status = torch.zeros(1, dtype=torch.int32, device=d)
    r = st.Round(aa, va, ca, dev_status=status)
    del aa, va, ca  # the arguments are frozen into the graph
    got = {"out": out, "lse": lse, **outs, "src_slot": src, "new_len": nl, "k": t["k"], "v": t["v"]}
    for case in (c1, c2):
        fresh = H.to_device(case, d)
        if case is c2:  # refill the round's inputs in place
            for key, val in fresh.items():
                if val is not None:
                    t[key].copy_(val)
            fresh = H.to_device(case, d)
        r.launch()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _same(got, _direct(case, fresh))
    r.close()


def test_round_rejects_bad_arguments_at_creation():
    H.dev()
    with pytest.raises(st.SpecError) as e:
        st.Round()
    assert e.value.code == 1
    case = _case("typical", 5)
    t = H.to_device(case, H.dev())
    va, _ = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], "typical", 0.5)
    va.temperature = 0.0  # typical acceptance needs tau > 0
    with pytest.raises(st.SpecError) as e:
        st.Round(verify=va)
    assert e.value.code == 1


def _round_vs_oracle(case, d):
    """Launch the captured round once on ``case`` and compare every output with the oracle:
    attention within the bf16 tolerances, accepted length / path / bonus / margin counts as in
    the direct-call tests, compacted caches and source slots bit for bit."""
    import oracle
    t = H.to_device(case, d)
    k0, v0 = case.k_cache.copy(), case.v_cache.copy()
    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                              case.eps, case.delta, case.seed, t["draft"], t["map"], path_cap=case.N)
    ca, src, nl = st.compact_args(t["k"], t["v"], t["prefix_len"], outs["path"], outs["accept_len"])
    status = torch.zeros(1, dtype=torch.int32, device=d)
    r = st.Round(aa, va, ca, dev_status=status)
    r.launch()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    H.check_attention(case, out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64))
    got = {k: v.cpu().numpy() for k, v in outs.items()}
    ref = H.oracle_verify(case)
    c = H.check_verify(case, got, ref)
    # compaction follows the accepted path: the oracle's where it was compared bit for bit, the
    # GPU's own (already checked for validity) where a margin case excluded the request
    paths, alen = [], []
    for b in range(case.B):
        if ref[b]["path_margins"]:
            n = int(got["accept_len"][b])
            paths.append(got["path"][b, : n + 1].tolist())
            alen.append(n)
        else:
            paths.append(ref[b]["path"])
            alen.append(ref[b]["accept_len"])
    kr, vr, sr, nr = oracle.compact_kv(k0, v0, case.prefix_len, paths, np.array(alen), case.N)
    view = np.int16 if case.dtype == "bf16" else np.float32
    kg = t["k"].view(torch.int16).cpu().numpy() if case.dtype == "bf16" else t["k"].cpu().numpy()
    vg = t["v"].view(torch.int16).cpu().numpy() if case.dtype == "bf16" else t["v"].cpu().numpy()
    assert (kg == kr.view(view)).all() and (vg == vr.view(view)).all()
    assert (src.cpu().numpy() == sr).all() and (nl.cpu().numpy() == nr).all()
    r.close()
    return c


@pytest.mark.parametrize("rule", ["greedy", "typical", "rejection"])
def test_round_against_the_oracle(rule):
    d = H.dev()
    c = _round_vs_oracle(_case(rule, 11), d)
    assert c.paths_exact >= 1 and c.exact + c.excluded == 2


def test_round_on_the_llama8b_b1_medusa63_workload_against_the_oracle():
    """The B1 / 2048-token prefix / static 63-node tree / typical acceptance workload, as one
    graph launch, against the oracle end to end."""
    d = H.dev()
    c = _round_vs_oracle(H.config_case(2, 0), d)
    assert c.exact == 1


def test_round_from_host_buffers_matches_the_device_round():
    """spec_round_launch_host: the step's inputs copied in from pinned host memory (the tree's
    K/V rows by one strided copy per request), the round, and the results copied out -- equal,
    bit for bit, to a round on the same inputs already on the device."""
    d = H.dev()
    case = _case("rejection", 21)
    t = H.to_device(case, d)
    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                              case.eps, case.delta, case.seed, t["draft"], t["map"], path_cap=case.N)
    ca, src, nl = st.compact_args(t["k"], t["v"], t["prefix_len"], outs["path"], outs["accept_len"])
    status = torch.zeros(1, dtype=torch.int32, device=d)
    r = st.Round(aa, va, ca, dev_status=status)
    # reference: the same inputs, already on the device
    r.launch()
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in outs.items()}
    ref_k, ref_nl = t["k"].clone(), nl.clone()
    # reset the round's buffers: caches back to the case's, inputs scrambled, outputs poisoned
    fresh = H.to_device(case, d)
    t["k"].copy_(fresh["k"])
    t["v"].copy_(fresh["v"])
    for key in ("q", "hidden", "tokens", "parent", "draft"):
        t[key].zero_()
    for v in outs.values():
        v.fill_(-7)
    nl.fill_(-7)
    n = int(case.n_nodes.max())
    Lp = [int(x) for x in case.prefix_len]
    host = {key: fresh[key].cpu().pin_memory() for key in ("q", "hidden", "tokens", "parent", "draft")}
    ins = [st.host_copy(host[key], t[key]) for key in host]
    for b in range(case.B):
        for name in ("k", "v"):
            cache = t[name]
            rows = fresh[name][b, :, Lp[b]: Lp[b] + n].contiguous().cpu().pin_memory()
            host[f"{name}{b}"] = rows  # the descriptors hold raw pointers: keep the buffers alive
            ins.append(st.host_copy(rows, cache[b, :, Lp[b]: Lp[b] + n], rows=case.Hkv))
            cache[b, :, Lp[b]: Lp[b] + n].zero_()  # the tree slots now arrive only from the host
    res = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
    res_nl = torch.empty(nl.shape, dtype=nl.dtype).pin_memory()
    outs_c = [st.host_copy(res[k], outs[k]) for k in res] + [st.host_copy(res_nl, nl)]
    torch.cuda.synchronize()
    r.launch_host(ins, outs_c)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k in res:
        assert torch.equal(res[k], ref[k].cpu()), k
    assert torch.equal(res_nl, ref_nl.cpu())
    assert torch.equal(t["k"].view(torch.int16), ref_k.view(torch.int16))
    r.close()


def test_host_round_steps_back_to_back():
    """Three spec_round_launch_host steps enqueued without a synchronisation in between, their
    inputs alternating between two variants (different hidden states and draft distributions):
    every step's results equal a device round on that step's inputs, so no step's copies overtake
    the previous step's readers (the verification's inputs and the draft distributions travel on
    streams of the round's own)."""
    d = H.dev()
    case = _case("rejection", 21)
    t = H.to_device(case, d)
    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                              case.eps, case.delta, case.seed, t["draft"], t["map"], path_cap=case.N)
    ca, src, nl = st.compact_args(t["k"], t["v"], t["prefix_len"], outs["path"], outs["accept_len"])
    status = torch.zeros(1, dtype=torch.int32, device=d)
    r = st.Round(aa, va, ca, dev_status=status)
    fresh = H.to_device(case, d)
    keys = ("q", "hidden", "tokens", "parent", "draft")
    var_a = {k: fresh[k].clone() for k in keys}
    var_b = {k: fresh[k].clone() for k in keys}
    var_b["hidden"] = (var_b["hidden"].float() * -0.75).to(var_b["hidden"].dtype)
    var_b["draft"] = torch.roll(var_b["draft"], shifts=1, dims=-1)

    def reset_caches():
        t["k"].copy_(fresh["k"])
        t["v"].copy_(fresh["v"])

    refs = []
    for var in (var_a, var_b):  # device rounds on each variant
        reset_caches()
        for k in keys:
            t[k].copy_(var[k])
        r.launch()
        torch.cuda.synchronize()
        refs.append(({k: v.clone() for k, v in outs.items()}, nl.clone()))
    reset_caches()
    for k in keys:
        t[k].zero_()
    n = int(case.n_nodes.max())
    Lp = [int(x) for x in case.prefix_len]
    tree_rows = []
    for b in range(case.B):
        for name in ("k", "v"):
            rows = fresh[name][b, :, Lp[b]: Lp[b] + n].contiguous().cpu().pin_memory()
            tree_rows.append((rows, t[name][b, :, Lp[b]: Lp[b] + n]))
    host_vars = [{k: v[k].cpu().pin_memory() for k in keys} for v in (var_a, var_b)]
    order = (0, 1, 0)
    results = []
    for step, vi in enumerate(order):  # the descriptors hold raw pointers: everything stays referenced
        ins = [st.host_copy(host_vars[vi][k], t[k]) for k in keys]
        ins += [st.host_copy(rows, dst, rows=case.Hkv) for rows, dst in tree_rows]
        res = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
        res_nl = torch.empty(nl.shape, dtype=nl.dtype).pin_memory()
        outs_c = [st.host_copy(res[k], outs[k]) for k in res] + [st.host_copy(res_nl, nl)]
        r.launch_host(ins, outs_c)
        results.append((vi, res, res_nl))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for vi, res, res_nl in results:
        ref, ref_nl = refs[vi]
        for k in res:
            assert torch.equal(res[k], ref[k].cpu()), (vi, k)
        assert torch.equal(res_nl, ref_nl.cpu()), vi
    assert any(not torch.equal(refs[0][0][k], refs[1][0][k]) for k in refs[0][0]), "variants should differ"
    r.close()


def test_host_round_with_compact_draft_rows():
    """The host-buffer round with the draft distributions of the expanded nodes only (compact
    [rows][Vd] plus a [B][N] row index, both copied from the host): the same results as the
    device round over the full [B][N][Vd] layout."""
    d = H.dev()
    case = _case("rejection", 23)
    t = H.to_device(case, d)
    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                              case.eps, case.delta, case.seed, t["draft"], t["map"], path_cap=case.N)
    ca, src, nl = st.compact_args(t["k"], t["v"], t["prefix_len"], outs["path"], outs["accept_len"])
    status = torch.zeros(1, dtype=torch.int32, device=d)
    r = st.Round(aa, va, ca, dev_status=status)
    r.launch()
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in outs.items()}
    ref_k, ref_nl = t["k"].clone(), nl.clone()
    r.close()

    rows, index = compact_draft(case.draft_probs, case.parent, case.n_nodes, rng=np.random.default_rng(4))
    t2 = H.to_device(case, d)
    t2["rows"], t2["index"] = H.tensor(rows, d), H.tensor(index, d)
    aa, out, lse = st.attn_args(t2["q"], t2["k"], t2["v"], t2["prefix_len"], t2["n_nodes"], t2["parent"])
    va, outs = st.verify_args(t2["hidden"], t2["W"], t2["tokens"], t2["parent"], t2["n_nodes"], case.rule, case.tau,
                              case.eps, case.delta, case.seed, t2["rows"], t2["map"], path_cap=case.N,
                              draft_rows=t2["index"])
    ca, src, nl = st.compact_args(t2["k"], t2["v"], t2["prefix_len"], outs["path"], outs["accept_len"])
    r = st.Round(aa, va, ca, dev_status=status)
    # parent and n_nodes are read by both branches (with the verification first, they are copied
    # with its group), prefix_len by the attention and the compaction
    keys = ("q", "hidden", "tokens", "parent", "n_nodes", "prefix_len", "rows", "index")
    host = {k: t2[k].cpu().pin_memory() for k in keys}
    for k in keys:
        t2[k].zero_()
    for v in outs.values():
        v.fill_(-7)
    ins = [st.host_copy(host[k], t2[k]) for k in keys]
    res = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
    res_nl = torch.empty(nl.shape, dtype=nl.dtype).pin_memory()
    outs_c = [st.host_copy(res[k], outs[k]) for k in res] + [st.host_copy(res_nl, nl)]
    torch.cuda.synchronize()
    r.launch_host(ins, outs_c)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k in res:
        assert torch.equal(res[k], ref[k].cpu()), k
    assert torch.equal(res_nl, ref_nl.cpu())
    assert torch.equal(t2["k"].view(torch.int16), ref_k.view(torch.int16))
    r.close()


def test_host_round_attention_first_with_draft_rows():
    """A round whose attention is the longer branch (prefixes of thousands of keys, a 64-token
    vocabulary): the host-buffer round copies the attention's inputs first, then the
    verification's, then the compact draft rows, and issues the attention first -- with the same
    results as the device round."""
    d = H.dev()
    rng = np.random.default_rng(31)
    parents = [T.random_bfs_tree(rng, 24, 4)[0], T.chain_tree(6), T.random_bfs_tree(rng, 24, 3)[0]]
    case = make_case(dtype="bf16", Hq=8, Hkv=2, d=128, Hd=64, V=64, prefix_len=[6000, 3100, 7777],
                     parents=parents, rule="rejection", tau=0.9, seed=8, tokens=("iid", 0.8, 0.4), rng=rng)
    rows, index = compact_draft(case.draft_probs, case.parent, case.n_nodes, rng=rng)
    t = H.to_device(case, d)
    t["rows"], t["index"] = H.tensor(rows, d), H.tensor(index, d)
    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                              case.eps, case.delta, case.seed, t["rows"], t["map"], path_cap=case.N,
                              draft_rows=t["index"])
    ca, src, nl = st.compact_args(t["k"], t["v"], t["prefix_len"], outs["path"], outs["accept_len"])
    status = torch.zeros(1, dtype=torch.int32, device=d)
    r = st.Round(aa, va, ca, dev_status=status)
    r.launch()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = {k: v.clone() for k, v in outs.items()}
    ref_out, ref_k, ref_nl = out.clone(), t["k"].clone(), nl.clone()
    fresh = H.to_device(case, d)
    t["k"].copy_(fresh["k"])
    t["v"].copy_(fresh["v"])
    keys = ("q", "hidden", "tokens", "parent", "rows", "index")
    host = {k: t[k].cpu().pin_memory() for k in keys}
    for k in keys:
        t[k].zero_()
    for v in outs.values():
        v.fill_(-7)
    out.zero_()
    ins = [st.host_copy(host[k], t[k]) for k in keys]
    res = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs.items()}
    res_nl = torch.empty(nl.shape, dtype=nl.dtype).pin_memory()
    outs_c = [st.host_copy(res[k], outs[k]) for k in res] + [st.host_copy(res_nl, nl)]
    torch.cuda.synchronize()
    r.launch_host(ins, outs_c)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k in res:
        assert torch.equal(res[k], ref[k].cpu()), k
    assert torch.equal(res_nl, ref_nl.cpu())
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(t["k"].view(torch.int16), ref_k.view(torch.int16))
    r.close()

"""The CUDA-graph verification round (spec_round_create / spec_round_launch) against the three
direct calls: the same kernels run, so every output must match bit for bit, also after the
inputs are refilled in place and the round is launched again."""

import numpy as np
import pytest
import torch

import tree_speculative_decoding_split_gb300 as st
from gen import make_case, trees as T
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

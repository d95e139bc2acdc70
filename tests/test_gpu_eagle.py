"""GPU parity of the layered dynamic draft tree (spec_eagle_expand / spec_eagle_tree) with the
oracle, bit for bit: every decision is taken on the same float32 scores on both sides."""

import numpy as np
import pytest
import torch

import oracle
import tree_speculative_decoding_split_gb300 as st
import gpu_helpers as H
from gen import compact_draft as gen_compact_draft

pytestmark = pytest.mark.gpu


def _logp(rng, shape, ties):
    z = rng.standard_normal(shape)
    if ties:
        z = np.round(z * 2) / 2
    lp = z - np.log(np.exp(z).sum(-1, keepdims=True))
    return lp.astype(np.float32)


@pytest.mark.parametrize("F,k,Vd,next_k,ties", [(8, 8, 32000, 8, False), (5, 3, 1000, 7, True),
                                                 (1, 16, 4096, 16, True), (32, 8, 7, 4, False)])
def test_expand_layer_matches_oracle(F, k, Vd, next_k, ties):
    d = H.dev()
    rng = np.random.default_rng(F * 100 + k)
    k = min(k, Vd)
    B = 3
    lp = _logp(rng, (B, F, Vd), ties)
    fs = (-rng.exponential(2.0, (B, F))).astype(np.float32)
    if ties:
        fs = np.round(fs).astype(np.float32)
    valid = np.ones((B, F), dtype=np.int32)
    if F > 2:
        valid[1, 2] = 0
    fc = rng.integers(0, 50, (B, F)).astype(np.int32)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    out = st.eagle_expand(H.tensor(lp, d), H.tensor(fs, d), k, next_k, frontier_valid=H.tensor(valid, d),
                          frontier_cand=H.tensor(fc, d), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = {key: v.cpu().numpy() for key, v in out.items()}
    for b in range(B):
        ref = oracle.expand_layer(lp[b], fs[b], k, next_k, frontier_valid=valid[b], frontier_cand=fc[b])
        assert (got["token"][b] == ref["token"]).all()
        assert (got["parent"][b] == ref["parent"]).all()
        assert np.array_equal(got["score"][b], ref["score"])
        assert (got["next_index"][b] == ref["next_index"]).all()
        assert np.array_equal(got["next_score"][b], ref["next_score"])


def _build(d, rng, B, F, k, Vd, D, N, ties=False, d2t=None):
    """Run D expansion layers on the device (random log-probabilities stand in for the draft
    model), stacking candidates into [B][D][C], then select the tree; the oracle replays it."""
    C = F * k
    S = torch.full((B, D, C), float("-inf"), dtype=torch.float32, device=d)
    Tk = torch.full((B, D, C), -1, dtype=torch.int32, device=d)
    P = torch.full((B, D, C), -1, dtype=torch.int32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    fs = torch.zeros((B, 1), dtype=torch.float32, device=d)
    valid = torch.ones((B, 1), dtype=torch.int32, device=d)
    fc = torch.full((B, 1), -1, dtype=torch.int32, device=d)
    lps = []
    ref_layers = [[] for _ in range(B)]
    ref_front = [(np.zeros(1, np.float32), np.ones(1, np.int32), np.full(1, -1)) for _ in range(B)]
    for l in range(D):
        Fl = fs.shape[1]
        lp = _logp(rng, (B, Fl, Vd), ties)
        lps.append(lp)
        outs = {"token": Tk[:, l], "score": S[:, l], "parent": P[:, l]}
        res = st.eagle_expand(H.tensor(lp, d), fs, k, F, frontier_valid=valid, frontier_cand=fc, outputs=outs,
                              cand_stride=D * C, dev_status=status)
        for b in range(B):
            r = oracle.expand_layer(lp[b], ref_front[b][0], k, F, frontier_valid=ref_front[b][1],
                                    frontier_cand=ref_front[b][2])
            ref_layers[b].append(r)
            ok = r["next_index"] >= 0
            ref_front[b] = (np.where(ok, r["next_score"], -np.inf).astype(np.float32), ok.astype(np.int32),
                            np.where(ok, r["next_index"], -1))
        fs = res["next_score"].clone()
        fc = res["next_index"].clone()
        valid = (fc >= 0).to(torch.int32)
    root = torch.from_numpy(rng.integers(0, 1000, B).astype(np.int32)).to(d)
    tmap = None if d2t is None else H.tensor(d2t, d)
    tree = st.eagle_tree(S, Tk, P, N, draft_to_target=tmap, root_token=root, dev_status=status)
    torch.cuda.synchronize()
    return tree, int(status.item()), ref_layers, root.cpu().numpy(), (S, Tk, P)


@pytest.mark.parametrize("F,k,Vd,D,N,ties", [(8, 8, 32000, 6, 63, False), (4, 4, 500, 8, 255, True),
                                              (2, 3, 50, 3, 10, True)])
def test_layers_and_tree_match_oracle(F, k, Vd, D, N, ties):
    d = H.dev()
    rng = np.random.default_rng(D * 10 + N)
    B = 4
    d2t = rng.permutation(Vd * 4)[:Vd].astype(np.int32)
    tree, status, ref_layers, root, (S, Tk, P) = _build(d, rng, B, F, k, Vd, D, N, ties, d2t)
    assert status == 0
    C = F * k
    for b in range(B):
        # the stacked candidates equal the oracle's layers bit for bit
        for l, r in enumerate(ref_layers[b]):
            c = len(r["score"])
            assert np.array_equal(S[b, l, :c].cpu().numpy(), r["score"])
            assert (Tk[b, l, :c].cpu().numpy() == r["token"]).all()
            assert (P[b, l, :c].cpu().numpy() == r["parent"]).all()
        tp, tt, nn, nc = oracle.select_tree(S[b].cpu().numpy(), Tk[b].cpu().numpy(), P[b].cpu().numpy(), N,
                                            root_token=int(root[b]), draft_to_target=d2t)
        assert int(tree["n_nodes"][b]) == nn
        assert (tree["parent"][b].cpu().numpy() == tp).all()
        assert (tree["tokens"][b].cpu().numpy() == tt).all()
        assert (tree["node_cand"][b].cpu().numpy() == nc).all()
        assert oracle.validate_tree(tp, nn)


def test_tree_errors():
    d = H.dev()
    # a child scoring above its parent breaks closure when the parent is cut
    S = torch.tensor([[[-1.0, -5.0], [-0.5, -9.0]]], dtype=torch.float32, device=d)
    Tk = torch.tensor([[[1, 2], [3, 4]]], dtype=torch.int32, device=d)
    P = torch.tensor([[[-1, -1], [1, 0]]], dtype=torch.int32, device=d)  # (1,0) has parent (0,1)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    tree = st.eagle_tree(S, Tk, P, 3, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 4 and int(tree["n_nodes"][0]) == 1
    status.zero_()
    m = torch.arange(3, dtype=torch.int32, device=d)  # token 4 is outside a 3-entry map
    tree = st.eagle_tree(S, Tk, P, 5, draft_to_target=m, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6


def test_dynamic_tree_verified_by_rejection_with_compact_draft_rows():
    """The dynamic draft tree end to end on the device: expansion layers and tree selection over a
    mapped draft vocabulary, then rejection-sampling verification of that tree whose draft
    distributions are the expanded nodes' rows only (draft_rows) -- against the oracle's
    verification of the same tree with the full [B][N][Vd] layout."""
    import dataclasses
    from gen import make_case
    d = H.dev()
    rng = np.random.default_rng(2024)
    B, F, k, Vd, D, N = 3, 4, 4, 500, 4, 31
    V = 4 * Vd
    d2t = rng.permutation(V)[:Vd].astype(np.int32)
    C = F * k
    S = torch.full((B, D, C), float("-inf"), dtype=torch.float32, device=d)
    Tk = torch.full((B, D, C), -1, dtype=torch.int32, device=d)
    P = torch.full((B, D, C), -1, dtype=torch.int32, device=d)
    status = torch.zeros(1, dtype=torch.int32, device=d)
    fs = torch.zeros((B, 1), dtype=torch.float32, device=d)
    valid = torch.ones((B, 1), dtype=torch.int32, device=d)
    fc = torch.full((B, 1), -1, dtype=torch.int32, device=d)
    lps, fronts = [], []  # per layer: log-probabilities of its frontier rows, and the candidates they are
    for l in range(D):
        lp = _logp(rng, (B, fs.shape[1], Vd), False)
        lps.append(lp)
        fronts.append(fc.cpu().numpy())  # frontier row f of layer l = candidate fronts[l][b][f] of layer l - 1
        outs = {"token": Tk[:, l], "score": S[:, l], "parent": P[:, l]}
        res = st.eagle_expand(H.tensor(lp, d), fs, k, F, frontier_valid=valid, frontier_cand=fc, outputs=outs,
                              cand_stride=D * C, dev_status=status)
        fs, fc = res["next_score"].clone(), res["next_index"].clone()
        valid = (fc >= 0).to(torch.int32)
    root = torch.from_numpy(rng.integers(0, V, B).astype(np.int32)).to(d)
    tree = st.eagle_tree(S, Tk, P, N, draft_to_target=H.tensor(d2t, d), root_token=root, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    parent = tree["parent"].cpu().numpy()
    tokens = tree["tokens"].cpu().numpy()
    n_nodes = tree["n_nodes"].cpu().numpy()
    node_cand = tree["node_cand"].cpu().numpy()
    # each node's draft distribution: the frontier row its children were drawn from
    full = np.zeros((B, N, Vd), dtype=np.float32)
    for b in range(B):
        full[b, 0] = np.exp(lps[0][b, 0])
        for i in range(1, int(n_nodes[b])):
            l, j = divmod(int(node_cand[b, i]), C)
            if l + 1 < D:
                f = np.nonzero(fronts[l + 1][b] == j)[0]
                if len(f):
                    full[b, i] = np.exp(lps[l + 1][b, f[0]])
    parents = [parent[b, : int(n_nodes[b])] for b in range(B)]
    case = make_case(dtype="bf16", Hq=4, Hkv=1, d=64, Hd=128, V=V, prefix_len=[4] * B, parents=parents, N=N,
                     rule="rejection", tau=1.0, seed=17, tokens=("given", tokens), rng=rng)
    case = dataclasses.replace(case, draft_probs=full, draft_to_target=d2t)
    rows, index = gen_compact_draft(full, case.parent, case.n_nodes)
    assert rows.shape[0] < B * N
    t = H.to_device(case, d)
    status.zero_()
    res = st.verify_accept(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], "rejection", 1.0,
                           seed=case.seed, draft_probs=H.tensor(rows, d), draft_to_target=t["map"],
                           draft_rows=H.tensor(index, d), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = {k_: v.cpu().numpy() for k_, v in res.items()}
    c = H.check_verify(case, got, H.oracle_verify(case))
    assert c.exact + c.excluded == case.B and c.paths_exact >= 1

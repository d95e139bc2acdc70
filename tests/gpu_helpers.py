"""Shared plumbing of the GPU parity tests: move a generated case to the device, run the C ABI
through the binding, run the oracle on the same inputs, and compare.

Tolerances (written here, used by every GPU test):
* attention output: max-abs 2e-2 (bf16 inputs/outputs) or 1e-5 (fp32);
* attention LSE: relative 1e-3;
* LM-head statistics (max, LSE, entropy of each row): absolute 2e-3 for bf16 (fp32 accumulation over a
  4096/8192-long bf16 dot product) and 1e-4 for fp32; argmax exact unless the oracle's top-2 gap is below
  the 1e-4 margin;
* accepted length, path, bonus token and compacted KV / source slots: bit-exact, except for requests
  whose evaluated decisions include a margin case (counted and reported), which are checked for
  validity instead;
* margin counts (decisions within 1e-4 of their threshold) and the bonus flag: the GPU's against the
  oracle's, up to decisions at the band's edge.
"""

from typing import NamedTuple

import numpy as np
import torch

import oracle
import tree_speculative_decoding_split_gb300 as st

ATTN_TOL = {"bf16": 2e-2, "f32": 1e-5}
LSE_RTOL = 1e-3
STAT_TOL = {"bf16": 2e-3, "f32": 1e-4}


_CASES = {}


def config_case(cfg, seed):
    """Workload inputs, generated once per test session."""
    from gen import make_config_case
    key = (cfg, seed)
    if key not in _CASES:
        if len(_CASES) >= 2:
            _CASES.clear()
        _CASES[key] = make_config_case(cfg, seed=seed)
    return _CASES[key]


def dev():
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need CUDA")
    st.build()
    st.lib()
    return torch.device("cuda:0")


def tensor(a, device, bf16=False):
    if bf16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_device(case, device):
    bf = case.dtype == "bf16"
    t = {
        "q": tensor(case.q, device, bf), "k": tensor(case.k_cache, device, bf), "v": tensor(case.v_cache, device, bf),
        "hidden": tensor(case.hidden, device, bf), "W": tensor(case.W, device, bf),
        "prefix_len": tensor(case.prefix_len.astype(np.int32), device),
        "n_nodes": tensor(case.n_nodes.astype(np.int32), device),
        "parent": tensor(case.parent.astype(np.int32), device),
        "tokens": tensor(case.tokens.astype(np.int32), device),
        "draft": None if case.draft_probs is None else tensor(case.draft_probs, device),
        "map": None if case.draft_to_target is None else tensor(case.draft_to_target.astype(np.int32), device),
    }
    return t


def gpu_attention(case, t):
    status = torch.zeros(1, dtype=torch.int32, device=t["q"].device)
    out, lse = st.tree_attention(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"],
                                 dev_status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), int(status.item())


def gpu_verify(case, t, hooks=True, path_cap=None):
    status = torch.zeros(1, dtype=torch.int32, device=t["hidden"].device)
    res = st.verify_accept(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                           case.eps, case.delta, case.seed, draft_probs=t["draft"], draft_to_target=t["map"],
                           path_cap=path_cap, hooks=hooks, dev_status=status)
    torch.cuda.synchronize()
    out = {k: v.cpu().numpy() for k, v in res.items()}
    out["status"] = int(status.item())
    return out


def oracle_verify(case, requests=None):
    return oracle.verify_accept(case.f64("hidden") if case.B * case.N * case.Hd < 5e7 else case.f32("hidden"),
                                case.f32("W"), case.tokens, case.parent, case.n_nodes, case.rule, case.tau,
                                case.eps, case.delta, case.seed, draft_probs=case.draft_probs,
                                draft_to_target=case.draft_to_target, requests=requests)


def check_attention(case, got_o, got_l, rows=None):
    """Compare with the oracle on all rows, or on sampled (b, i, h) rows."""
    tol = ATTN_TOL[case.dtype]
    if rows is None:
        O, L = oracle.tree_attention(case.f64("q"), case.f64("k_cache"), case.f64("v_cache"), case.prefix_len,
                                     case.n_nodes, case.parent)
        err = np.abs(got_o - O).max()
        lerr = (np.abs(got_l - L) / np.maximum(np.abs(L), 1e-6)).max()
    else:
        qf = case.f32("q")
        kf = case.f32("k_cache")
        vf = case.f32("v_cache")
        O, L = oracle.tree_attention_rows(qf, kf, vf, case.prefix_len, case.n_nodes, case.parent, rows)
        go = np.stack([got_o[b, i, h] for b, i, h in rows])
        gl = np.array([got_l[b, i, h] for b, i, h in rows])
        err = np.abs(go - O).max()
        lerr = (np.abs(gl - L) / np.maximum(np.abs(L), 1e-6)).max()
    assert err < tol, f"attention max-abs error {err} >= {tol}"
    assert lerr < LSE_RTOL, f"LSE relative error {lerr} >= {LSE_RTOL}"
    return err, lerr


class VerifyCheck(NamedTuple):
    exact: int           # requests whose path, length and bonus were compared bit for bit
    excluded: int        # requests with a margin case (path or bonus) among their decisions
    paths_exact: int     # requests whose path and length were compared bit for bit
    margins_gpu: int     # margin cases the GPU counted over the compared requests
    margins_oracle: int  # margin cases the oracle counted over the same requests


def oracle_request_at_band(case, b, band):
    """The oracle's verdict on request b with the margin band set to ``band``.  Decisions do not
    depend on the band; only which of them count as near-threshold does."""
    import oracle.accept as acc
    old = acc.MARGIN
    acc.MARGIN = band
    try:
        return oracle_verify(case, requests=[b])[b]
    finally:
        acc.MARGIN = old


def _check_margins(case, b, got, r):
    """The GPU's margin count and bonus flag against the oracle's.  A decision the oracle puts
    within the band is evaluated by the GPU as well (every decision before it is outside the band,
    so both sides agree on it), so an oracle count >= 1 implies a GPU count >= 1 and a count of 0
    implies 0 -- unless a decision sits at the band's edge, where float32 and float64 may fall on
    either side; those are recognised by re-running the oracle with the band 10 % wider or narrower."""
    gm = int(got["margin_count"][b])
    gb = int(got["bonus_margin"][b])
    if r["path_margins"] == 0:
        if gm != 0:
            wide = oracle_request_at_band(case, b, oracle.MARGIN * 1.1)
            assert gm <= wide["path_margins"], (b, gm, r["path_margins"], wide["path_margins"])
    elif gm == 0:
        narrow = oracle_request_at_band(case, b, oracle.MARGIN * 0.9)
        assert narrow["path_margins"] == 0, (b, gm, r["path_margins"])
    same_end = int(got["accept_len"][b]) == r["accept_len"] and \
        got["path"][b, r["accept_len"]] == r["path"][-1]
    if same_end and bool(gb) != bool(r["bonus_margin"]):
        # the bonus decision is taken at the same endpoint: the flags must agree up to the edge
        other = oracle_request_at_band(case, b, oracle.MARGIN * (1.1 if gb else 0.9))
        assert bool(other["bonus_margin"]) == bool(gb), (b, gb, r["bonus_margin"])


def check_verify(case, got, ref, requests=None, stats_rows=None):
    """Bit-exact comparison of accept_len / path / bonus outside margin cases, and of the margin
    counts against the oracle's; returns a VerifyCheck."""
    todo = range(case.B) if requests is None else requests
    exact = excluded = paths_exact = mg_gpu = mg_orc = 0
    for b in todo:
        r = ref[b]
        n = int(case.n_nodes[b])
        gl = int(got["accept_len"][b])
        gp = got["path"][b]
        # validity holds always: a root path of increasing, parent-linked nodes
        assert gp[0] == 0
        for j in range(1, gl + 1):
            assert 0 < gp[j] < n and case.parent[b, gp[j]] == gp[j - 1], (b, gp[: gl + 1])
        assert (gp[gl + 1:] == -1).all()
        if "margin_count" in got and "bonus_margin" in got:
            _check_margins(case, b, got, r)
            mg_gpu += int(got["margin_count"][b])
            mg_orc += int(r["path_margins"])
        if r["path_margins"]:
            excluded += 1
            continue
        assert gl == r["accept_len"], (b, gl, r["accept_len"])
        assert gp[: gl + 1].tolist() == r["path"], (b, gp[: gl + 1], r["path"])
        paths_exact += 1
        if r["bonus_margin"]:
            lo, hi = r["bonus_window"]
            assert lo <= int(got["bonus_token"][b]) <= hi, (b, got["bonus_token"][b], r["bonus_window"])
            excluded += 1
        else:
            assert int(got["bonus_token"][b]) == r["bonus"], (b, got["bonus_token"][b], r["bonus"])
            exact += 1
    return VerifyCheck(exact, excluded, paths_exact, mg_gpu, mg_orc)


def check_row_stats(case, got, rows):
    """Compare the GPU's per-row statistics hooks with the oracle on (b, i) rows."""
    tol = STAT_TOL[case.dtype]
    H = np.stack([case.f64("hidden")[b, i] for b, i in rows]) if case.dtype == "f32" else \
        np.stack([case.f32("hidden")[b, i].astype(np.float64) for b, i in rows])
    z = oracle.logits(H, case.f32("W"))
    tau = case.tau if case.rule != "greedy" else 0.0
    worst = 0.0
    for r, (b, i) in enumerate(rows):
        s = oracle.row_stats(z[r], tau)
        for key, gk in (("max", "row_max"), ("lse", "row_lse"), ("entropy", "row_entropy")):
            e = abs(float(got[gk][b, i]) - s[key])
            worst = max(worst, e)
            assert e < tol, (key, b, i, float(got[gk][b, i]), s[key])
        if s["gap"] >= oracle.MARGIN:
            assert int(got["row_argmax"][b, i]) == s["argmax"], (b, i)
        else:
            am = int(got["row_argmax"][b, i])
            assert z[r, am] >= z[r].max() - oracle.MARGIN
    return worst

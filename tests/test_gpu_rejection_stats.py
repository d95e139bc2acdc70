"""Losslessness of the GPU rejection-sampling kernel ([GUIDE] section "棄却サンプリング": the output
distribution is exactly the target's).

Tiny vocabulary (8 tokens), W = identity and hidden state = log T, so the target distribution at the
root is exactly T.  Each request is a root with three children drawn i.i.d. from D.  The first
emitted token (the accepted child's token, or the bonus sample when all are rejected) must follow T:
chi-square over 10^6 seeded trials (p > 1e-3), while the same counts must be rejected against D
(the test can tell the two apart).  A subset of trials is also compared one by one with the oracle.
"""

import numpy as np
import pytest
import torch
from scipy.stats import chisquare

import oracle
import tree_speculative_decoding_split_gb300 as st
import gpu_helpers as H

pytestmark = pytest.mark.gpu

V = 8
T_ROOT = np.array([0.30, 0.05, 0.20, 0.10, 0.02, 0.13, 0.15, 0.05])
D_ROOT = np.array([0.05, 0.25, 0.10, 0.10, 0.20, 0.05, 0.05, 0.20])


def _batch(rng, B):
    parent = np.tile(np.array([-1, 0, 0, 0], dtype=np.int32), (B, 1))
    tokens = np.zeros((B, 4), dtype=np.int32)
    tokens[:, 1:] = rng.choice(V, size=(B, 3), p=D_ROOT)
    hidden = np.tile(np.log(np.full(V, 1.0 / V)), (B, 4, 1)).astype(np.float32)
    hidden[:, 0, :] = np.log(T_ROOT)
    draft = np.zeros((B, 4, V), dtype=np.float32)
    draft[:, 0, :] = D_ROOT
    return parent, tokens, hidden, draft


def _run(d, parent, tokens, hidden, draft, seed):
    B = parent.shape[0]
    res = st.verify_accept(H.tensor(hidden, d), torch.eye(V, dtype=torch.float32, device=d),
                           H.tensor(tokens, d), H.tensor(parent, d),
                           torch.full((B,), 4, dtype=torch.int32, device=d), "rejection", 1.0, seed=seed,
                           draft_probs=H.tensor(draft, d), path_cap=4)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in res.items()}


def test_gpu_rejection_sampling_matches_target_distribution():
    d = H.dev()
    rng = np.random.default_rng(1234)
    counts = np.zeros(V, dtype=np.int64)
    calls, B = 4, 250_000
    for call in range(calls):
        parent, tokens, hidden, draft = _batch(rng, B)
        r = _run(d, parent, tokens, hidden, draft, seed=777 + call)
        acc = r["accept_len"] >= 1
        first = np.where(acc, tokens[np.arange(B), np.maximum(r["path"][:, 1], 0)], r["bonus_token"])
        assert (first >= 0).all() and (first < V).all()
        counts += np.bincount(first, minlength=V)
    n = calls * B
    assert chisquare(counts, n * T_ROOT).pvalue > 1e-3, counts
    assert chisquare(counts, n * D_ROOT).pvalue < 1e-3  # the test distinguishes T from D


def test_gpu_rejection_trials_match_oracle_one_by_one():
    d = H.dev()
    rng = np.random.default_rng(99)
    B = 3000
    parent, tokens, hidden, draft = _batch(rng, B)
    r = _run(d, parent, tokens, hidden, draft, seed=31337)
    z = hidden.astype(np.float64)
    mism = 0
    for b in range(B):
        ref = oracle.verify_request(parent[b], 4, tokens[b], z[b], "rejection", 1.0, 0, 0, 31337, b,
                                    draft_row=lambda e: D_ROOT if e == 0 else np.zeros(V))
        if ref["path_margins"] or ref["bonus_margin"]:
            continue
        ok = (r["accept_len"][b] == ref["accept_len"] and list(r["path"][b, : ref["accept_len"] + 1]) == ref["path"]
              and r["bonus_token"][b] == ref["bonus"])
        mism += not ok
    assert mism == 0

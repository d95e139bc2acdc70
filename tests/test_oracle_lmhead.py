"""Pins for the oracle's LM head and row statistics: closed forms and library routines."""

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp, softmax
from scipy.stats import entropy


def test_uniform_row_closed_form():
    from oracle import row_stats
    for V in (1, 8, 2048, 128256):
        s = row_stats(np.zeros(V), 1.0)
        assert abs(s["entropy"] - np.log(V)) < 1e-9
        assert abs(s["lse"] - np.log(V)) < 1e-9
        assert s["argmax"] == 0  # all tied -> lowest index


def test_one_hot_limit_and_two_point():
    from oracle import row_stats
    z = np.zeros(100)
    z[37] = 60.0
    s = row_stats(z, 1.0)
    assert s["argmax"] == 37 and s["entropy"] < 1e-20 and abs(s["gap"] - 60.0) < 1e-12
    # two equiprobable logits among -inf-like others: H = ln 2; at tau = 2 logits halve
    z = np.full(10, -1e4)
    z[[2, 5]] = 3.0
    s = row_stats(z, 2.0)
    assert abs(s["entropy"] - np.log(2)) < 1e-12 and s["argmax"] == 2 and s["gap"] == 0
    # binary entropy closed form for p = sigmoid(a)
    a = 1.3
    s = row_stats(np.array([a, 0.0]), 1.0)
    p = 1 / (1 + np.exp(-a))
    assert abs(s["entropy"] - (-p * np.log(p) - (1 - p) * np.log(1 - p))) < 1e-14


@pytest.mark.parametrize("tau", [0.7, 1.0, 2.5])
def test_row_stats_match_library(tau):
    from oracle import row_stats
    rng = np.random.default_rng(1)
    z = rng.standard_normal(5000) * 3
    s = row_stats(z, tau)
    y = z / tau
    assert abs(s["max"] - y.max()) == 0
    assert abs(s["lse"] - logsumexp(y)) < 1e-12
    np.testing.assert_allclose(s["p"], softmax(y), rtol=1e-12, atol=0)
    assert abs(s["entropy"] - entropy(softmax(y))) < 1e-10
    srt = np.sort(z)
    assert s["argmax"] == int(np.argmax(z)) and abs(s["gap"] - (srt[-1] - srt[-2])) < 1e-15


def test_logits_match_library_linear():
    from oracle import logits
    rng = np.random.default_rng(4)
    H = rng.standard_normal((7, 64))
    W = rng.standard_normal((1000, 64)).astype(np.float32)
    z = logits(H, W, chunk=333)
    ref = F.linear(torch.from_numpy(H), torch.from_numpy(W.astype(np.float64))).numpy()
    np.testing.assert_allclose(z, ref, rtol=1e-13, atol=1e-12)

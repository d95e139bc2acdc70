"""Pins for the oracle's margin detector (decisions within 1e-4 of their threshold) and for the
draft-to-target scatter of the rejection rule, on hand-computed cases.

The margin detector decides which requests leave the bit-exact GPU comparison, so a band that is
too wide or too narrow, a decision counted that the walk never evaluates, or an off-by-one in the
bonus window must each fail one of these:

* greedy: a top-2 logit gap of 5e-5 is flagged, 2e-4 is not; a node below a rejected node is
  never evaluated and never counted; the bonus flag follows the endpoint row's gap;
* typical (jisaku glossary "Medusa", section "Medusa-1: 典型的採択"): |ln p(x) - ln thr| of
  5e-5 is flagged on both sides of the threshold, 2e-4 is not, with either eps or
  delta * exp(-H) binding;
* rejection (qiita guide, section "棄却サンプリング：出力品質を保証する"): |u - min(1, R[x]/D[x])|
  of 5e-5 is flagged on both sides, 2e-4 is not; the count runs over every sibling the walk
  tries, with the ratio of the second sibling taken against the updated residual;
* bonus window: u' * sum R next to a cumulative boundary gives the hand-derived (lo, hi);
* draft map (EAGLE-3's 32000-entry draft vocabulary): the draft row lands on the mapped target
  ids and is zero elsewhere, and the walk's decisions follow that scattered row.
"""

import math

import numpy as np
import pytest

import oracle
from oracle.accept import draft_in_target_vocab

M = oracle.MARGIN


def _chain(n):
    return np.array([-1] + list(range(n - 1)))


# ---- greedy ---------------------------------------------------------------------------------

@pytest.mark.parametrize("gap,flagged", [(5e-5, True), (2e-4, False), (9.9e-5, True), (1.01e-4, False)])
def test_greedy_gap_band(gap, flagged):
    parent = np.array([-1, 0])
    z = np.array([[0.0, 1.0, 1.0 - gap, -1.0, 0.5],
                  [3.0, 0.0, 0.0, 0.0, 0.0]])          # endpoint row: clear argmax 0
    r = oracle.verify_request(parent, 2, np.array([0, 1]), z, "greedy", 0.0, 0, 0, 0, 0)
    assert r["path"] == [0, 1]                        # token 1 is the argmax either way
    assert r["path_margins"] == (1 if flagged else 0)
    assert r["bonus"] == 0 and r["bonus_margin"] is False and r["bonus_window"] == (0, 0)


def test_greedy_unevaluated_node_is_not_counted():
    # root -> 1 -> 2; node 1 is rejected, so node 2 (whose parent row has a 5e-5 gap) is never
    # evaluated; the root row's own gap is wide
    parent = _chain(3)
    z = np.array([[2.0, 0.0, 0.0, 0.0],
                  [0.0, 1.0, 1.0 - 5e-5, 0.0],
                  [0.0, 0.0, 0.0, 1.0]])
    r = oracle.verify_request(parent, 3, np.array([0, 3, 1]), z, "greedy", 0.0, 0, 0, 0, 0)
    assert r["path"] == [0] and r["path_margins"] == 0
    # accepting node 1 instead evaluates node 2 and counts it
    r = oracle.verify_request(parent, 3, np.array([0, 0, 1]), z, "greedy", 0.0, 0, 0, 0, 0)
    assert r["path"] == [0, 1, 2] and r["path_margins"] == 1


def test_greedy_bonus_flag_follows_endpoint_gap():
    parent = np.array([-1, 0])
    z = np.array([[0.0, 1.0, -1.0],
                  [0.5, 0.5 - 3e-5, 0.1]])
    r = oracle.verify_request(parent, 2, np.array([0, 1]), z, "greedy", 0.0, 0, 0, 0, 0)
    assert r["path"] == [0, 1] and r["path_margins"] == 0
    assert r["bonus"] == 0 and r["bonus_margin"] is True and r["bonus_window"] == (0, 0)


# ---- typical --------------------------------------------------------------------------------

def _typical(p_row, token, eps, delta):
    parent = np.array([-1, 0])
    z = np.log(np.stack([np.asarray(p_row), np.full(len(p_row), 1.0 / len(p_row))]))
    return oracle.verify_request(parent, 2, np.array([0, token]), z, "typical", 1.0, eps, delta, 0, 0)


@pytest.mark.parametrize("log_ratio,accepted,flagged", [
    (5e-5, True, True), (-5e-5, False, True), (2e-4, True, False), (-2e-4, False, False)])
def test_typical_band_with_eps_binding(log_ratio, accepted, flagged):
    # V = 4, eps = 0.25 and delta = 10: delta * exp(-H) >= 10 / 4 > eps, so thr = 0.25;
    # p(x) = 0.25 * e^{log_ratio}, the other three share the rest
    p0 = 0.25 * math.exp(log_ratio)
    r = _typical([p0] + [(1 - p0) / 3] * 3, 0, eps=0.25, delta=10.0)
    assert r["path"] == ([0, 1] if accepted else [0])
    assert r["path_margins"] == (1 if flagged else 0)


@pytest.mark.parametrize("log_ratio,accepted,flagged", [
    (5e-5, True, True), (-5e-5, False, True), (3e-4, True, False), (-3e-4, False, False)])
def test_typical_band_with_entropy_binding(log_ratio, accepted, flagged):
    # p = (0.4, 0.2, 0.2, 0.2): H = -0.4 ln 0.4 - 0.6 ln 0.2 = 1.332179...; eps = 0.9 does not
    # bind; delta is set so that thr = delta e^{-H} = 0.4 e^{-log_ratio}
    H = -0.4 * math.log(0.4) - 3 * 0.2 * math.log(0.2)
    assert abs(H - 1.3321790402101223) < 1e-12
    delta = 0.4 * math.exp(-log_ratio) * math.exp(H)
    r = _typical([0.4, 0.2, 0.2, 0.2], 0, eps=0.9, delta=delta)
    assert r["path"] == ([0, 1] if accepted else [0])
    assert r["path_margins"] == (1 if flagged else 0)


def test_typical_zero_threshold_is_never_a_margin():
    r = _typical([0.4, 0.2, 0.2, 0.2], 3, eps=0.0, delta=0.3)   # thr = 0 accepts everything
    assert r["path"] == [0, 1] and r["path_margins"] == 0


# ---- rejection ------------------------------------------------------------------------------

_T = np.array([0.5, 0.3, 0.2])
_D = np.array([0.2, 0.6, 0.2])


def _rejection(parent, tokens, u0, u1=0.5):
    n = len(parent)
    z = np.log(np.stack([_T] * n))
    return oracle.verify_request(parent, n, np.asarray(tokens), z, "rejection", 1.0, 0, 0, 0, 0,
                                 draft_row=lambda e: _D,
                                 u_fn=lambda node, purpose: u0[node] if purpose == 0 else u1)


@pytest.mark.parametrize("du,accepted,flagged", [
    (5e-5, False, True), (-5e-5, True, True), (2e-4, False, False), (-2e-4, True, False)])
def test_rejection_band(du, accepted, flagged):
    # x = 1: a = min(1, 0.3 / 0.6) = 0.5; u = 0.5 + du
    r = _rejection(np.array([-1, 0]), [0, 1], {1: 0.5 + du})
    assert r["path"] == ([0, 1] if accepted else [0])
    assert r["path_margins"] == (1 if flagged else 0)
    if not accepted:
        # residual relu(T - D) / sum = (0.3, 0, 0) / 0.3: the bonus is token 0 for any u'
        assert r["bonus"] == 0


def test_rejection_counts_every_sibling_tried():
    # two siblings: the first (x = 1, a = 0.5) is rejected inside the band; the residual becomes
    # (1, 0, 0), so the second (x = 0, D = 0.2) has a = min(1, 1 / 0.2) = 1 and u = 0.99995 is
    # inside the band and accepted
    r = _rejection(np.array([-1, 0, 0]), [0, 1, 0], {1: 0.50005, 2: 0.99995})
    assert r["path"] == [0, 2] and r["path_margins"] == 2
    # against the un-updated R (a plausible mistake) the second ratio would be 0.5 / 0.2 -> 1 as
    # well, so also pin a case where the update decides: x = 2 after the first rejection has
    # R[2] = 0 -> a = 0, rejected whatever u is (u = 3e-5 is then a margin case)
    r = _rejection(np.array([-1, 0, 0]), [0, 1, 2], {1: 0.9, 2: 3e-5})
    assert r["path"] == [0] and r["path_margins"] == 1


# ---- bonus window ---------------------------------------------------------------------------

@pytest.mark.parametrize("u1,bonus,near,window", [
    (0.30003, 2, True, (1, 2)),     # 3e-5 above the boundary C_1 = 0.3
    (0.29997, 1, True, (1, 2)),     # 3e-5 below it
    (0.45, 2, False, (2, 2)),
    (0.59998, 2, True, (2, 3)),
    (0.99995, 3, True, (3, 3)),     # the window is clipped to the last index
    (0.5e-4, 0, True, (0, 0)),      # within the band of the start of the first interval
])
def test_bonus_window_hand_cumsum(u1, bonus, near, window):
    # root-only tree, R = T_root = (0.1, 0.2, 0.3, 0.4): cumulative sums 0.1, 0.3, 0.6, 1.0
    z = np.log(np.array([[0.1, 0.2, 0.3, 0.4]]))
    r = oracle.verify_request(np.array([-1]), 1, np.array([0]), z, "rejection", 1.0, 0, 0, 0, 0,
                              draft_row=lambda e: None, u_fn=lambda node, purpose: u1)
    assert r["path"] == [0] and r["path_margins"] == 0
    assert r["bonus"] == bonus
    assert r["bonus_margin"] is near
    assert r["bonus_window"] == window


# ---- draft-to-target scatter ----------------------------------------------------------------

def test_draft_scatter_hand_example():
    got = draft_in_target_vocab([0.5, 0.3, 0.2], np.array([4, 1, 2]), 6)
    assert got.tolist() == [0.0, 0.3, 0.2, 0.0, 0.5, 0.0]
    ident = draft_in_target_vocab([0.1, 0.9], None, 2)
    assert ident.tolist() == [0.1, 0.9]


def _mapped_case(token, seed):
    """B = 1, root + one child, V = 6 target ids, draft vocabulary of 3 mapped to ids (4, 1, 2).
    W = I and hidden = ln T make the logits exactly ln T."""
    V = 6
    T = np.array([0.01, 0.29, 0.2, 0.1, 0.01, 0.39])
    hidden = np.log(np.stack([T, np.full(V, 1.0 / V)]))[None]      # [1][2][6]
    W = np.eye(V)
    draft = np.zeros((1, 2, 3))
    draft[0, 0] = [0.5, 0.3, 0.2]
    draft[0, 1] = [1 / 3] * 3
    return oracle.verify_accept(hidden, W, np.array([[0, token]]), np.array([[-1, 0]]), np.array([2]),
                                "rejection", 1.0, 0, 0, seed, draft_probs=draft,
                                draft_to_target=np.array([4, 1, 2]))[0], T


def test_draft_map_drives_the_walk():
    seed = 123
    u = float(oracle.uniforms(seed, 0, 1, 0))
    assert u > 0.02          # precondition of the cases below
    # target id 0 is outside the map: D[0] = 0 < T[0], ratio 1 -> accepted whatever u is (read
    # through the identity instead, D[0] would be 0.5 and a = 0.02 < u would reject)
    r, _ = _mapped_case(0, seed)
    assert r["path"] == [0, 1]
    # target id 4 is draft id 0: D[4] = 0.5, a = 0.01 / 0.5 = 0.02 < u -> rejected; the residual
    # relu(T - D) is zero on ids 1 (0.29 - 0.3 < 0) and 4, so the bonus is never 1 or 4
    r, T = _mapped_case(4, seed)
    assert r["path"] == [0]
    res = np.maximum(T - np.array([0.0, 0.3, 0.2, 0.0, 0.5, 0.0]), 0)
    C = np.cumsum(res / res.sum())
    u1 = float(oracle.uniforms(seed, 0, 0, 1))
    assert r["bonus"] == int(np.searchsorted(C, u1 * C[-1], side="right"))
    assert r["bonus"] not in (1, 4)

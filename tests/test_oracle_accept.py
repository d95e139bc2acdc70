"""Pins for the oracle's acceptance rules, longest-path selection and bonus token.

* hand-computed typical-acceptance example (probabilities 1/2, 1/4, 1/8, 1/8: H = 1.75 ln 2);
* special cases: tokens equal to the parent's argmax accept the deepest node; delta = 0 accepts
  everything; a threshold above 1 rejects everything; T == D accepts the first child at every
  depth; D[x] = 0 < T[x] always accepts;
* invariants on random trees, checked by an independent breadth-first search: the output is a
  root path, every node on it is accepted, no deeper node is reachable, ties go to the lowest
  index;
* losslessness of rejection sampling ([GUIDE] section "棄却サンプリング": the output has exactly
  the target distribution): chi-square of the first emitted token against T over 10^6 seeded
  trials, and a planted mistake (resampling from T instead of the residual) that must fail.
"""

import concurrent.futures as cf
import multiprocessing as mp
import os
from collections import deque

import numpy as np
import pytest
from scipy.stats import chisquare

import oracle
import oracle.accept as acc
from gen import trees as T


def _bfs_expected(parent, n, accepted):
    """Deepest node reachable from the root through accepted nodes (lowest index on ties)."""
    depth = {0: 0}
    best = 0
    q = deque([0])
    while q:
        e = q.popleft()
        for c in range(1, n):
            if parent[c] == e and accepted[c]:
                depth[c] = depth[e] + 1
                q.append(c)
                if depth[c] > depth[best] or (depth[c] == depth[best] and c < best):
                    best = c
    return best, depth[best]


def _random_case(rng, n, V):
    parent = np.full(n, -1)
    for i in range(1, n):
        parent[i] = rng.integers(0, i)
    z = rng.standard_normal((n, V))
    return parent, z


@pytest.mark.parametrize("seed", range(6))
def test_greedy_invariants_random_trees(seed):
    rng = np.random.default_rng(seed)
    n, V = int(rng.integers(1, 40)), 50
    parent, z = _random_case(rng, n, V)
    coin = rng.random(n) < 0.7
    tokens = np.zeros(n, dtype=int)
    for c in range(1, n):
        am = int(np.argmax(z[parent[c]]))
        tokens[c] = am if coin[c] else (am + 1 + rng.integers(0, V - 1)) % V
    r = oracle.verify_request(parent, n, tokens, z, "greedy", 0.0, 0, 0, 0, 0)
    accepted = [True] + [tokens[c] == int(np.argmax(z[parent[c]])) for c in range(1, n)]
    best, dep = _bfs_expected(parent, n, accepted)
    assert r["path"][-1] == best and r["accept_len"] == dep == len(r["path"]) - 1
    assert r["path"][0] == 0 and all(parent[r["path"][j + 1]] == r["path"][j] for j in range(dep))
    assert all(accepted[c] for c in r["path"])
    assert r["bonus"] == int(np.argmax(z[best]))


def test_greedy_all_argmax_reaches_deepest_lowest_index():
    rng = np.random.default_rng(9)
    parent, _ = T.random_bfs_tree(rng, 80, 6)
    n, V = len(parent), 30
    z = rng.standard_normal((n, V))
    tokens = np.array([0] + [int(np.argmax(z[parent[c]])) for c in range(1, n)])
    r = oracle.verify_request(parent, n, tokens, z, "greedy", 0.0, 0, 0, 0, 0)
    d = T.depths(parent)
    deepest = int(np.nonzero(d == d.max())[0][0])
    assert r["accept_len"] == d.max() and r["path"][-1] == deepest


def test_typical_hand_example():
    # p = (1/2, 1/4, 1/8, 1/8): H = 1.75 ln 2, exp(-H) = 2^-1.75 = 0.29730;
    # eps = 0.2, delta = 0.5 -> thr = min(0.2, 0.14865) = 0.14865: tokens 0 and 1 pass, 2 and 3 fail.
    z = np.log(np.array([[0.5, 0.25, 0.125, 0.125]] * 5))
    parent = np.array([-1, 0, 0, 0, 0])
    for tok, ok in ((0, True), (1, True), (2, False), (3, False)):
        tokens = np.array([0, tok, tok, tok, tok])
        r = oracle.verify_request(parent, 5, tokens, z, "typical", 1.0, 0.2, 0.5, 0, 0)
        assert r["accept_len"] == (1 if ok else 0)
        assert r["path"] == ([0, 1] if ok else [0])
    # eps binds instead: eps = 0.3 < delta e^-H = 1.2 * 0.2973 = 0.357 -> only token 0 (0.5)
    tokens = np.array([0, 1, 0, 2, 3])
    r = oracle.verify_request(parent, 5, tokens, z, "typical", 1.0, 0.3, 1.2, 0, 0)
    assert r["path"] == [0, 2]


def test_typical_extremes():
    rng = np.random.default_rng(3)
    parent, _ = T.random_bfs_tree(rng, 40, 5)
    n, V = len(parent), 64
    z = rng.standard_normal((n, V)) * 4
    tokens = rng.integers(0, V, n)
    r = oracle.verify_request(parent, n, tokens, z, "typical", 1.0, 0.09, 0.0, 0, 0)  # thr = 0
    d = T.depths(parent)
    assert r["accept_len"] == d.max() and r["path"][-1] == int(np.nonzero(d == d.max())[0][0])
    r = oracle.verify_request(parent, n, tokens, z, "typical", 1.0, 1.5, 1e9, 0, 0)   # thr > 1
    assert r["accept_len"] == 0 and r["path"] == [0] and r["bonus"] == int(np.argmax(z[0]))


def test_typical_invariants_random():
    for seed in range(5):
        rng = np.random.default_rng(100 + seed)
        n, V = int(rng.integers(2, 50)), 40
        parent, z = _random_case(rng, n, V)
        tokens = rng.integers(0, V, n)
        tau, eps, delta = 0.8, 0.05, 0.3
        r = oracle.verify_request(parent, n, tokens, z, "typical", tau, eps, delta, 0, 0)
        accepted = [True]
        for c in range(1, n):
            y = z[parent[c]] / tau
            p = np.exp(y - y.max())
            p /= p.sum()
            H = -(p * np.log(p)).sum()
            accepted.append(p[tokens[c]] >= min(eps, delta * np.exp(-H)))
        best, dep = _bfs_expected(parent, n, accepted)
        assert r["path"][-1] == best and r["accept_len"] == dep


def _rej(parent, tokens, z, D, seed=1, b=0):
    n = len(parent)
    return oracle.verify_request(parent, n, tokens, z, "rejection", 1.0, 0, 0, seed, b,
                                 draft_row=lambda e: D[e])


def test_rejection_equal_distributions_accepts_first_children():
    rng = np.random.default_rng(4)
    parent, _ = T.random_bfs_tree(rng, 50, 6)
    n, V = len(parent), 16
    D = rng.dirichlet(np.ones(V), n)
    z = np.log(D)
    tokens = rng.integers(0, V, n)
    for seed in range(5):
        r = _rej(parent, tokens, z, D, seed=seed)
        e, path = 0, [0]
        while True:
            kids = oracle.children(parent, n, e)
            if not kids:
                break
            e = kids[0]
            path.append(e)
        assert r["path"] == path


def test_rejection_zero_draft_mass_accepts_and_zero_target_rejects():
    parent = np.array([-1, 0, 0])
    V = 4
    T0 = np.array([0.4, 0.3, 0.2, 0.1])
    D0 = np.array([0.5, 0.5, 0.0, 0.0])
    z = np.log(np.stack([T0, T0, T0]))
    D = np.stack([D0, D0, D0])
    r = _rej(parent, np.array([0, 2, 1]), z, D)          # D[2] = 0 < T[2]: always accepted
    assert r["path"] == [0, 1]
    T1 = np.array([0.5, 0.5, 0.0, 0.0])                   # T[2] = 0: always rejected
    z1 = np.log(np.maximum(np.stack([T1, T1, T1]), 1e-300))
    z1[:, 2:] = -np.inf
    for seed in range(20):
        r = _rej(parent, np.array([0, 2, 2]), z1, np.stack([np.full(4, 0.25)] * 3), seed=seed)
        assert r["path"] == [0] and r["bonus"] in (0, 1)


def test_rejection_path_invariants_and_window():
    rng = np.random.default_rng(8)
    for trial in range(20):
        parent, _ = T.random_bfs_tree(rng, 30, 5)
        n, V = len(parent), 200
        z = rng.standard_normal((n, V)) * 2
        D = rng.dirichlet(np.ones(V) * 0.3, n)
        tokens = np.array([0] + [rng.choice(V, p=D[parent[c]]) for c in range(1, n)])
        r = _rej(parent, tokens, z, D, seed=trial, b=trial)
        p = r["path"]
        assert p[0] == 0 and all(parent[p[j + 1]] == p[j] for j in range(len(p) - 1))
        lo, hi = r["bonus_window"]
        assert lo <= r["bonus"] <= hi


# ---- losslessness: chi-square over 10^6 seeded trials ---------------------------------------

_V = 8
_T_ROOT = np.array([0.30, 0.05, 0.20, 0.10, 0.02, 0.13, 0.15, 0.05])
_D_ROOT = np.array([0.05, 0.25, 0.10, 0.10, 0.20, 0.05, 0.05, 0.20])
_SEED = 20241202


def _chisq_worker(args):
    lo, hi, planted = args
    import oracle.accept as a
    if planted:  # the planted mistake: resample from R itself instead of relu(R - D)
        a._residual = lambda R, De: R
    rng = np.random.default_rng(lo)
    parent = np.array([-1, 0, 0, 0])
    z = np.log(np.stack([_T_ROOT, np.full(_V, 1 / _V), np.full(_V, 1 / _V), np.full(_V, 1 / _V)]))
    reqs = np.arange(lo, hi)
    u0 = np.stack([oracle.uniforms(_SEED, reqs, c, 0) for c in range(4)], axis=1)
    u1 = np.stack([oracle.uniforms(_SEED, reqs, e, 1) for e in range(4)], axis=1)
    draws = rng.choice(_V, size=(hi - lo, 3), p=_D_ROOT)
    counts = np.zeros(_V, dtype=np.int64)
    for t in range(hi - lo):
        tokens = np.array([0, draws[t, 0], draws[t, 1], draws[t, 2]])
        r = a.verify_request(parent, 4, tokens, z, "rejection", 1.0, 0, 0, _SEED, lo + t,
                             draft_row=lambda e: _D_ROOT,
                             u_fn=lambda node, purpose: (u0 if purpose == 0 else u1)[t, node])
        first = tokens[r["path"][1]] if r["accept_len"] >= 1 else r["bonus"]
        counts[first] += 1
    return counts


def _run_trials(n, planted):
    workers = max(1, min(16, os.cpu_count() or 1))
    chunks = [(i * n // workers, (i + 1) * n // workers, planted) for i in range(workers)]
    with cf.ProcessPoolExecutor(workers, mp_context=mp.get_context("spawn")) as ex:
        return sum(ex.map(_chisq_worker, chunks))


def test_rejection_sampling_is_lossless_chi_square():
    n = 1_000_000
    counts = _run_trials(n, planted=False)
    assert counts.sum() == n
    p = chisquare(counts, n * _T_ROOT).pvalue
    assert p > 1e-3, (counts, p)


def test_chi_square_catches_planted_residual_mistake():
    n = 200_000
    counts = _run_trials(n, planted=True)
    p = chisquare(counts, n * _T_ROOT).pvalue
    assert p < 1e-3, (counts, p)

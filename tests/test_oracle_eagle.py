"""Pins of the oracle's layered (EAGLE-2 style) dynamic tree construction."""

import itertools

import numpy as np

import oracle


def test_expand_hand_example():
    lp = np.log(np.array([[0.5, 0.2, 0.2, 0.1],
                          [0.1, 0.6, 0.3, 0.0001]], dtype=np.float64)).astype(np.float32)
    fs = np.array([-0.1, -1.0], dtype=np.float32)
    r = oracle.expand_layer(lp, fs, topk=2, next_k=3, frontier_cand=[7, 9])
    assert r["token"].tolist() == [0, 1, 1, 2]          # ties (0.2, 0.2) go to the lower id
    assert r["parent"].tolist() == [7, 7, 9, 9]
    # scores by hand: -0.1 + ln .5 = -0.793, -0.1 + ln .2 = -1.709, -1 + ln .6 = -1.511, -1 + ln .3 = -2.204
    assert np.allclose(r["score"], [-0.793147, -1.709438, -1.510826, -2.203973], atol=1e-5)
    assert r["score"].dtype == np.float32 and r["score"][0] == np.float32(fs[0] + lp[0, 0])
    assert r["next_index"].tolist() == [0, 2, 1]
    assert r["next_score"].tolist() == [r["score"][0], r["score"][2], r["score"][1]]


def test_invalid_frontier_rows_have_no_children():
    lp = np.log(np.full((3, 5), 0.2)).astype(np.float32)
    r = oracle.expand_layer(lp, np.zeros(3, np.float32), topk=2, next_k=8, frontier_valid=[1, 0, 1])
    assert (r["token"][2:4] == -1).all() and (r["score"][2:4] == -np.inf).all()
    assert r["next_index"].tolist() == [0, 1, 4, 5, -1, -1, -1, -1]


def _closed(kept, parent):
    return all(l == 0 or (l - 1, int(parent[l][j])) in kept for (l, j) in kept)


def test_selected_tree_is_the_best_closed_set_by_brute_force():
    """Scores non-increasing along parents: the kept set is closed and has the largest score sum
    of all parent-closed candidate sets of its size (enumerated)."""
    rng = np.random.default_rng(0)
    for _ in range(60):
        D, C = 3, 3
        parent = rng.integers(0, C, size=(D, C))
        score = np.zeros((D, C), dtype=np.float32)
        score[0] = -rng.exponential(1.0, C).astype(np.float32)
        for l in range(1, D):
            for j in range(C):
                score[l, j] = np.float32(score[l - 1, parent[l, j]] - np.float32(rng.exponential(1.0)))
        n = int(rng.integers(1, D * C + 2))
        tp, tt, nn, nc = oracle.select_tree(score, np.arange(D * C).reshape(D, C), parent, n)
        kept = {(int(c) // C, int(c) % C) for c in nc[1:nn]}
        assert nn == min(n, D * C + 1) and _closed(kept, parent)
        best = -np.inf
        allc = [(l, j) for l in range(D) for j in range(C)]
        for sub in itertools.combinations(allc, nn - 1):
            if _closed(set(sub), parent):
                best = max(best, sum(float(score[lj]) for lj in sub))
        assert abs(sum(float(score[lj]) for lj in kept) - best) < 1e-4
        # breadth-first numbering and parent links
        for i in range(1, nn):
            l, j = divmod(int(nc[i]), C)
            assert (i == 1 or nc[i - 1] < nc[i]) and tt[i] == l * C + j
            assert tp[i] == 0 if l == 0 else nc[tp[i]] == (l - 1) * C + parent[l, j]


def test_multi_layer_scores_are_path_sums():
    """Expand three layers from random log-probabilities; every kept node's score equals the
    float32 running sum of log p along its path."""
    rng = np.random.default_rng(1)
    F, k, Vd, D, n = 4, 3, 50, 3, 20
    lps, layers = [], []
    front_score, front_cand = np.zeros(1, np.float32), np.full(1, -1)
    for l in range(D):
        Fl = len(front_score)
        z = rng.standard_normal((Fl, Vd))
        lp = (z - np.log(np.exp(z).sum(1, keepdims=True))).astype(np.float32)
        r = oracle.expand_layer(lp, front_score, k, F, frontier_cand=front_cand)
        lps.append((lp, front_cand.copy()))
        layers.append(r)
        good = r["next_index"] >= 0
        front_cand = r["next_index"][good]
        front_score = r["next_score"][good]
    C = max(len(r["score"]) for r in layers)
    S = np.full((D, C), -np.inf, np.float32)
    Tk = np.full((D, C), -1)
    P = np.full((D, C), -1)
    for l, r in enumerate(layers):
        S[l, : len(r["score"])] = r["score"]
        Tk[l, : len(r["token"])] = r["token"]
        P[l, : len(r["parent"])] = r["parent"]
    tp, tt, nn, nc = oracle.select_tree(S, Tk, P, n)
    for i in range(1, nn):
        path, x = [], i
        while x > 0:
            path.append(int(nc[x]))
            x = tp[x]
        acc = np.float32(0.0)
        for c in reversed(path):
            l, j = divmod(c, C)
            f = j // k
            acc = np.float32(acc + lps[l][0][f, Tk[l, j]])
        assert acc == S[divmod(int(nc[i]), C)]

"""Seeded construction of complete tree-verification inputs.

Every array comes from one ``numpy.random.Generator(PCG64(seed))``.  Recipe:

* q, K/V cache, hidden states ~ N(0, 1); LM-head weight W ~ N(0, 1/hidden).  bf16 workloads
  round those float32 draws to bf16 (round to nearest even) and store the bit patterns.
* KV cache layout [B][Hkv][L_cap][d]: request b's prefix occupies slots [0, L_b); tree node i
  sits in slot L_b + i (its key/value as computed by the target's forward for that node).
* Drafted tokens (the drafter is simulated; see the package docstring):
    - "rank": child of p with sibling rank r takes the rank-r token of the draft logits
      rho * z_p + sqrt(1 - rho^2) * xi, xi ~ N(0, 1) per vocab entry, z_p = W h_p (float32).
    - "iid": draft distribution D_p = softmax((z_p + xi) / tau), xi ~ N(0, sigma^2); the
      children of p are drawn i.i.d. from D_p.
    - "dynamic": best-first tree over a draft vocabulary mapped injectively into the target
      vocabulary; D_p = softmax(z_p[map] + xi), xi ~ N(0, sigma^2); the unexpanded node with
      the highest cumulative ln D (depth limit) is expanded with its top-k draft tokens until
      the tree has its node budget.
* The acceptance uniforms are not drawn here: both sides derive them from a counter-based
  generator keyed by (seed, request, node, purpose).
"""

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import trees as T
from .bf16 import bf16_bits_to_f32, bf16_bits_to_f64, normal_bf16
from .configs import CONFIGS


@dataclass
class Case:
    name: str
    dtype: str            # "f32" or "bf16" (bf16 arrays hold uint16 bit patterns)
    B: int
    N: int                # padded nodes per request (root included)
    Hq: int
    Hkv: int
    d: int
    Hd: int
    V: int
    L_cap: int
    q: np.ndarray         # [B][N][Hq][d]
    k_cache: np.ndarray   # [B][Hkv][L_cap][d]
    v_cache: np.ndarray   # [B][Hkv][L_cap][d]
    prefix_len: np.ndarray  # int32 [B]
    n_nodes: np.ndarray     # int32 [B]
    parent: np.ndarray      # int32 [B][N], -1 for the root and for padded nodes
    hidden: np.ndarray      # [B][N][Hd]
    W: np.ndarray           # [V][Hd]
    tokens: np.ndarray      # int32 [B][N] (target-vocab ids; 0 for the root and padding)
    rule: str               # "greedy" | "typical" | "rejection"
    tau: float
    eps: float
    delta: float
    seed: int               # key of the acceptance uniforms
    draft_probs: Optional[np.ndarray] = None      # float32 [B][N][Vd] (rejection only)
    draft_to_target: Optional[np.ndarray] = None  # int32 [Vd] (None = identity)
    meta: dict = field(default_factory=dict)

    def f64(self, name):
        """Exact float64 view of a floating-point input (bf16 bits are widened exactly)."""
        a = getattr(self, name)
        if self.dtype == "bf16":
            return bf16_bits_to_f64(a)
        return np.asarray(a, dtype=np.float64)

    def f32(self, name):
        a = getattr(self, name)
        if self.dtype == "bf16":
            return bf16_bits_to_f32(a)
        return np.asarray(a, dtype=np.float32)

    @property
    def draft_vocab(self):
        return 0 if self.draft_probs is None else self.draft_probs.shape[-1]


def _normal(rng, shape, dtype, std=1.0):
    if dtype == "bf16":
        return normal_bf16(rng, shape, std)
    out = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def _as_f32(a, dtype):
    return bf16_bits_to_f32(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


def _draft_target_logits(W, rows, dtype, chunk=8192):
    """Float32 W @ h for the drafter simulation (rows: [n][Hd] float32) -> [n][V] float32."""
    V = W.shape[0]
    out = np.empty((rows.shape[0], V), dtype=np.float32)
    for v0 in range(0, V, chunk):
        w = _as_f32(W[v0:v0 + chunk], dtype)
        out[:, v0:v0 + chunk] = rows @ w.T
    return out


def _top_ranks(scores, k):
    """Indices of the k largest scores, largest first, lower index first on ties."""
    k = min(k, scores.size)
    idx = np.argpartition(-scores, k - 1)[:k] if k < scores.size else np.arange(scores.size)
    order = np.lexsort((idx, -scores[idx]))
    return idx[order]


def _softmax64(x):
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def make_case(*, dtype, Hq, Hkv, d, Hd, V, prefix_len, parents, ranks=None, N=None,
              rule="greedy", tau=0.0, eps=0.09, delta=0.3, seed=0, tokens=("rank", 0.7),
              name="custom", L_cap=None, draft_vocab=None, rng=None):
    """Build a Case from explicit trees.

    parents: list of per-request parent arrays (topological order, root first).
    tokens:  ("rank", rho) | ("iid", tau_d, sigma) | ("given", int array [B][N]).
    """
    rng = np.random.default_rng(seed) if rng is None else rng
    B = len(parents)
    n_nodes = np.array([len(p) for p in parents], dtype=np.int32)
    N = int(n_nodes.max()) if N is None else int(N)
    if N < n_nodes.max():
        raise ValueError("N smaller than a tree")
    prefix_len = np.asarray(prefix_len, dtype=np.int32).reshape(B)
    if L_cap is None:
        L_cap = int((prefix_len + N).max())
    parent = np.full((B, N), -1, dtype=np.int32)
    rank = np.zeros((B, N), dtype=np.int32)
    for b, p in enumerate(parents):
        parent[b, : len(p)] = p
        rank[b, : len(p)] = T.sibling_rank(p) if ranks is None else ranks[b]

    q = _normal(rng, (B, N, Hq, d), dtype)
    k_cache = _normal(rng, (B, Hkv, L_cap, d), dtype)
    v_cache = _normal(rng, (B, Hkv, L_cap, d), dtype)
    hidden = _normal(rng, (B, N, Hd), dtype)
    W = _normal(rng, (V, Hd), dtype, std=1.0 / np.sqrt(Hd))

    toks = np.zeros((B, N), dtype=np.int32)
    draft_probs = None
    draft_to_target = None
    mode = tokens[0]
    if mode == "given":
        toks[:] = np.asarray(tokens[1], dtype=np.int32)
    elif mode in ("rank", "iid"):
        internal = [(b, p) for b in range(B) for p in sorted(set(parent[b, 1:n_nodes[b]].tolist()))]
        if mode == "iid":
            Vd = V if draft_vocab is None else draft_vocab
            if Vd != V:
                raise ValueError("iid drafting draws over the full target vocabulary")
            draft_probs = np.zeros((B, N, V), dtype=np.float32)
        if internal:
            hs = np.stack([_as_f32(hidden[b, p], dtype) for b, p in internal])
            z = _draft_target_logits(W, hs, dtype)
            for row, (b, p) in enumerate(internal):
                kids = [c for c in range(1, n_nodes[b]) if parent[b, c] == p]
                if mode == "rank":
                    rho = tokens[1]
                    s = rho * z[row] + np.sqrt(1.0 - rho * rho) * rng.standard_normal(V, dtype=np.float32)
                    top = _top_ranks(s, int(max(rank[b, c] for c in kids)) + 1)
                    for c in kids:
                        toks[b, c] = top[rank[b, c]]
                else:
                    tau_d, sigma = tokens[1], tokens[2]
                    Dp = _softmax64((z[row].astype(np.float64) + sigma * rng.standard_normal(V)) / tau_d)
                    draft_probs[b, p] = Dp.astype(np.float32)
                    draws = rng.choice(V, size=len(kids), p=Dp)
                    for c, x in zip(kids, draws):
                        toks[b, c] = x
    else:
        raise ValueError(f"unknown token mode {mode}")

    return Case(name=name, dtype=dtype, B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, Hd=Hd, V=V, L_cap=int(L_cap),
                q=q, k_cache=k_cache, v_cache=v_cache, prefix_len=prefix_len, n_nodes=n_nodes,
                parent=parent, hidden=hidden, W=W, tokens=toks, rule=rule, tau=float(tau),
                eps=float(eps), delta=float(delta), seed=int(seed),
                draft_probs=draft_probs, draft_to_target=draft_to_target)


def _make_dynamic(spec, seed, rng):
    """Best-first dynamic trees over a mapped draft vocabulary (EAGLE-2/3-style drafting)."""
    B, Hq, Hkv, d, Hd, V = spec["B"], spec["Hq"], spec["Hkv"], spec["d"], spec["Hd"], spec["V"]
    dtype = spec["dtype"]
    _, n_total, max_depth, topk = spec["tree"]
    _, Vd, sigma = spec["tokens"]
    prefix_len = np.asarray(spec["prefix"][1], dtype=np.int32)
    N = n_total
    L_cap = int((prefix_len + N).max())
    q = _normal(rng, (B, N, Hq, d), dtype)
    k_cache = _normal(rng, (B, Hkv, L_cap, d), dtype)
    v_cache = _normal(rng, (B, Hkv, L_cap, d), dtype)
    hidden = _normal(rng, (B, N, Hd), dtype)
    W = _normal(rng, (V, Hd), dtype, std=1.0 / np.sqrt(Hd))
    dmap = rng.permutation(V)[:Vd].astype(np.int32)

    parent = np.full((B, N), -1, dtype=np.int32)
    toks = np.zeros((B, N), dtype=np.int32)
    draft_probs = np.zeros((B, N, Vd), dtype=np.float32)
    cum = np.full((B, N), -np.inf)
    cum[:, 0] = 0.0
    depth = np.zeros((B, N), dtype=np.int32)
    count = np.ones(B, dtype=np.int32)
    expanded = np.zeros((B, N), dtype=bool)
    while (count < n_total).any():
        pick = []
        for b in range(B):
            if count[b] >= n_total:
                continue
            cand = [i for i in range(count[b]) if not expanded[b, i] and depth[b, i] < max_depth]
            if not cand:
                count[b] = n_total  # nothing left to expand: the tree stays smaller
                continue
            best = max(cand, key=lambda i: (cum[b, i], -i))
            pick.append((b, best))
        if not pick:
            break
        hs = np.stack([_as_f32(hidden[b, p], dtype) for b, p in pick])
        z = _draft_target_logits(W, hs, dtype)
        for row, (b, p) in enumerate(pick):
            expanded[b, p] = True
            Dp = _softmax64(z[row, dmap].astype(np.float64) + sigma * rng.standard_normal(Vd))
            draft_probs[b, p] = Dp.astype(np.float32)
            top = _top_ranks(Dp, topk)
            for j in top:
                if count[b] >= n_total:
                    break
                c = count[b]
                parent[b, c] = p
                toks[b, c] = dmap[j]
                cum[b, c] = cum[b, p] + np.log(Dp[j])
                depth[b, c] = depth[b, p] + 1
                count[b] += 1
    n_nodes = np.array([(parent[b, 1:] >= 0).sum() + 1 for b in range(B)], dtype=np.int32)
    return Case(name=spec["name"], dtype=dtype, B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, Hd=Hd, V=V,
                L_cap=L_cap, q=q, k_cache=k_cache, v_cache=v_cache, prefix_len=prefix_len,
                n_nodes=n_nodes, parent=parent, hidden=hidden, W=W, tokens=toks,
                rule=spec["rule"], tau=float(spec["tau"]), eps=float(spec["eps"]),
                delta=float(spec["delta"]), seed=int(seed), draft_probs=draft_probs,
                draft_to_target=dmap)


def make_config_case(cfg_id, seed=0):
    """Inputs of workload ``cfg_id`` (1..5) from one integer seed."""
    spec = dict(CONFIGS[cfg_id])
    rng = np.random.default_rng(seed)
    if spec["tree"][0] == "dynamic":
        case = _make_dynamic(spec, seed, rng)
        case.meta["config"] = cfg_id
        return case
    B = spec["B"]
    kind = spec["tree"][0]
    if kind == "root3x2":
        parents = [T.tree_root_3x2() for _ in range(B)]
        ranks = None
    elif kind == "static":
        p, r = T.static_topk_tree(spec["tree"][1], spec["tree"][2])
        parents, ranks = [p] * B, [r] * B
    elif kind == "bfs":
        made = [T.random_bfs_tree(rng, spec["tree"][1], spec["tree"][2]) for _ in range(B)]
        parents, ranks = [m[0] for m in made], [m[1] for m in made]
    else:
        raise ValueError(kind)
    N = max(len(p) for p in parents)
    if kind == "bfs":
        N = spec["tree"][1]  # padded to the node budget
    pre = spec["prefix"]
    if pre[0] == "fixed":
        prefix_len = np.asarray(pre[1], dtype=np.int32)
    else:
        prefix_len = rng.integers(pre[1], pre[2] + 1, size=B).astype(np.int32)
    case = make_case(dtype=spec["dtype"], Hq=spec["Hq"], Hkv=spec["Hkv"], d=spec["d"], Hd=spec["Hd"],
                     V=spec["V"], prefix_len=prefix_len, parents=parents, ranks=ranks, N=N,
                     rule=spec["rule"], tau=spec["tau"], eps=spec["eps"], delta=spec["delta"],
                     seed=seed, tokens=spec["tokens"], name=spec["name"], rng=rng)
    case.meta["config"] = cfg_id
    return case


def compact_draft(draft_probs, parent, n_nodes, rng=None):
    """The draft distributions of the nodes that have children, as a compact [rows][Vd] array and
    a [B][N] row index (-1 for nodes without children): the layout a dynamic drafter produces,
    since it expands only some nodes.  ``rng`` shuffles the row order (a layout check for tests)."""
    B, N = parent.shape
    keys = sorted({(b, int(parent[b, c])) for b in range(B) for c in range(1, int(n_nodes[b]))})
    if rng is not None:
        keys = [keys[i] for i in rng.permutation(len(keys))]
    index = np.full((B, N), -1, dtype=np.int32)
    rows = np.zeros((max(len(keys), 1), draft_probs.shape[-1]), dtype=np.float32)
    for r, (b, e) in enumerate(keys):
        index[b, e] = r
        rows[r] = draft_probs[b, e]
    return rows, index

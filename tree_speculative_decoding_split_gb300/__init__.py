"""GB300-native tree verification for Medusa/EAGLE-style speculative decoding.

Thin ctypes binding of ``libspectree.so`` (C ABI in ``include/spectree.h``).  This module only
marshals arguments: it checks tensor placement, dtype and contiguity, carves nothing itself,
and passes raw device pointers plus the current CUDA stream.  Every step of the computation
runs in the library's CUDA kernels; if the library has not been built, every call raises.

    tree_attention(...)   -> (out, lse)          one attention layer over the draft tree
    verify_accept(...)    -> dict of outputs      LM head, acceptance, longest path, bonus token
    verify_accept_compact(...) -> dict            the same, with the KV compaction folded in
    compact_kv(...)       -> (src_slot, new_len)  in-place KV compaction of the accepted path
    medusa_expand(...)    -> dict of outputs      draft tree tokens from Medusa heads' top-k
    medusa_topology(...)  -> (parent, rank)       pruned Cartesian topology (host arrays)
    eagle_expand(...)     -> dict of outputs      one layer of a dynamic (EAGLE-2 style) draft tree
    eagle_tree(...)       -> dict of outputs      the tree from all layers' candidates
    Round(...)                                    the three verification calls as one graph launch
                                                  (also from host buffers: Round.launch_host)
"""

import ctypes
import os

from ._build import LIB as _LIB_PATH
from ._build import build  # noqa: F401

SPEC_OK = 0
STATUS_NAMES = {
    0: "SPEC_OK", 1: "SPEC_ERR_INVALID_ARGUMENT", 2: "SPEC_ERR_UNSUPPORTED",
    3: "SPEC_ERR_WORKSPACE_TOO_SMALL", 4: "SPEC_ERR_BAD_TREE", 5: "SPEC_ERR_CUDA",
    6: "SPEC_ERR_BAD_TOKEN", 7: "SPEC_ERR_CAPACITY", 8: "SPEC_ERR_TIMEOUT",
}
DTYPE_F32, DTYPE_BF16 = 0, 1
RULES = {"greedy": 0, "typical": 1, "rejection": 2}
MAX_NODES = 255

_vp = ctypes.c_void_p


class AttnArgs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("batch", ctypes.c_int32), ("n_max", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("kv_capacity", ctypes.c_int64), ("scale", ctypes.c_float),
                ("schedule", ctypes.c_int32), ("q", _vp), ("k_cache", _vp), ("v_cache", _vp),
                ("prefix_len", _vp), ("n_nodes", _vp), ("parent", _vp), ("out", _vp), ("lse", _vp),
                ("timing_begin", _vp), ("timing_end", _vp), ("block_table", _vp), ("block_size", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("num_blocks", ctypes.c_int32), ("reserved1", ctypes.c_int32)]


class VerifyArgs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("batch", ctypes.c_int32), ("n_max", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("vocab", ctypes.c_int32), ("rule", ctypes.c_int32),
                ("temperature", ctypes.c_float), ("eps", ctypes.c_float), ("delta", ctypes.c_float),
                ("draft_vocab", ctypes.c_int32), ("path_cap", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("seed", ctypes.c_uint64), ("hidden_states", _vp), ("lm_head_weight", _vp), ("tokens", _vp),
                ("parent", _vp), ("n_nodes", _vp), ("draft_probs", _vp), ("draft_to_target", _vp),
                ("accept_len", _vp), ("path", _vp), ("bonus_token", _vp), ("margin_count", _vp),
                ("bonus_margin", _vp), ("row_max", _vp), ("row_lse", _vp), ("row_entropy", _vp),
                ("row_argmax", _vp), ("timing_begin", _vp), ("timing_end", _vp), ("draft_ready", _vp),
                ("draft_rows", _vp), ("n_draft_rows", ctypes.c_int32), ("reserved1", ctypes.c_int32)]


class CompactArgs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("batch", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("kv_capacity", ctypes.c_int64), ("path_cap", ctypes.c_int32),
                ("reserved0", ctypes.c_int32), ("k_cache", _vp), ("v_cache", _vp), ("prefix_len", _vp),
                ("path", _vp), ("accept_len", _vp), ("src_slot", _vp), ("new_len", _vp), ("block_table", _vp),
                ("block_size", ctypes.c_int32), ("max_blocks", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("reserved1", ctypes.c_int32)]


class HostCopy(ctypes.Structure):
    _fields_ = [("host", _vp), ("device", _vp), ("row_bytes", ctypes.c_size_t), ("rows", ctypes.c_size_t),
                ("host_pitch", ctypes.c_size_t), ("device_pitch", ctypes.c_size_t)]


class MedusaArgs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("n_nodes", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("head_logits", _vp), ("topo_parent", _vp), ("topo_rank", _vp), ("root_token", _vp),
                ("tokens", _vp), ("parent_out", _vp), ("n_nodes_out", _vp), ("topk_index", _vp)]


class EagleExpandArgs(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("frontier", ctypes.c_int32), ("draft_vocab", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("next_k", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("cand_stride", ctypes.c_int64), ("logp", _vp), ("frontier_score", _vp), ("frontier_valid", _vp),
                ("frontier_cand", _vp), ("cand_token", _vp), ("cand_score", _vp), ("cand_parent", _vp),
                ("next_index", _vp), ("next_score", _vp)]


class EagleTreeArgs(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("layers", ctypes.c_int32), ("cands", ctypes.c_int32),
                ("n_max", ctypes.c_int32), ("draft_vocab", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("score", _vp), ("token", _vp), ("parent", _vp), ("draft_to_target", _vp), ("root_token", _vp),
                ("tree_parent", _vp), ("tree_token", _vp), ("n_nodes", _vp), ("node_cand", _vp)]


_lib_handle = None


def lib():
    """The loaded libspectree.so (raises if it has not been built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "tree_speculative_decoding_split_gb300.build() (no fallback exists)")
        L = ctypes.CDLL(_LIB_PATH)
        for name, argt in (("spec_tree_attention", [ctypes.POINTER(AttnArgs), _vp, ctypes.c_size_t, _vp, _vp]),
                           ("spec_verify_accept", [ctypes.POINTER(VerifyArgs), _vp, ctypes.c_size_t, _vp, _vp]),
                           ("spec_compact_kv", [ctypes.POINTER(CompactArgs), _vp, _vp])):
            fn = getattr(L, name)
            fn.argtypes = argt
            fn.restype = ctypes.c_int32
        L.spec_tree_attention_workspace.argtypes = [ctypes.POINTER(AttnArgs)]
        L.spec_tree_attention_workspace.restype = ctypes.c_size_t
        L.spec_verify_accept_workspace.argtypes = [ctypes.POINTER(VerifyArgs)]
        L.spec_verify_accept_workspace.restype = ctypes.c_size_t
        L.spec_status_string.argtypes = [ctypes.c_int32]
        L.spec_status_string.restype = ctypes.c_char_p
        L.spec_verify_accept_compact.argtypes = [ctypes.POINTER(VerifyArgs), _vp, ctypes.c_size_t,
                                                 ctypes.POINTER(CompactArgs), _vp, _vp]
        L.spec_verify_accept_compact.restype = ctypes.c_int32
        L.spec_round_create.argtypes = [ctypes.POINTER(AttnArgs), _vp, ctypes.c_size_t, ctypes.POINTER(VerifyArgs),
                                        _vp, ctypes.c_size_t, ctypes.POINTER(CompactArgs), _vp,
                                        ctypes.POINTER(_vp)]
        L.spec_round_create.restype = ctypes.c_int32
        L.spec_round_launch.argtypes = [_vp, _vp]
        L.spec_round_launch.restype = ctypes.c_int32
        L.spec_round_launch_host.argtypes = [_vp, ctypes.POINTER(HostCopy), ctypes.c_int32,
                                             ctypes.POINTER(HostCopy), ctypes.c_int32, _vp]
        L.spec_round_launch_host.restype = ctypes.c_int32
        L.spec_round_destroy.argtypes = [_vp]
        L.spec_round_destroy.restype = None
        L.spec_medusa_expand_workspace.argtypes = [ctypes.POINTER(MedusaArgs)]
        L.spec_medusa_expand_workspace.restype = ctypes.c_size_t
        L.spec_medusa_expand.argtypes = [ctypes.POINTER(MedusaArgs), _vp, ctypes.c_size_t, _vp, _vp]
        L.spec_medusa_expand.restype = ctypes.c_int32
        _i32p = ctypes.POINTER(ctypes.c_int32)
        L.spec_medusa_topology.argtypes = [_i32p, ctypes.c_int32, ctypes.c_int32, _i32p, _i32p]
        L.spec_medusa_topology.restype = ctypes.c_int32
        L.spec_eagle_expand_workspace.argtypes = [ctypes.POINTER(EagleExpandArgs)]
        L.spec_eagle_expand_workspace.restype = ctypes.c_size_t
        L.spec_eagle_expand.argtypes = [ctypes.POINTER(EagleExpandArgs), _vp, ctypes.c_size_t, _vp, _vp]
        L.spec_eagle_expand.restype = ctypes.c_int32
        L.spec_eagle_tree.argtypes = [ctypes.POINTER(EagleTreeArgs), _vp, _vp]
        L.spec_eagle_tree.restype = ctypes.c_int32
        _lib_handle = L
    return _lib_handle


def status_string(code):
    return lib().spec_status_string(int(code)).decode()


class SpecError(RuntimeError):
    def __init__(self, code, where):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS_NAMES.get(self.code, self.code)} ({status_string(code)})")


def _check(code, where):
    if code != SPEC_OK:
        raise SpecError(code, where)


# ---- torch marshalling (torch is used for device memory and streams only) ---------------------

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else _vp(t.data_ptr())


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need(t, name, dtype=None, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return _vp(s.cuda_stream)


def _workspace(nbytes, device, workspace):
    torch = _torch()
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def _status_buffer(dev_status, device):
    torch = _torch()
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=device)
    return dev_status


def _paged(k_cache, block_table, B, dev):
    """(block_size, max_blocks, num_blocks, Hkv) of a paged pool [num_blocks][Hkv][block_size][d]."""
    torch = _torch()
    _need(block_table, "block_table", torch.int32, dev)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B][max_blocks]")
    nb, Hkv, bs, _ = k_cache.shape
    return bs, block_table.shape[1], nb, Hkv


SCHEDULES = {"split_kv": 0, "stream_k": 1}


def attn_args(q, k_cache, v_cache, prefix_len, n_nodes, parent, out=None, lse=None, scale=0.0, block_table=None,
              schedule="split_kv"):
    """Build the C argument struct for tree attention (tensors are validated here).  With
    ``block_table`` [B][max_blocks] the caches are paged pools [num_blocks][Hkv][block_size][d];
    ``schedule`` is "split_kv" (default) or "stream_k" (see spec_attn_args.schedule)."""
    torch = _torch()
    _need(q, "q")
    dev = q.device
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, name, q.dtype, dev)
    for name, t in (("prefix_len", prefix_len), ("n_nodes", n_nodes), ("parent", parent)):
        _need(t, name, torch.int32, dev)
    B, N, Hq, d = q.shape
    paged = (0, 0, 0)
    if block_table is not None:
        bs, mb, nb, Hkv = _paged(k_cache, block_table, B, dev)
        L_cap = mb * bs
        paged = (bs, mb, nb)
        if v_cache.shape != k_cache.shape or k_cache.shape[3] != d:
            raise ValueError("pools must be [num_blocks][Hkv][block_size][d]")
    else:
        Hkv, L_cap = k_cache.shape[1], k_cache.shape[2]
        if k_cache.shape != (B, Hkv, L_cap, d) or v_cache.shape != k_cache.shape:
            raise ValueError("cache shape must be [B][Hkv][L_cap][d]")
    if tuple(parent.shape) != (B, N) or prefix_len.numel() != B or n_nodes.numel() != B:
        raise ValueError("parent must be [B][N], prefix_len and n_nodes [B]")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
    _need(out, "out", q.dtype, dev)
    _need(lse, "lse", torch.float32, dev)
    a = AttnArgs(dtype=_dtype_code(q), batch=B, n_max=N, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                 kv_capacity=L_cap, scale=float(scale), schedule=SCHEDULES[schedule], q=_ptr(q), k_cache=_ptr(k_cache),
                 v_cache=_ptr(v_cache), prefix_len=_ptr(prefix_len), n_nodes=_ptr(n_nodes), parent=_ptr(parent),
                 out=_ptr(out), lse=_ptr(lse), block_table=_ptr(block_table), block_size=paged[0],
                 max_blocks=paged[1], num_blocks=paged[2], reserved1=0)
    return a, out, lse


def tree_attention(q, k_cache, v_cache, prefix_len, n_nodes, parent, out=None, lse=None, scale=0.0,
                   workspace=None, dev_status=None, stream=None, block_table=None, schedule="split_kv"):
    """Tree attention (see spec_tree_attention).  Returns (out, lse)."""
    a, out, lse = attn_args(q, k_cache, v_cache, prefix_len, n_nodes, parent, out, lse, scale, block_table,
                            schedule)
    L = lib()
    need = L.spec_tree_attention_workspace(ctypes.byref(a))
    if need == 0:
        _check(L.spec_tree_attention(ctypes.byref(a), None, 0, None, None), "spec_tree_attention")
    ws = _workspace(need, q.device, workspace)
    st = _status_buffer(dev_status, q.device)
    _check(L.spec_tree_attention(ctypes.byref(a), _ptr(ws), need, _ptr(st), _stream(stream)), "spec_tree_attention")
    return out, lse


def verify_args(hidden, weight, tokens, parent, n_nodes, rule, temperature=0.0, eps=0.09, delta=0.3,
                seed=0, draft_probs=None, draft_to_target=None, path_cap=None, hooks=False, outputs=None,
                draft_rows=None):
    """Build the C argument struct for verify_accept; returns (args, outputs dict).

    ``draft_probs`` is [B][N][Vd], or with ``draft_rows`` (int32 [B][N], -1 for nodes without
    children) a compact [rows][Vd] array holding only the expanded nodes' distributions."""
    torch = _torch()
    _need(hidden, "hidden")
    dev = hidden.device
    _need(weight, "weight", hidden.dtype, dev)
    for name, t in (("tokens", tokens), ("parent", parent), ("n_nodes", n_nodes)):
        _need(t, name, torch.int32, dev)
    B, N, Hd = hidden.shape
    V = weight.shape[0]
    if weight.shape[1] != Hd or tuple(tokens.shape) != (B, N) or tuple(parent.shape) != (B, N):
        raise ValueError("shape mismatch")
    if path_cap is None:
        path_cap = N
    rule_code = RULES[rule] if isinstance(rule, str) else int(rule)
    Vd = 0
    if draft_probs is not None:
        _need(draft_probs, "draft_probs", torch.float32, dev)
        Vd = draft_probs.shape[-1]
    if draft_to_target is not None:
        _need(draft_to_target, "draft_to_target", torch.int32, dev)
    n_draft_rows = 0
    if draft_rows is not None:
        _need(draft_rows, "draft_rows", torch.int32, dev)
        if draft_probs is None or draft_probs.dim() != 2 or tuple(draft_rows.shape) != (B, N):
            raise ValueError("draft_rows [B][N] goes with a compact draft_probs [rows][Vd]")
        n_draft_rows = draft_probs.shape[0]
    if outputs is None:
        outputs = dict(
            accept_len=torch.empty(B, dtype=torch.int32, device=dev),
            path=torch.empty((B, path_cap), dtype=torch.int32, device=dev),
            bonus_token=torch.empty(B, dtype=torch.int32, device=dev),
            margin_count=torch.empty(B, dtype=torch.int32, device=dev),
            bonus_margin=torch.empty(B, dtype=torch.int32, device=dev))
        if hooks:
            outputs.update(row_max=torch.empty((B, N), dtype=torch.float32, device=dev),
                           row_lse=torch.empty((B, N), dtype=torch.float32, device=dev),
                           row_entropy=torch.empty((B, N), dtype=torch.float32, device=dev),
                           row_argmax=torch.empty((B, N), dtype=torch.int32, device=dev))
    o = outputs
    a = VerifyArgs(dtype=_dtype_code(hidden), batch=B, n_max=N, hidden=Hd, vocab=V, rule=rule_code,
                   temperature=float(temperature), eps=float(eps), delta=float(delta), draft_vocab=Vd,
                   path_cap=int(path_cap), reserved0=0, seed=int(seed) & 0xFFFFFFFFFFFFFFFF,
                   hidden_states=_ptr(hidden), lm_head_weight=_ptr(weight), tokens=_ptr(tokens),
                   parent=_ptr(parent), n_nodes=_ptr(n_nodes), draft_probs=_ptr(draft_probs),
                   draft_to_target=_ptr(draft_to_target), accept_len=_ptr(o["accept_len"]), path=_ptr(o["path"]),
                   bonus_token=_ptr(o["bonus_token"]), margin_count=_ptr(o.get("margin_count")),
                   bonus_margin=_ptr(o.get("bonus_margin")), row_max=_ptr(o.get("row_max")),
                   row_lse=_ptr(o.get("row_lse")), row_entropy=_ptr(o.get("row_entropy")),
                   row_argmax=_ptr(o.get("row_argmax")), draft_rows=_ptr(draft_rows), n_draft_rows=n_draft_rows,
                   reserved1=0)
    return a, outputs


def verify_accept(hidden, weight, tokens, parent, n_nodes, rule, temperature=0.0, eps=0.09, delta=0.3, seed=0,
                  draft_probs=None, draft_to_target=None, path_cap=None, hooks=False, workspace=None,
                  dev_status=None, stream=None, outputs=None, draft_rows=None):
    """LM head + acceptance + longest path (see spec_verify_accept).  Returns a dict of tensors."""
    a, outputs = verify_args(hidden, weight, tokens, parent, n_nodes, rule, temperature, eps, delta, seed,
                             draft_probs, draft_to_target, path_cap, hooks, outputs, draft_rows)
    L = lib()
    need = L.spec_verify_accept_workspace(ctypes.byref(a))
    if need == 0:
        _check(L.spec_verify_accept(ctypes.byref(a), None, 0, None, None), "spec_verify_accept")
    ws = _workspace(need, hidden.device, workspace)
    st = _status_buffer(dev_status, hidden.device)
    _check(L.spec_verify_accept(ctypes.byref(a), _ptr(ws), need, _ptr(st), _stream(stream)), "spec_verify_accept")
    return outputs


def compact_args(k_cache, v_cache, prefix_len, path, accept_len, src_slot=None, new_len=None, block_table=None):
    torch = _torch()
    _need(k_cache, "k_cache")
    dev = k_cache.device
    _need(v_cache, "v_cache", k_cache.dtype, dev)
    for name, t in (("prefix_len", prefix_len), ("path", path), ("accept_len", accept_len)):
        _need(t, name, torch.int32, dev)
    B = prefix_len.numel()
    paged = (0, 0, 0)
    if block_table is not None:
        bs, mb, nb, Hkv = _paged(k_cache, block_table, B, dev)
        d = k_cache.shape[3]
        L_cap = mb * bs
        paged = (bs, mb, nb)
    else:
        B, Hkv, L_cap, d = k_cache.shape
    path_cap = path.shape[1]
    if src_slot is None:
        src_slot = torch.empty((B, path_cap), dtype=torch.int32, device=dev)
    if new_len is None:
        new_len = torch.empty(B, dtype=torch.int32, device=dev)
    a = CompactArgs(dtype=_dtype_code(k_cache), batch=B, num_kv_heads=Hkv, head_dim=d, kv_capacity=L_cap,
                    path_cap=path_cap, reserved0=0, k_cache=_ptr(k_cache), v_cache=_ptr(v_cache),
                    prefix_len=_ptr(prefix_len), path=_ptr(path), accept_len=_ptr(accept_len),
                    src_slot=_ptr(src_slot), new_len=_ptr(new_len), block_table=_ptr(block_table),
                    block_size=paged[0], max_blocks=paged[1], num_blocks=paged[2], reserved1=0)
    return a, src_slot, new_len


def compact_kv(k_cache, v_cache, prefix_len, path, accept_len, src_slot=None, new_len=None, dev_status=None,
               stream=None, block_table=None):
    """In-place KV compaction (see spec_compact_kv).  Returns (src_slot, new_len)."""
    a, src_slot, new_len = compact_args(k_cache, v_cache, prefix_len, path, accept_len, src_slot, new_len,
                                        block_table)
    st = _status_buffer(dev_status, k_cache.device)
    _check(lib().spec_compact_kv(ctypes.byref(a), _ptr(st), _stream(stream)), "spec_compact_kv")
    return src_slot, new_len


def verify_accept_compact(hidden, weight, tokens, parent, n_nodes, rule, k_cache, v_cache, prefix_len,
                          temperature=0.0, eps=0.09, delta=0.3, seed=0, draft_probs=None, draft_to_target=None,
                          path_cap=None, hooks=False, workspace=None, dev_status=None, stream=None, outputs=None,
                          block_table=None):
    """verify_accept, then the in-place compaction of the accepted paths (spec_verify_accept_compact:
    the compaction runs inside the acceptance kernels).  Returns the verify outputs plus
    ``src_slot`` and ``new_len``."""
    a, outputs = verify_args(hidden, weight, tokens, parent, n_nodes, rule, temperature, eps, delta, seed,
                             draft_probs, draft_to_target, path_cap, hooks, outputs)
    c, src_slot, new_len = compact_args(k_cache, v_cache, prefix_len, outputs["path"], outputs["accept_len"],
                                        block_table=block_table)
    L = lib()
    need = L.spec_verify_accept_workspace(ctypes.byref(a))
    if need == 0:
        _check(L.spec_verify_accept(ctypes.byref(a), None, 0, None, None), "spec_verify_accept")
    ws = _workspace(need, hidden.device, workspace)
    st = _status_buffer(dev_status, hidden.device)
    _check(L.spec_verify_accept_compact(ctypes.byref(a), _ptr(ws), need, ctypes.byref(c), _ptr(st), _stream(stream)),
           "spec_verify_accept_compact")
    outputs["src_slot"] = src_slot
    outputs["new_len"] = new_len
    return outputs


def verify_accept_noalloc(hidden, weight, tokens, parent, n_nodes, rule, temperature=0.0, eps=0.09, delta=0.3,
                          seed=0, draft_probs=None, draft_to_target=None, path_cap=None, hooks=False,
                          dev_status=None, stream=None, outputs=None):
    """verify_accept for callers that cannot allocate device scratch memory.

    Same computation as ``verify_accept``; the library takes its scratch from a fixed device array
    (``NOALLOC_SCRATCH_BYTES``) instead of a workspace, so nothing is allocated for scratch.  Output
    tensors are still the caller's (created here only when ``outputs`` is None).  Calls whose
    kernels overlap on the GPU share that array and race; the first call on a device should come
    before any stream capture.
    """
    a, outputs = verify_args(hidden, weight, tokens, parent, n_nodes, rule, temperature, eps, delta, seed,
                             draft_probs, draft_to_target, path_cap, hooks, outputs)
    fn = lib().spec_verify_accept_noalloc
    fn.argtypes = [ctypes.POINTER(VerifyArgs), _vp, _vp]
    fn.restype = ctypes.c_int32
    st = _status_buffer(dev_status, hidden.device)
    _check(fn(ctypes.byref(a), _ptr(st), _stream(stream)), "spec_verify_accept_noalloc")
    return outputs


NOALLOC_SCRATCH_BYTES = 8 << 20


class Round:
    """One verification round (spec_round_create): tree attention, LM head + acceptance and KV
    compaction captured into a CUDA graph and enqueued with one launch.

    Each of ``attn``, ``verify``, ``compact`` is an argument struct from ``attn_args`` /
    ``verify_args`` / ``compact_args`` (or None to leave that call out).  Every pointer and scalar
    in them is frozen into the graph; refill the tensors they point at in place between
    launches.  The workspaces are allocated here and kept, with the structs' tensors, for the
    round's lifetime.
    """

    def __init__(self, attn=None, verify=None, compact=None, dev_status=None, keep=()):
        torch = _torch()
        L = lib()
        dev = torch.device("cuda", torch.cuda.current_device())
        self._keep = list(keep)
        need_a = L.spec_tree_attention_workspace(ctypes.byref(attn)) if attn is not None else 0
        need_v = L.spec_verify_accept_workspace(ctypes.byref(verify)) if verify is not None else 0
        self.ws_attn = torch.empty(max(need_a, 1), dtype=torch.uint8, device=dev)
        self.ws_verify = torch.empty(max(need_v, 1), dtype=torch.uint8, device=dev)
        self.status = _status_buffer(dev_status, dev)
        self._args = (attn, verify, compact)
        handle = _vp()
        code = L.spec_round_create(ctypes.byref(attn) if attn is not None else None, _ptr(self.ws_attn), need_a,
                                   ctypes.byref(verify) if verify is not None else None, _ptr(self.ws_verify),
                                   need_v, ctypes.byref(compact) if compact is not None else None,
                                   _ptr(self.status), ctypes.byref(handle))
        _check(code, "spec_round_create")
        self._handle = handle

    def launch(self, stream=None):
        """Enqueue the whole round on ``stream`` (default: the current torch stream)."""
        if self._handle is None:
            raise RuntimeError("round destroyed")
        _check(lib().spec_round_launch(self._handle, _stream(stream)), "spec_round_launch")

    def launch_host(self, inputs, outputs, stream=None):
        """One round from host memory (spec_round_launch_host): ``inputs`` and ``outputs`` are
        sequences of HostCopy descriptors (see ``host_copy``), copied in before and out after the
        round, all enqueued on ``stream`` by one C call.  Synchronise before reading the outputs."""
        if self._handle is None:
            raise RuntimeError("round destroyed")
        ins = (HostCopy * max(len(inputs), 1))(*inputs)
        outs = (HostCopy * max(len(outputs), 1))(*outputs)
        _check(lib().spec_round_launch_host(self._handle, ins, len(inputs), outs, len(outputs), _stream(stream)),
               "spec_round_launch_host")

    def close(self):
        if getattr(self, "_handle", None) is not None:
            lib().spec_round_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def host_copy(host, device, rows=None):
    """HostCopy descriptor between a host tensor and a device tensor of the same byte size.

    With ``rows`` = None both must be contiguous (one block).  With ``rows`` = r, the host tensor is
    contiguous [r][...] and ``device`` is a view of r equal-sized rows at a constant stride (e.g. a
    request's tree slots of every KV head in a [Hkv][L_cap][d] cache block); each row must itself
    be contiguous.  The descriptor holds raw pointers: keep both tensors alive until the copies
    have run."""
    nbytes = host.numel() * host.element_size()
    if rows is None:
        if not (host.is_contiguous() and device.is_contiguous()) or \
                device.numel() * device.element_size() != nbytes:
            raise ValueError("host_copy: contiguous tensors of equal size expected")
        return HostCopy(host=_vp(host.data_ptr()), device=_vp(device.data_ptr()), row_bytes=nbytes, rows=1)
    r = int(rows)
    if device.shape[0] != r or not host.is_contiguous() or not device[0].is_contiguous() or \
            device.numel() * device.element_size() != nbytes:
        raise ValueError("host_copy: rows of the device view must be contiguous and match the host tensor")
    row = nbytes // r
    pitch = device.stride(0) * device.element_size()
    return HostCopy(host=_vp(host.data_ptr()), device=_vp(device.data_ptr()), row_bytes=row, rows=r,
                    host_pitch=row, device_pitch=pitch)


def medusa_topology(topk, n_nodes):
    """(parent, rank) numpy int32 arrays of the Cartesian topology of per-head candidate counts
    ``topk`` pruned to ``n_nodes`` nodes (spec_medusa_topology; host only)."""
    import numpy as np
    k = np.ascontiguousarray(np.asarray(topk, dtype=np.int32))
    parent = np.zeros(int(n_nodes), dtype=np.int32)
    rank = np.zeros(int(n_nodes), dtype=np.int32)
    _i32p = ctypes.POINTER(ctypes.c_int32)
    code = lib().spec_medusa_topology(k.ctypes.data_as(_i32p), len(k), int(n_nodes), parent.ctypes.data_as(_i32p),
                                      rank.ctypes.data_as(_i32p))
    _check(code, "spec_medusa_topology")
    return parent, rank


def medusa_args(head_logits, topo_parent, topo_rank, topk, root_token=None, outputs=None):
    """Argument struct and output tensors of spec_medusa_expand.  head_logits [B][K][V] (fp32 or
    bf16); topo_parent / topo_rank int32 [N] on the same device."""
    torch = _torch()
    _need(head_logits, "head_logits")
    dev = head_logits.device
    B, K, V = head_logits.shape
    _need(topo_parent, "topo_parent", torch.int32, dev)
    _need(topo_rank, "topo_rank", torch.int32, dev)
    N = topo_parent.shape[0]
    if root_token is not None:
        _need(root_token, "root_token", torch.int32, dev)
    if outputs is None:
        outputs = {"tokens": torch.empty((B, N), dtype=torch.int32, device=dev),
                   "parent": torch.empty((B, N), dtype=torch.int32, device=dev),
                   "n_nodes": torch.empty(B, dtype=torch.int32, device=dev),
                   "topk_index": torch.empty((B, K, int(topk)), dtype=torch.int32, device=dev)}
    a = MedusaArgs(dtype=_dtype_code(head_logits), batch=B, num_heads=K, vocab=V, n_nodes=N, topk=int(topk),
                   head_logits=_ptr(head_logits), topo_parent=_ptr(topo_parent), topo_rank=_ptr(topo_rank),
                   root_token=_ptr(root_token), tokens=_ptr(outputs["tokens"]), parent_out=_ptr(outputs.get("parent")),
                   n_nodes_out=_ptr(outputs.get("n_nodes")), topk_index=_ptr(outputs.get("topk_index")))
    return a, outputs


def medusa_expand(head_logits, topo_parent, topo_rank, topk, root_token=None, workspace=None, dev_status=None,
                  stream=None, outputs=None):
    """Static Medusa tree expansion (spec_medusa_expand).  Returns a dict of tensors: tokens
    [B][N], parent [B][N], n_nodes [B], topk_index [B][K][topk]."""
    a, outputs = medusa_args(head_logits, topo_parent, topo_rank, topk, root_token, outputs)
    L = lib()
    need = L.spec_medusa_expand_workspace(ctypes.byref(a))
    if need == 0:
        _check(L.spec_medusa_expand(ctypes.byref(a), None, 0, None, None), "spec_medusa_expand")
    ws = _workspace(need, head_logits.device, workspace)
    st = _status_buffer(dev_status, head_logits.device)
    _check(L.spec_medusa_expand(ctypes.byref(a), _ptr(ws), need, _ptr(st), _stream(stream)), "spec_medusa_expand")
    return outputs


def eagle_expand_args(logp, frontier_score, topk, next_k, frontier_valid=None, frontier_cand=None, outputs=None,
                      cand_stride=0):
    """Build the C argument struct for eagle_expand (tensors are validated here); returns
    (args, outputs dict)."""
    torch = _torch()
    _need(logp, "logp", torch.float32)
    dev = logp.device
    B, F, Vd = logp.shape
    _need(frontier_score, "frontier_score", torch.float32, dev)
    for name, t in (("frontier_valid", frontier_valid), ("frontier_cand", frontier_cand)):
        if t is not None:
            _need(t, name, torch.int32, dev)
    C = F * int(topk)
    if outputs is None:
        outputs = {"token": torch.empty((B, C), dtype=torch.int32, device=dev),
                   "score": torch.empty((B, C), dtype=torch.float32, device=dev),
                   "parent": torch.empty((B, C), dtype=torch.int32, device=dev)}
    outputs.setdefault("next_index", torch.empty((B, int(next_k)), dtype=torch.int32, device=dev))
    outputs.setdefault("next_score", torch.empty((B, int(next_k)), dtype=torch.float32, device=dev))
    a = EagleExpandArgs(batch=B, frontier=F, draft_vocab=Vd, topk=int(topk), next_k=int(next_k), reserved0=0,
                        cand_stride=int(cand_stride), logp=_ptr(logp), frontier_score=_ptr(frontier_score),
                        frontier_valid=_ptr(frontier_valid), frontier_cand=_ptr(frontier_cand),
                        cand_token=_vp(outputs["token"].data_ptr()), cand_score=_vp(outputs["score"].data_ptr()),
                        cand_parent=_vp(outputs["parent"].data_ptr()), next_index=_ptr(outputs["next_index"]),
                        next_score=_ptr(outputs["next_score"]))
    return a, outputs


def eagle_expand(logp, frontier_score, topk, next_k, frontier_valid=None, frontier_cand=None, outputs=None,
                 cand_stride=0, workspace=None, dev_status=None, stream=None):
    """One layer of the dynamic draft tree (spec_eagle_expand).  logp float32 [B][F][Vd];
    frontier_score float32 [B][F].  ``outputs`` may pass views into stacked [B][layers][C]
    buffers together with ``cand_stride``.  Returns a dict of tensors."""
    a, outputs = eagle_expand_args(logp, frontier_score, topk, next_k, frontier_valid, frontier_cand, outputs,
                                   cand_stride)
    dev = logp.device
    L = lib()
    need = L.spec_eagle_expand_workspace(ctypes.byref(a))
    if need == 0:
        _check(L.spec_eagle_expand(ctypes.byref(a), None, 0, None, None), "spec_eagle_expand")
    ws = _workspace(need, dev, workspace)
    st = _status_buffer(dev_status, dev)
    _check(L.spec_eagle_expand(ctypes.byref(a), _ptr(ws), need, _ptr(st), _stream(stream)), "spec_eagle_expand")
    return outputs


def eagle_tree_args(score, token, parent, n_max, draft_to_target=None, root_token=None):
    """Build the C argument struct for eagle_tree (tensors are validated here); returns (args,
    outputs dict)."""
    torch = _torch()
    _need(score, "score", torch.float32)
    dev = score.device
    B, D, C = score.shape
    _need(token, "token", torch.int32, dev)
    _need(parent, "parent", torch.int32, dev)
    Vd = 0
    if draft_to_target is not None:
        _need(draft_to_target, "draft_to_target", torch.int32, dev)
        Vd = draft_to_target.numel()
    if root_token is not None:
        _need(root_token, "root_token", torch.int32, dev)
    N = int(n_max)
    out = {"parent": torch.empty((B, N), dtype=torch.int32, device=dev),
           "tokens": torch.empty((B, N), dtype=torch.int32, device=dev),
           "n_nodes": torch.empty(B, dtype=torch.int32, device=dev),
           "node_cand": torch.empty((B, N), dtype=torch.int32, device=dev)}
    a = EagleTreeArgs(batch=B, layers=D, cands=C, n_max=N, draft_vocab=Vd, reserved0=0, score=_ptr(score),
                      token=_ptr(token), parent=_ptr(parent), draft_to_target=_ptr(draft_to_target),
                      root_token=_ptr(root_token), tree_parent=_ptr(out["parent"]), tree_token=_ptr(out["tokens"]),
                      n_nodes=_ptr(out["n_nodes"]), node_cand=_ptr(out["node_cand"]))
    return a, out


def eagle_tree(score, token, parent, n_max, draft_to_target=None, root_token=None, dev_status=None, stream=None):
    """The draft tree from stacked candidates [B][layers][C] (spec_eagle_tree).  Returns a dict:
    parent [B][N], tokens [B][N], n_nodes [B], node_cand [B][N]."""
    a, out = eagle_tree_args(score, token, parent, n_max, draft_to_target, root_token)
    dev = score.device
    st = _status_buffer(dev_status, dev)
    _check(lib().spec_eagle_tree(ctypes.byref(a), _ptr(st), _stream(stream)), "spec_eagle_tree")
    return out

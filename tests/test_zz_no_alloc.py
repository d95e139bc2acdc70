"""The no-allocation variant of spec_verify_accept, called through the C ABI.

Some callers cannot allocate device memory (for instance a plugin inside a host framework that
gives it no access to the allocator, or a latency-critical loop where cudaMalloc would
synchronise the device).  spec_verify_accept_noalloc serves them from a fixed device array.  This
file is collected last so that a failure here leaves every other test already run; it passes both
alone in a fresh process and after the rest of the suite.
"""

import ctypes

import numpy as np
import pytest
import torch

import tree_speculative_decoding_split_gb300 as st
from gen import make_case, trees as T
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _case(dtype, seed, rule):
    rng = np.random.default_rng(seed)
    parents = [T.random_bfs_tree(rng, int(n), 6)[0] for n in (63, 20, 1)]
    return make_case(dtype=dtype, Hq=4, Hkv=1, d=64, Hd=256 if dtype == "bf16" else 64, V=5000,
                     prefix_len=[4, 4, 4], parents=parents, rule=rule, tau=0.0 if rule == "greedy" else 1.0,
                     eps=0.09, delta=0.3, seed=seed, tokens=("rank", 0.8), rng=rng)


def _call(fn_name, case, t, workspace=None):
    a, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                             case.eps, case.delta, case.seed, path_cap=case.N, hooks=True)
    status = torch.zeros(1, dtype=torch.int32, device=t["hidden"].device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    L = st.lib()
    if fn_name == "spec_verify_accept":
        need = L.spec_verify_accept_workspace(ctypes.byref(a))
        ws = torch.empty(need, dtype=torch.uint8, device=t["hidden"].device)
        code = L.spec_verify_accept(ctypes.byref(a), ctypes.c_void_p(ws.data_ptr()), need,
                                    ctypes.c_void_p(status.data_ptr()), stream)
    else:
        fn = L.spec_verify_accept_noalloc
        fn.argtypes = [ctypes.POINTER(st.VerifyArgs), ctypes.c_void_p, ctypes.c_void_p]
        fn.restype = ctypes.c_int32
        code = fn(ctypes.byref(a), ctypes.c_void_p(status.data_ptr()), stream)
    torch.cuda.synchronize()
    assert code == 0, st.status_string(code)
    assert int(status.item()) == 0
    return {k: v.cpu().numpy() for k, v in outs.items()}


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    d = H.dev()
    for seed, dtype, rule in ((1, "bf16", "typical"), (2, "f32", "greedy")):
        case = _case(dtype, seed, rule)
        t = H.to_device(case, d)
        ref = _call("spec_verify_accept", case, t)
        got = _call("spec_verify_accept_noalloc", case, t)
        for k in ("accept_len", "path", "bonus_token", "margin_count", "bonus_margin", "row_argmax"):
            assert (got[k] == ref[k]).all(), k
        tol = H.STAT_TOL[dtype]
        for k in ("row_max", "row_lse", "row_entropy"):
            assert np.abs(got[k] - ref[k]).max() < tol, k


def test_noalloc_rejects_shapes_beyond_its_scratch():
    d = H.dev()
    # rejection sampling keeps fp32 logits: 32 rows x 128256 tokens x 4 B = 16 MB of scratch
    B, N, Hd, V = 1, 32, 256, 128256
    hid = torch.zeros((B, N, Hd), dtype=torch.bfloat16, device=d)
    W = torch.zeros((V, Hd), dtype=torch.bfloat16, device=d)
    tok = torch.zeros((B, N), dtype=torch.int32, device=d)
    par = torch.full((B, N), -1, dtype=torch.int32, device=d)
    nn = torch.full((B,), N, dtype=torch.int32, device=d)
    draft = torch.zeros((B, N, V), dtype=torch.float32, device=d)
    a, _ = st.verify_args(hid, W, tok, par, nn, "rejection", 1.0, 0.09, 0.3, 0, draft_probs=draft, path_cap=N)
    assert st.lib().spec_verify_accept_workspace(ctypes.byref(a)) > st.NOALLOC_SCRATCH_BYTES
    fn = st.lib().spec_verify_accept_noalloc
    fn.argtypes = [ctypes.POINTER(st.VerifyArgs), ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    assert fn(ctypes.byref(a), None, None) == 3  # SPEC_ERR_WORKSPACE_TOO_SMALL, nothing launched

"""C ABI checks that need no GPU: the library loads, exports every declared function, its struct
layouts match the header, and host-side argument errors come back before any launch."""

import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import tree_speculative_decoding_split_gb300 as st

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spectree.h")


@pytest.fixture(scope="module")
def L():
    st.build()
    return st.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert {"spec_tree_attention", "spec_verify_accept", "spec_compact_kv", "spec_status_string",
            "spec_tree_attention_workspace", "spec_verify_accept_workspace"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_struct_layout_matches_header():
    src = r"""
#include <stddef.h>
#include <stdio.h>
#include "spectree.h"
#define P(T, f) printf(#T " " #f " %zu\n", offsetof(T, f));
int main(void) {
  printf("spec_attn_args size %zu\n", sizeof(spec_attn_args));
  printf("spec_verify_args size %zu\n", sizeof(spec_verify_args));
  printf("spec_compact_args size %zu\n", sizeof(spec_compact_args));
  printf("spec_host_copy size %zu\n", sizeof(spec_host_copy));
  P(spec_attn_args, kv_capacity) P(spec_attn_args, q) P(spec_attn_args, lse) P(spec_attn_args, timing_end)
  P(spec_verify_args, seed) P(spec_verify_args, hidden_states) P(spec_verify_args, row_argmax) P(spec_verify_args, timing_end)
  P(spec_compact_args, kv_capacity) P(spec_compact_args, k_cache) P(spec_compact_args, new_len)
  P(spec_host_copy, row_bytes) P(spec_host_copy, device_pitch)
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "l.c")
        exe = os.path.join(td, "l")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {}
    for line in out:
        if line:
            t, f, v = line.split()
            got[(t, f)] = int(v)
    py = {"spec_attn_args": st.AttnArgs, "spec_verify_args": st.VerifyArgs, "spec_compact_args": st.CompactArgs,
          "spec_host_copy": st.HostCopy}
    for (t, f), v in got.items():
        cls = py[t]
        if f == "size":
            assert ctypes.sizeof(cls) == v, t
        else:
            assert getattr(cls, f).offset == v, (t, f)


def test_status_strings(L):
    for code in range(9):
        assert st.status_string(code) and st.status_string(code) != "unknown status"
    assert st.status_string(99) == "unknown status"


def test_host_argument_errors_return_before_launch(L):
    assert L.spec_tree_attention(None, None, 0, None, None) == 1
    assert L.spec_verify_accept(None, None, 0, None, None) == 1
    assert L.spec_compact_kv(None, None, None) == 1
    a = st.AttnArgs(dtype=1, batch=1, n_max=4, num_q_heads=4, num_kv_heads=1, head_dim=96, kv_capacity=16)
    assert L.spec_tree_attention(ctypes.byref(a), None, 0, None, None) == 2          # head_dim 96
    assert L.spec_tree_attention_workspace(ctypes.byref(a)) == 0
    a.head_dim = 64
    assert L.spec_tree_attention(ctypes.byref(a), None, 0, None, None) == 1          # null tensors
    a.n_max = 256
    assert L.spec_tree_attention(ctypes.byref(a), None, 0, None, None) == 2          # > 255 nodes
    fake = ctypes.c_void_p(1 << 20)
    a = st.AttnArgs(dtype=1, batch=1, n_max=4, num_q_heads=12, num_kv_heads=4, head_dim=64, kv_capacity=16,
                    q=fake, k_cache=fake, v_cache=fake, prefix_len=fake, n_nodes=fake, parent=fake, out=fake)
    a.schedule = 2
    assert L.spec_tree_attention(ctypes.byref(a), None, 0, None, None) == 1          # unknown schedule
    a.schedule = 1
    assert L.spec_tree_attention(ctypes.byref(a), None, 0, None, None) == 2          # stream-K: 128 % G != 0
    a.num_q_heads, a.dtype = 8, 0
    assert L.spec_tree_attention(ctypes.byref(a), None, 0, None, None) == 2          # stream-K: bf16 only
    v = st.VerifyArgs(dtype=1, batch=1, n_max=4, hidden=100, vocab=50, rule=0, path_cap=4)
    assert L.spec_verify_accept(ctypes.byref(v), None, 0, None, None) == 2           # bf16 hidden % 64
    v.hidden, v.rule, v.temperature = 128, 2, 0.0
    assert L.spec_verify_accept(ctypes.byref(v), None, 0, None, None) == 1           # tau must be > 0
    # compact draft rows: a row index needs at least one row; the reserved word must be 0
    fake2 = ctypes.c_void_p(1 << 20)
    r = st.VerifyArgs(dtype=1, batch=1, n_max=4, hidden=128, vocab=50, rule=2, temperature=1.0, draft_vocab=50,
                      path_cap=4, hidden_states=fake2, lm_head_weight=fake2, tokens=fake2, parent=fake2,
                      n_nodes=fake2, draft_probs=fake2, accept_len=fake2, path=fake2, bonus_token=fake2)
    assert L.spec_verify_accept_workspace(ctypes.byref(r)) > 0
    r.draft_rows = fake2
    assert L.spec_verify_accept_workspace(ctypes.byref(r)) == 0                       # n_draft_rows 0
    r.n_draft_rows = 7
    assert L.spec_verify_accept_workspace(ctypes.byref(r)) > 0
    r.reserved1 = 1
    assert L.spec_verify_accept_workspace(ctypes.byref(r)) == 0                       # reserved word set
    c = st.CompactArgs(dtype=0, batch=1, num_kv_heads=1, head_dim=64, kv_capacity=8, path_cap=0)
    assert L.spec_compact_kv(ctypes.byref(c), None, None) == 1                        # path_cap 0
    handle = ctypes.c_void_p(123)
    assert L.spec_round_create(None, None, 0, None, None, 0, None, None, ctypes.byref(handle)) == 1
    assert handle.value is None                                                       # no call given
    assert L.spec_round_create(None, None, 0, None, None, 0, None, None, None) == 1   # out == NULL
    assert L.spec_round_launch(None, None) == 1
    L.spec_round_destroy(None)
    # the host-buffer launch checks its copy descriptors (and the round) before enqueuing anything
    fn = L.spec_round_launch_host
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    fake = ctypes.c_void_p(1 << 20)
    assert fn(None, None, 0, None, 0, None) == 1                      # no round
    assert fn(fake, None, -1, None, 0, None) == 1                     # negative count
    assert fn(fake, None, 1, None, 0, None) == 1                      # NULL array, positive count
    bad = (st.HostCopy * 1)(st.HostCopy(host=None, device=fake, row_bytes=16, rows=1))
    assert fn(fake, ctypes.cast(bad, ctypes.c_void_p), 1, None, 0, None) == 1   # NULL host pointer
    pitch = (st.HostCopy * 1)(st.HostCopy(host=fake, device=fake, row_bytes=64, rows=4, host_pitch=32,
                                          device_pitch=64))
    assert fn(fake, None, 0, ctypes.cast(pitch, ctypes.c_void_p), 1, None) == 1  # pitch below a row


def test_workspace_queries_are_host_only(L):
    fake = ctypes.c_void_p(1 << 20)  # aligned non-null pointers, never dereferenced by the query
    a = st.AttnArgs(dtype=1, batch=2, n_max=63, num_q_heads=32, num_kv_heads=8, head_dim=128, kv_capacity=4096,
                    q=fake, k_cache=fake, v_cache=fake, prefix_len=fake, n_nodes=fake, parent=fake, out=fake)
    need = L.spec_tree_attention_workspace(ctypes.byref(a))
    assert need > 2 * 63 * 32 * 128 * 4
    # the partials leave through bulk copies, so a workspace off a 16-byte boundary is refused
    # before anything is launched (as are a missing one and a short one)
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert L.spec_tree_attention(ctypes.byref(a), odd, need, None, None) == 1
    assert L.spec_tree_attention(ctypes.byref(a), None, need, None, None) == 1
    assert L.spec_tree_attention(ctypes.byref(a), fake, need - 1, None, None) == 3
    v = st.VerifyArgs(dtype=1, batch=1, n_max=63, hidden=4096, vocab=128256, rule=2, temperature=1.0,
                      draft_vocab=128256, path_cap=64, hidden_states=fake, lm_head_weight=fake, tokens=fake,
                      parent=fake, n_nodes=fake, draft_probs=fake, accept_len=fake, path=fake, bonus_token=fake)
    need = L.spec_verify_accept_workspace(ctypes.byref(v))
    assert need >= 63 * 128256 * 4  # rejection keeps the fp32 logits
    # records and logits are stored as 16-byte vectors: a workspace off a 16-byte boundary, a
    # missing one and a short one are refused before anything is launched
    assert L.spec_verify_accept(ctypes.byref(v), odd, need, None, None) == 1
    assert L.spec_verify_accept(ctypes.byref(v), None, need, None, None) == 1
    assert L.spec_verify_accept(ctypes.byref(v), fake, need - 1, None, None) == 3
    # the folded compaction must name the verification's own path and length
    c = st.CompactArgs(dtype=1, batch=1, num_kv_heads=8, head_dim=128, kv_capacity=4096, path_cap=64,
                       k_cache=fake, v_cache=fake, prefix_len=fake, path=fake, accept_len=fake)
    other = ctypes.c_void_p((1 << 20) + 4096)
    c.path = other
    assert L.spec_verify_accept_compact(ctypes.byref(v), fake, need, ctypes.byref(c), None, None) == 1
    c.path, c.path_cap = fake, 63
    assert L.spec_verify_accept_compact(ctypes.byref(v), fake, need, ctypes.byref(c), None, None) == 1
    c.path_cap, c.head_dim = 64, 96
    assert L.spec_verify_accept_compact(ctypes.byref(v), fake, need, ctypes.byref(c), None, None) == 2
    v.rule = 0
    assert L.spec_verify_accept_workspace(ctypes.byref(v)) < need


def test_attention_split_plan_from_the_workspace_query(L):
    """The key-split count shows in the workspace (bf16 partials per split).  A batch of 32
    4096-token prefixes (256 CTAs of 65 key tiles fill more than one round of SMs) runs one split
    per KV head; a single 2048-token request is cut into 4-tile splits so that its 16 row groups
    reach every SM.  Batches of 8 or 16 such prefixes stay unsplit too: one round that leaves
    SMs idle beats two filled rounds plus the merge by more than 15 %.  Eight 8192-token
    capacities with 127-node trees take three splits: the filling grid is preferred, since
    requests shorter than the capacity make it cheaper than estimated."""
    fake = ctypes.c_void_p(1 << 20)

    def splits(B, L_cap, N=63):
        a = st.AttnArgs(dtype=1, batch=B, n_max=N, num_q_heads=32, num_kv_heads=8, head_dim=128,
                        kv_capacity=L_cap, q=fake, k_cache=fake, v_cache=fake, prefix_len=fake,
                        n_nodes=fake, parent=fake, out=fake)
        rows = B * N * 32
        ws = L.spec_tree_attention_workspace(ctypes.byref(a))
        return ws // (rows * (128 * 2 + 8))  # bf16 partial rows + (max, sum); everything else is far smaller

    assert splits(32, 4096 + 63) == 1
    assert splits(1, 2048 + 63) == 9
    assert splits(16, 4096 + 63) == 1
    assert splits(8, 4096 + 63) == 1
    assert splits(8, 8192 + 127, N=127) == 3


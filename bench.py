#!/usr/bin/env python3
"""Benchmark of one tree-verification step on GB300.

A step is the whole verification hot path over one batch: tree attention (one layer), LM head +
acceptance + longest accepted path, and KV compaction -- the three C-ABI calls
spec_tree_attention, spec_verify_accept and spec_compact_kv, launched as one captured round.
Metric: verified tree-tokens/s (tree nodes verified per second).

The headline workload is the largest one that fits one GPU: a 70B-shaped layer (64 query heads,
8 KV heads, head_dim 128, hidden 8192, vocabulary 128256, bf16), batch 4 with prefixes of 32768,
65536, 98304 and 131072 tokens, 255-node trees (depth <= 8, branching 1-4), greedy acceptance.
The EAGLE-3-shaped batch-32 workload (8B layer, prefix 4096, dynamic 63-node trees, mapped
draft vocabulary, rejection sampling) is measured in the same run and reported as a second full
line under "second_workload".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Under torchrun each rank runs an independent replica on its own GPU (the path needs no exchange);
the JSON line reports the whole-job rate from the slowest rank.  ``--impl reference`` times the
fp64 CPU oracle on the host cores instead, one bounded sample per step.
"""

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tree-tokens/s per GB300 and % of roofline (HBM / bf16 TC) vs CPU oracle"
UNIT = "tree-tokens/s"
WORKLOAD = 5         # gen.configs: llama70b-b4-l32kto128k-bfs255-greedy (largest single-GPU workload)
SECOND_WORKLOAD = 4  # gen.configs: eagle3-llama8b-b32-l4096-dynamic63-rejection
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
CSRC = os.path.join(ROOT, "tree_speculative_decoding_split_gb300", "csrc")
# kernel -> the source files its counters depend on (a committed traffic figure is used only
# while these are unchanged)
KERNEL_SOURCES = {
    "attn_tc_kernel": ["attention_tc.cu", "tc_ptx.cuh", "common.cuh"],
    "attn_sk_kernel": ["attention_sk.cu", "tc_ptx.cuh", "common.cuh"],
    "attn_merge_bf16_kernel": ["attention.cu", "common.cuh"],
    "lmhead_tc_kernel": ["lmhead.cu", "tc_ptx.cuh", "common.cuh"],
    "lmhead_tc_rows_kernel": ["lmhead.cu", "tc_ptx.cuh", "common.cuh"],
    "lmhead_tc_pair_kernel": ["lmhead.cu", "tc_ptx.cuh", "common.cuh"],
    "compact_kv_kernel": ["compact.cu", "compact.cuh", "common.cuh"],
}


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--mode", default="graph", choices=["graph", "direct"],
                   help="graph: each step is one spec_round_launch of the captured round (default); "
                        "direct: the three C-ABI calls per step")
    p.add_argument("--workload", type=int, default=WORKLOAD,
                   help="gen.configs workload id (the headline metric is quoted on the default)")
    p.add_argument("--second-workload", type=int, default=SECOND_WORKLOAD,
                   help="workload reported as a second full line (0: none)")
    p.add_argument("--no-next", action="store_true", help="leave out the next_rows measurements")
    p.add_argument("--profile", action="store_true",
                   help="profiling harness: run the workload's three calls --warmup + --steps times "
                        "without timing anything and print nothing (for ncu)")
    p.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of oracle work for cpu_baseline")
    p.add_argument("--ref-budget", type=float, default=150.0,
                   help="--impl reference: stop taking steps after this many seconds of oracle work")
    return p.parse_args()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def _threads_used():
    try:
        from threadpoolctl import threadpool_info
        n = sum(i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas")
        if n:
            return n
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---- workload accounting ------------------------------------------------------------------------

def _work(case):
    """Algorithmic bytes / flops of the step and of its kernels (no tile re-reads counted)."""
    import numpy as np
    from gen import trees as T
    nodes = int(case.n_nodes.sum())
    rows = case.B * case.N
    kv_bytes = sum(2 * case.Hkv * (int(case.prefix_len[b]) + int(case.n_nodes[b])) * case.d * 2
                   for b in range(case.B))
    qo_bytes = 2 * nodes * case.Hq * case.d * 2 + nodes * case.Hq * 4
    w_bytes = case.V * case.Hd * 2
    h_bytes = rows * case.Hd * 2
    logits_bytes = rows * case.V * 4 if case.rule == "rejection" else 0
    lm_flops = 2.0 * rows * case.Hd * case.V
    # prefix keys for every node, plus each node's ancestors-or-self among the tree keys
    tree_keys = sum(int((T.depths(case.parent[b, : case.n_nodes[b]]) + 1).sum()) for b in range(case.B))
    attn_flops = 4.0 * case.d * case.Hq * (sum(int(case.n_nodes[b]) * int(case.prefix_len[b])
                                               for b in range(case.B)) + tree_keys)
    return dict(nodes=nodes, kv_bytes=kv_bytes, qo_bytes=qo_bytes, w_bytes=w_bytes, h_bytes=h_bytes,
                logits_bytes=logits_bytes, lm_flops=lm_flops, attn_flops=attn_flops,
                lm_kernel_bytes=w_bytes + h_bytes + logits_bytes, attn_kernel_bytes=kv_bytes + qo_bytes,
                tree_keys=int(np.int64(tree_keys)))


def _sources_sha(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, []):
        h.update(open(os.path.join(CSRC, f), "rb").read())
    return h.hexdigest()


def traffic_entry(kernel, workload):
    """DRAM read + write bytes per launch of ``kernel`` on ``workload`` from the committed ncu
    summary profiles/traffic.json, if the kernel's sources are unchanged since the counters were
    taken (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    for e in json.load(open(path)).get("entries", []):
        if e.get("kernel") == kernel and e.get("workload") == workload:
            if e.get("sources_sha256") == _sources_sha(kernel):
                return e
    return None


def _roofline(kernel, flops, nbytes, ms, hbm, tc, peak_kind, workload):
    """Roofline object of one kernel: the binding roof among HBM bytes and bf16 tensor FLOPs."""
    t_bytes = nbytes / (hbm * 1e9)
    t_flops = flops / (tc * 1e12)
    e = traffic_entry(kernel, workload)
    traffic = e["traffic_bytes_per_launch"] if e else None
    if t_flops > t_bytes:
        ach = flops / (ms * 1e-3) / 1e12
        return {"kernel": kernel, "bound": "tensor", "achieved": ach, "peak": tc, "unit": "TFLOP/s", "frac": ach / tc,
                "traffic": traffic, "algorithmic_flops": flops, "algorithmic_bytes": nbytes, "ms": ms,
                "peak_source": f"{peak_kind} bf16_tflops (burst)"}
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
            "traffic": traffic, "algorithmic_bytes": nbytes, "algorithmic_flops": flops, "ms": ms,
            "peak_source": f"{peak_kind} hbm_gbs"}


# ---- clocks -------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---- replicas ------------------------------------------------------------------------------------

def aggregate_ranks(times_ms, dist=None, device=None):
    """Slowest rank's times: every rank runs an independent replica of the workload, so the job's
    rate is (ranks x work per rank) / the maximum time.  Without a process group, identity."""
    if dist is None:
        return list(times_ms)
    import torch
    buf = torch.tensor(list(times_ms), dtype=torch.float64, device=device)
    dist.all_reduce(buf, op=dist.ReduceOp.MAX)
    return [float(x) for x in buf]


def job_rate(world, units_per_rank, ms):
    """Whole-job throughput in units/s from the slowest rank's per-step time."""
    return world * units_per_rank / (ms * 1e-3)


# ---- native arm ---------------------------------------------------------------------------------

def _device_tensors(case, dev):
    import numpy as np
    import torch

    def t(a, bf=False):
        if bf:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    bf = case.dtype == "bf16"
    return dict(q=t(case.q, bf), k=t(case.k_cache, bf), v=t(case.v_cache, bf), hidden=t(case.hidden, bf),
                W=t(case.W, bf), prefix_len=t(case.prefix_len.astype(np.int32)), n_nodes=t(case.n_nodes.astype(np.int32)),
                parent=t(case.parent.astype(np.int32)), tokens=t(case.tokens.astype(np.int32)),
                draft=None if case.draft_probs is None else t(case.draft_probs),
                map=None if case.draft_to_target is None else t(case.draft_to_target.astype(np.int32)))


def _attention_plan(L, aa, case, sms):
    """(stream_k, key splits) of the attention plan, read back from the workspace query: the
    stream-K kernel's workspace holds two 256-row partial slots per SM, the split kernel's partials
    of d bf16 values and two floats per row and split."""
    ws = int(L.spec_tree_attention_workspace(ctypes.byref(aa)))
    sk = sms * 2 * 256 * (case.d * 4 + 8)
    if case.dtype == "bf16" and sk <= ws < sk + (8 << 20):
        return True, 1
    rows = case.B * case.N * case.Hq
    return False, max(1, ws // (rows * (case.d * 2 + 8)))


def _launches_per_step(case, n_split, stream_k, fused):
    if case.dtype != "bf16":
        attn = 2                                                       # tree prep + fp32 rows
    else:
        attn = 2 if (stream_k or n_split > 1) else 1                   # counters memset + stream-K | split-KV [+ merge]
    # LM head, then the row finalisation -- or for rejection the walk, which merges its rows'
    # statistics itself (no per-row outputs are requested here) [+ fp32 statistics]
    verify = 2 if case.dtype == "bf16" else 3
    if case.rule == "rejection" and case.draft_to_target is not None:
        verify += 1                                                    # draft-map inversion
    return attn + verify + (0 if fused else 1)                         # compaction folded into acceptance


class _Flush:
    """Writes, then reads back, a buffer twice the size of L2, so that the next step starts from a
    cold L2 of clean lines (the flush's write-backs are not charged to the step)."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.sink = torch.empty(1, dtype=torch.int64, device=dev)

    def __call__(self):
        import torch
        self.buf.zero_()
        torch.sum(self.buf.view(torch.int64), dim=0, keepdim=True, out=self.sink)


def measure_workload(a, cfg, rank, world, dist, seed, with_cpu):
    """Times the workload's verification step and returns its JSON line (rank 0) or None."""
    import numpy as np
    import torch
    import tree_speculative_decoding_split_gb300 as st
    from gen import make_config_case

    L = st.lib()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    case = make_config_case(cfg, seed=seed)
    t = _device_tensors(case, dev)
    t["draft_rows"] = None
    if case.draft_probs is not None:
        # a drafter has distributions only for the nodes it expanded: pass those rows compactly
        from gen import compact_draft
        rows, index = compact_draft(case.draft_probs, case.parent, case.n_nodes)
        t["draft"] = torch.from_numpy(rows).to(dev)
        t["draft_rows"] = torch.from_numpy(index).to(dev)
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                              case.eps, case.delta, case.seed, t["draft"], t["map"], path_cap=case.N,
                              draft_rows=t["draft_rows"])
    ca, src_slot, new_len = st.compact_args(t["k"], t["v"], t["prefix_len"], outs["path"], outs["accept_len"])
    need_a = L.spec_tree_attention_workspace(ctypes.byref(aa))
    need_v = L.spec_verify_accept_workspace(ctypes.byref(va))
    ws_a = torch.empty(need_a, dtype=torch.uint8, device=dev)
    ws_v = torch.empty(need_v, dtype=torch.uint8, device=dev)
    pa, pv, pst = ctypes.c_void_p(ws_a.data_ptr()), ctypes.c_void_p(ws_v.data_ptr()), ctypes.c_void_p(status.data_ptr())
    l2_flush = _Flush(dev)
    stream_k, n_split = _attention_plan(L, aa, case, torch.cuda.get_device_properties(dev).multi_processor_count)

    def step():
        c1 = L.spec_tree_attention(ctypes.byref(aa), pa, need_a, pst, sp)
        c2 = L.spec_verify_accept(ctypes.byref(va), pv, need_v, pst, sp)
        c3 = L.spec_compact_kv(ctypes.byref(ca), pst, sp)
        if c1 or c2 or c3:
            raise RuntimeError(f"C ABI returned {c1} {c2} {c3}")

    def check_status():
        if int(status.item()) != 0:
            raise RuntimeError("device status " + st.status_string(int(status.item())))

    if a.profile:
        for _ in range(max(1, a.warmup) + max(1, a.steps)):
            step()
        torch.cuda.synchronize()
        check_status()
        return None

    def events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)  # materialise the underlying cudaEvent_t
        return evs

    W = max(3, a.warmup)
    for _ in range(W):
        l2_flush()
        step()
    torch.cuda.synchronize()
    check_status()

    K = a.steps

    def timed_direct(n):
        """n steps of the three direct calls; per-step and per-kernel device times (ms)."""
        ev_s, ev_e = events(n), events(n)
        ev_ab, ev_ae, ev_lb, ev_le = events(n), events(n), events(n), events(n)
        torch.cuda.synchronize()
        for i in range(n):
            l2_flush()
            aa.timing_begin, aa.timing_end = ev_ab[i].cuda_event, ev_ae[i].cuda_event
            va.timing_begin, va.timing_end = ev_lb[i].cuda_event, ev_le[i].cuda_event
            ev_s[i].record(stream)
            step()
            ev_e[i].record(stream)
        torch.cuda.synchronize()
        aa.timing_begin = aa.timing_end = va.timing_begin = va.timing_end = None
        return ([ev_s[i].elapsed_time(ev_e[i]) for i in range(n)], [ev_ab[i].elapsed_time(ev_ae[i]) for i in range(n)],
                [ev_lb[i].elapsed_time(ev_le[i]) for i in range(n)])

    def timed_graph(rnd, n):
        """n steps, each one launch of the captured round."""
        ev_s, ev_e = events(n), events(n)
        torch.cuda.synchronize()
        for i in range(n):
            l2_flush()
            ev_s[i].record(stream)
            rnd.launch(stream)
            ev_e[i].record(stream)
        torch.cuda.synchronize()
        return [ev_s[i].elapsed_time(ev_e[i]) for i in range(n)]

    rnd = st.Round(aa, va, ca, dev_status=status)
    for _ in range(W):
        l2_flush()
        rnd.launch(stream)
    torch.cuda.synchronize()

    # ---- end to end through spec_round_launch_host: pinned host inputs -> device, the round,
    # results -> pinned host, one C call per step ----
    n_tree = int(case.n_nodes.max())
    Lp = [int(x) for x in case.prefix_len]
    step_inputs = ["q", "hidden", "tokens", "parent", "n_nodes", "prefix_len"]
    if t["draft"] is not None:  # rejection sampling: the expanded nodes' draft distributions and
        step_inputs += ["draft", "draft_rows"]  # their row index arrive with every step
    host = {k: t[k].cpu().pin_memory() for k in step_inputs}
    ins = [st.host_copy(host[k], t[k]) for k in step_inputs]
    for b in range(case.B):  # the tree's new K/V rows, one strided copy per request and cache
        for name in ("k", "v"):
            rows = t[name][b, :, Lp[b]: Lp[b] + n_tree].contiguous().cpu().pin_memory()
            host[f"{name}_tree_{b}"] = rows
            ins.append(st.host_copy(rows, t[name][b, :, Lp[b]: Lp[b] + n_tree], rows=case.Hkv))
    out_names = ("accept_len", "path", "bonus_token", "margin_count", "bonus_margin")
    res_host = {k: torch.empty(outs[k].shape, dtype=outs[k].dtype).pin_memory() for k in out_names}
    res_host["new_len"] = torch.empty(new_len.shape, dtype=new_len.dtype).pin_memory()
    outs_c = [st.host_copy(res_host[k], outs[k]) for k in out_names] + [st.host_copy(res_host["new_len"], new_len)]
    h2d = sum(c.row_bytes * c.rows for c in ins)
    d2h = sum(c.row_bytes * c.rows for c in outs_c)
    for _ in range(3):
        l2_flush()
        rnd.launch_host(ins, outs_c, stream)
    torch.cuda.synchronize()

    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    # Per-kernel device times (the roofline's inputs) come from the direct calls, whose
    # library-recorded events bracket the attention and LM-head kernels; events recorded inside
    # a CUDA graph are not timable.  The step time comes from the round's launches.
    direct_ms, attn_ms, lm_ms = timed_direct(K)
    graph_ms = timed_graph(rnd, K)
    step_ms = graph_ms if a.mode == "graph" else direct_ms
    KE = max(10, min(K, 500))
    es, ee = events(KE), events(KE)
    torch.cuda.synchronize()
    for i in range(KE):
        l2_flush()
        es[i].record(stream)
        rnd.launch_host(ins, outs_c, stream)
        ee[i].record(stream)
    torch.cuda.synchronize()
    e2e_list = [es[i].elapsed_time(ee[i]) for i in range(KE)]
    clk = clocks.stop()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    check_status()
    ms = statistics.median(step_ms)
    other_ms = statistics.median(direct_ms if a.mode == "graph" else graph_ms)
    e2e_ms = statistics.median(e2e_list)
    # margin cases (decisions within 1e-4 of their threshold) of the last step, counted on the GPU
    margins = int(res_host["margin_count"].sum())
    bonus_margins = int(res_host["bonus_margin"].sum())
    alen = [int(x) for x in res_host["accept_len"]]

    ms, e2e_ms, other_ms = aggregate_ranks([ms, e2e_ms, other_ms], dist, dev)
    if rank != 0:
        rnd.close()
        return None

    w = _work(case)
    hbm, tc, tc_sus, peak_kind = _peaks()
    lm_med = statistics.median(lm_ms)
    attn_med = statistics.median(attn_ms)
    # the LM-head kernel the library picks for this many tree rows (bf16): vocabulary on M up to
    # 64 rows, rows on M up to 128, CTA pairs above
    R = case.B * case.N
    lm_kernel = "lmhead_tc_pair_kernel" if R > 128 else ("lmhead_tc_rows_kernel" if R > 64 else "lmhead_tc_kernel")
    rf_attn = _roofline("attn_sk_kernel" if stream_k else "attn_tc_kernel", w["attn_flops"], w["attn_kernel_bytes"], attn_med, hbm, tc, peak_kind,
                        case.name)
    rf_lm = _roofline(lm_kernel, w["lm_flops"], w["lm_kernel_bytes"], lm_med, hbm, tc, peak_kind, case.name)
    dominant = rf_attn if attn_med >= lm_med else rf_lm
    # the step's combined roofline: max(KV + weight bytes at HBM bandwidth, LM-head FLOPs at the
    # bf16 tensor peak); the full one adds every byte and the attention FLOPs
    step_bytes = w["kv_bytes"] + w["qo_bytes"] + w["w_bytes"] + w["h_bytes"] + w["logits_bytes"]
    t_comb = max((w["kv_bytes"] + w["w_bytes"]) / (hbm * 1e9), w["lm_flops"] / (tc * 1e12))
    t_full = max(step_bytes / (hbm * 1e9), (w["lm_flops"] + w["attn_flops"]) / (tc * 1e12))
    line = {
        "metric": METRIC, "value": job_rate(world, w["nodes"], ms), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": case.name, "batch": case.B, "prefix_len": [int(x) for x in case.prefix_len][:8],
                   "tree_nodes": [int(x) for x in case.n_nodes][:8], "q_heads": case.Hq, "kv_heads": case.Hkv,
                   "head_dim": case.d, "hidden": case.Hd, "vocab": case.V, "rule": case.rule, "temperature": case.tau,
                   "eps": case.eps, "delta": case.delta, "parallelism": f"replicas x{world}",
                   "draft_distributions": (None if t["draft"] is None else
                                           f"{t['draft'].shape[0]} rows (the expanded nodes') of "
                                           f"{t['draft'].shape[1]} fp32, indexed by draft_rows [B][N]"),
                   "l2": "flushed before every step (256 MB write, then read)",
                   "launch": ("one CUDA-graph launch of the captured round per step (spec_round_launch; "
                              "tree attention and verification as parallel branches, the longer one first, "
                              "compaction after both)"
                              if a.mode == "graph" else "three C-ABI calls per step"),
                   "statistic": "median over the timed steps"},
        "e2e": {"value": job_rate(world, w["nodes"], e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "call": ("spec_round_launch_host: pinned host inputs copied in group after group (the longer "
                         "branch's first -- the verification's go on the round's own stream --, then the other "
                         "branch's, then the draft distributions beside the LM head), the round, results copied "
                         "out; every step's copies are inside the timed region")},
        # the graph runs attention and verification as parallel branches, so its compaction is a
        # launch of its own, as in the direct calls
        "gpu_launches": K * _launches_per_step(case, n_split, stream_k, False),
        "roofline": dominant,
        "roofline_kernels": {"tree_attention": rf_attn, "lm_head": rf_lm},
        "kernels": {"tree_attention_ms": attn_med, "lmhead_ms": lm_med,
                    "attention_kernel": "persistent stream-K" if stream_k else f"split-KV, {n_split} key splits",
                    "attention_roofline_frac": rf_attn["frac"], "lmhead_roofline_frac": rf_lm["frac"]},
        "roofline_step": {"combined_s": t_comb, "frac_combined": t_comb / (ms * 1e-3),
                          "full_s": t_full, "frac_full": t_full / (ms * 1e-3),
                          "peaks": f"{peak_kind}: hbm {hbm} GB/s, bf16 {tc} TFLOP/s (burst)",
                          "frac_combined_sustained_peak": max((w["kv_bytes"] + w["w_bytes"]) / (hbm * 1e9),
                                                              w["lm_flops"] / (tc_sus * 1e12)) / (ms * 1e-3)},
        "margins": {"decisions_within_1e-4": margins, "bonus_within_1e-4": bonus_margins,
                    "requests": case.B, "accept_len": alen[:8]},
        "clocks": clk,
        ("direct_calls" if a.mode == "graph" else "graph_round"): {
            "ms_per_step": other_ms, "value": job_rate(world, w["nodes"], other_ms),
            "note": "same workload, " + ("the three C-ABI calls per step" if a.mode == "graph" else "one graph launch")},
    }
    if world == 1 and with_cpu and not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, a.cpu_budget)
    if world == 1 and not a.no_next and cfg == a.workload:
        line["next_rows"] = {
            "llama8b_b1_round": _bench_b1_round(a, st, L, dev, stream, l2_flush, events, K),
            "medusa_expand": _bench_medusa(st, L, dev, stream, l2_flush, events, K, hbm),
            "eagle_dynamic_tree": _bench_eagle(st, L, dev, stream, l2_flush, events, K),
            "paged_attention": {f"block_{bs}": _bench_paged(st, L, dev, stream, l2_flush, events, K, t, w, hbm, tc, bs,
                                                            attn_med) for bs in (16, 64)},
        }
    rnd.close()
    del t, ws_a, ws_v, l2_flush
    torch.cuda.empty_cache()
    return line


def _timed_calls(l2_flush, events, stream, call, n):
    import torch
    for _ in range(3):
        l2_flush()
        call()
    es, ee = events(n), events(n)
    torch.cuda.synchronize()
    for i in range(n):
        l2_flush()
        es[i].record(stream)
        call()
        ee[i].record(stream)
    torch.cuda.synchronize()
    return statistics.median(es[i].elapsed_time(ee[i]) for i in range(n))


def _bench_b1_round(a, st, L, dev, stream, l2_flush, events, K):
    """The batch-1 Llama-8B-shaped round (2048-token prefix, static 63-node tree, typical
    acceptance), where launches are a visible share of the step: one graph launch (attention and
    verification as parallel branches, compaction after both), the three C-ABI calls, and two
    calls with the compaction folded into acceptance."""
    import torch
    from gen import make_config_case
    case = make_config_case(2, seed=a.seed)
    t = _device_tensors(case, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                              case.eps, case.delta, case.seed, None, None, path_cap=case.N)
    ca, src_slot, new_len = st.compact_args(t["k"], t["v"], t["prefix_len"], outs["path"], outs["accept_len"])
    need_a = L.spec_tree_attention_workspace(ctypes.byref(aa))
    need_v = L.spec_verify_accept_workspace(ctypes.byref(va))
    ws_a = torch.empty(need_a, dtype=torch.uint8, device=dev)
    ws_v = torch.empty(need_v, dtype=torch.uint8, device=dev)
    pa, pv, pst = ctypes.c_void_p(ws_a.data_ptr()), ctypes.c_void_p(ws_v.data_ptr()), ctypes.c_void_p(status.data_ptr())
    sp = ctypes.c_void_p(stream.cuda_stream)

    def three():
        if (L.spec_tree_attention(ctypes.byref(aa), pa, need_a, pst, sp) or
                L.spec_verify_accept(ctypes.byref(va), pv, need_v, pst, sp) or L.spec_compact_kv(ctypes.byref(ca), pst, sp)):
            raise RuntimeError("C ABI call failed")

    def two():
        if (L.spec_tree_attention(ctypes.byref(aa), pa, need_a, pst, sp) or
                L.spec_verify_accept_compact(ctypes.byref(va), pv, need_v, ctypes.byref(ca), pst, sp)):
            raise RuntimeError("C ABI call failed")

    rnd = st.Round(aa, va, ca, dev_status=status)
    n = min(K, 200)
    res = {"graph_ms": _timed_calls(l2_flush, events, stream, lambda: rnd.launch(stream), n),
           "three_calls_ms": _timed_calls(l2_flush, events, stream, three, n),
           "two_calls_folded_compaction_ms": _timed_calls(l2_flush, events, stream, two, n), "steps": n,
           "tree_tokens": int(case.n_nodes.sum())}
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status " + st.status_string(int(status.item())))
    res["graph_tree_tokens_per_s"] = res["tree_tokens"] / (res["graph_ms"] * 1e-3)
    rnd.close()
    return res


def _bench_medusa(st, L, dev, stream, l2_flush, events, K, hbm):
    """Static Medusa expansion at the 8B-shaped batch-1 shapes: 5 heads of bf16 logits over the
    128256-token vocabulary, the 63-node topology from per-head top-(3, 3, 2, 2, 1)."""
    import numpy as np
    import torch
    from gen import bf16 as BF
    B, V = 1, 128256
    topk_heads = (3, 3, 2, 2, 1)
    parent, rank = st.medusa_topology(topk_heads, 63)
    rng = np.random.default_rng(5)
    x = BF.f32_to_bf16_bits(rng.standard_normal((B, len(topk_heads), V)).astype(np.float32))
    logits = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
    tp, tr = torch.from_numpy(parent).to(dev), torch.from_numpy(rank).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ma, outs = st.medusa_args(logits, tp, tr, max(topk_heads))
    need = L.spec_medusa_expand_workspace(ctypes.byref(ma))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    pw, pst, sp = ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream.cuda_stream)

    def call():
        if L.spec_medusa_expand(ctypes.byref(ma), pw, need, pst, sp):
            raise RuntimeError("spec_medusa_expand failed")

    n = min(K, 500)
    ms = _timed_calls(l2_flush, events, stream, call, n)
    if int(status.item()) != 0:
        raise RuntimeError("device status " + st.status_string(int(status.item())))
    nbytes = logits.numel() * 2
    return {"ms": ms, "steps": n, "bound": "hbm", "bytes": nbytes, "achieved_gbs": nbytes / (ms * 1e-3) / 1e9,
            "frac": nbytes / (ms * 1e-3) / 1e9 / hbm, "launches_per_call": 2,
            "shape": {"batch": B, "heads": len(topk_heads), "vocab": V, "topk": list(topk_heads),
                      "nodes": int(len(parent)), "dtype": "bf16"}}


def _bench_eagle(st, L, dev, stream, l2_flush, events, K):
    """Dynamic draft tree at the EAGLE-3 batch of 32: one expansion layer (frontier 8, top-8 over a
    32000-entry draft vocabulary) and the selection of a 63-node tree from 8 stacked layers."""
    import numpy as np
    import torch
    B, F, k, Vd, D, N = 32, 8, 8, 32000, 8, 63
    rng = np.random.default_rng(9)
    z = rng.standard_normal((B, F, Vd)).astype(np.float32)
    lp = torch.from_numpy(z - np.log(np.exp(z.astype(np.float64)).sum(-1, keepdims=True)).astype(np.float32)).to(dev)
    fs = torch.from_numpy((-rng.exponential(2.0, (B, F))).astype(np.float32)).to(dev)
    C = F * k
    # stacked candidates as the expansion produces them: a child scores its parent's score plus
    # a log-probability (<= 0)
    Pn = rng.integers(0, C, (B, D, C)).astype(np.int32)
    Sn = np.zeros((B, D, C), dtype=np.float32)
    Sn[:, 0] = -rng.exponential(1.0, (B, C))
    for layer in range(1, D):
        Sn[:, layer] = np.take_along_axis(Sn[:, layer - 1], Pn[:, layer], axis=1) - rng.exponential(1.0, (B, C))
    S = torch.from_numpy(Sn).to(dev)
    Tk = torch.from_numpy(rng.integers(0, Vd, (B, D, C)).astype(np.int32)).to(dev)
    P = torch.from_numpy(Pn).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # argument structs and workspace built once; the timed calls are the C ABI's
    ea, e_out = st.eagle_expand_args(lp, fs, k, F)  # the structs point into e_out / t_out: keep both
    need = L.spec_eagle_expand_workspace(ctypes.byref(ea))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    ta, t_out = st.eagle_tree_args(S, Tk, P, N)
    pw, pst, sp = ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream.cuda_stream)

    def expand():
        if L.spec_eagle_expand(ctypes.byref(ea), pw, need, pst, sp):
            raise RuntimeError("spec_eagle_expand failed")

    def tree():
        if L.spec_eagle_tree(ctypes.byref(ta), pst, sp):
            raise RuntimeError("spec_eagle_tree failed")

    n = min(K, 300)
    layer_ms = _timed_calls(l2_flush, events, stream, expand, n)
    tree_ms = _timed_calls(l2_flush, events, stream, tree, n)
    torch.cuda.synchronize()
    del e_out, t_out
    if int(status.item()) != 0:
        raise RuntimeError("device status " + st.status_string(int(status.item())))
    return {"expand_layer_ms": layer_ms, "select_tree_ms": tree_ms, "steps": n,
            "shape": {"batch": B, "frontier": F, "topk": k, "draft_vocab": Vd, "layers": D, "nodes": N},
            "note": "C ABI calls with argument structs built once"}


def _bench_paged(st, L, dev, stream, l2_flush, events, K, t, w, hbm, tc, bs, contiguous_ms):
    """Tree attention of the workload with its KV cache scattered over a shuffled block pool."""
    import torch
    B, Hkv, L_cap, d = t["k"].shape
    mb = (L_cap + bs - 1) // bs
    nb = B * mb
    g = torch.Generator(device="cpu").manual_seed(bs)
    table = torch.randperm(nb, generator=g).reshape(B, mb).to(torch.int32).to(dev)

    def pool_of(cache):
        pool = torch.empty((nb, Hkv, bs, d), dtype=cache.dtype, device=dev)
        flat = table.reshape(-1).long()
        for b in range(B):  # one request at a time keeps the temporary small
            padded = torch.zeros((Hkv, mb * bs, d), dtype=cache.dtype, device=dev)
            padded[:, :L_cap] = cache[b]
            pool[flat[b * mb:(b + 1) * mb]] = padded.view(Hkv, mb, bs, d).permute(1, 0, 2, 3)
        return pool

    pk, pv = pool_of(t["k"]), pool_of(t["v"])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    aa, out, lse = st.attn_args(t["q"], pk, pv, t["prefix_len"], t["n_nodes"], t["parent"], block_table=table)
    need = L.spec_tree_attention_workspace(ctypes.byref(aa))
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    pw, pst, sp = ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream.cuda_stream)

    def call():
        if L.spec_tree_attention(ctypes.byref(aa), pw, need, pst, sp):
            raise RuntimeError("spec_tree_attention (paged) failed")

    for _ in range(3):
        l2_flush()
        call()
    n = min(K, 300)
    eb, ee = events(n), events(n)
    torch.cuda.synchronize()
    for i in range(n):
        l2_flush()
        aa.timing_begin, aa.timing_end = eb[i].cuda_event, ee[i].cuda_event
        call()
    torch.cuda.synchronize()
    aa.timing_begin = aa.timing_end = None
    if int(status.item()) != 0:
        raise RuntimeError("device status " + st.status_string(int(status.item())))
    ms = statistics.median(eb[i].elapsed_time(ee[i]) for i in range(n))
    frac = max(w["attn_kernel_bytes"] / (hbm * 1e9), w["attn_flops"] / (tc * 1e12)) / (ms * 1e-3)
    del pk, pv
    return {"kernel_ms": ms, "contiguous_kernel_ms": contiguous_ms, "roofline_frac": frac, "steps": n,
            "pool_blocks": nb, "table_entries_per_request": mb}


# ---- oracle (CPU baseline / reference arm) ------------------------------------------------------

def _widen(case, name, sl):
    """float64 copy of a slice of one input (bf16 bits widened exactly)."""
    import numpy as np
    from gen import bf16 as BF
    a = getattr(case, name)[sl]
    return BF.bf16_bits_to_f64(a) if case.dtype == "bf16" else np.asarray(a, dtype=np.float64)


def oracle_request_sample(case, b, g):
    """Times the oracle on request b: tree attention on KV head g (its G query heads), the LM head,
    acceptance and longest path, and KV compaction.  Returns (tree nodes of b, estimated seconds
    of the whole request = Hkv x the attention sample + the rest)."""
    import numpy as np
    import oracle
    G = case.Hq // case.Hkv
    Lb, n = int(case.prefix_len[b]), int(case.n_nodes[b])
    q = _widen(case, "q", np.s_[b: b + 1, :, g * G:(g + 1) * G])
    k = _widen(case, "k_cache", np.s_[b: b + 1, g: g + 1, : Lb + n])
    v = _widen(case, "v_cache", np.s_[b: b + 1, g: g + 1, : Lb + n])
    h = _widen(case, "hidden", np.s_[b: b + 1])
    Wt = case.f32("W") if not hasattr(case, "_W32") else case._W32
    case._W32 = Wt
    sl = np.s_[b: b + 1]
    t0 = time.perf_counter()
    oracle.tree_attention(q, k, v, case.prefix_len[sl], case.n_nodes[sl], case.parent[sl])
    t1 = time.perf_counter()
    res = oracle.verify_accept(h, Wt, case.tokens[sl], case.parent[sl], case.n_nodes[sl], case.rule, case.tau,
                               case.eps, case.delta, case.seed,
                               draft_probs=None if case.draft_probs is None else case.draft_probs[sl],
                               draft_to_target=case.draft_to_target)
    t2 = time.perf_counter()
    oracle.compact_kv(case.k_cache[sl], case.v_cache[sl], case.prefix_len[sl], [res[0]["path"]],
                      [res[0]["accept_len"]], case.N)
    t3 = time.perf_counter()
    return n, case.Hkv * (t1 - t0) + (t2 - t1) + (t3 - t2)


def cpu_baseline(case, budget_s=20.0):
    """The oracle on a bounded sample of the workload: requests in order (cycling the KV head that
    stands for all of them), until ``budget_s`` seconds of oracle work have been spent (at least
    one request).  Rate = sampled tree nodes / their estimated oracle time."""
    nodes = est = 0.0
    done = []
    spent = 0.0
    b = 0
    while not done or spent < budget_s:
        t0 = time.perf_counter()
        n, e = oracle_request_sample(case, b % case.B, b % case.Hkv)
        spent += time.perf_counter() - t0
        nodes += n
        est += e
        done.append(b % case.B)
        b += 1
        if b >= 4 * case.B:
            break
    return {"value": nodes / est, "unit": UNIT, "cores": _threads_used(), "kind": "oracle",
            "sample": (f"{len(done)} request samples (requests {sorted(set(done))[:8]} of {case.B}): per request, "
                       f"tree attention of one KV head (its {case.Hq // case.Hkv} query heads, all nodes, all keys) "
                       f"scaled by {case.Hkv} KV heads, plus LM head over the full vocabulary, acceptance, longest "
                       "path and KV compaction in full"),
            "oracle_seconds": spent, "s_per_step_estimate": est / nodes * float(case.n_nodes.sum())}


def run_reference(a):
    from gen import make_config_case
    case = make_config_case(a.workload, seed=a.seed)
    for i in range(min(a.warmup, 1)):
        oracle_request_sample(case, i % case.B, i % case.Hkv)
    nodes = est = 0.0
    steps = 0
    t_start = time.perf_counter()
    for i in range(a.steps):  # at least one step; then as many as fit the time budget
        if steps and time.perf_counter() - t_start > a.ref_budget:
            break
        n, e = oracle_request_sample(case, i % case.B, i % case.Hkv)
        nodes += n
        est += e
        steps += 1
    v = nodes / est
    ms = float(case.n_nodes.sum()) / v * 1e3
    sample = (f"{steps} steps of {a.steps} requested (stopped after {a.ref_budget:.0f} s of oracle work), step i = "
              f"request i mod {case.B}: tree attention of KV head i mod {case.Hkv} scaled by {case.Hkv}, plus LM "
              f"head, acceptance and compaction of that request in full")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": a.gpus, "steps": steps,
            "warmup": min(a.warmup, 1), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": case.name, "batch": case.B, "prefix_len": [int(x) for x in case.prefix_len][:8],
                       "tree_nodes": [int(x) for x in case.n_nodes][:8], "rule": case.rule},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": _threads_used(), "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_native(a, rank, world, dist):
    import torch
    import tree_speculative_decoding_split_gb300 as st
    st.build()
    st.lib()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    line = measure_workload(a, a.workload, rank, world, dist, a.seed + rank, with_cpu=True)
    if a.profile:
        return None
    if a.second_workload and a.second_workload != a.workload:
        second = measure_workload(a, a.second_workload, rank, world, dist, a.seed + rank, with_cpu=True)
        if line is not None:
            line["second_workload"] = second
    return line


def main():
    a = _args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if a.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(a)), flush=True)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    line = run_native(a, rank, world, dist)
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

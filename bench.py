#!/usr/bin/env python3
"""Benchmark of one tree-verification step on GB300.

A step is the whole verification hot path over one batch: tree attention (one layer), LM head +
acceptance + longest accepted path, and KV compaction -- the three C-ABI calls
spec_tree_attention, spec_verify_accept and spec_compact_kv.  The workload is the Llama-3.1-8B
shaped layer with batch 1, a 2048-token prefix, the static 63-node Medusa-style tree and typical
acceptance (eps 0.09, delta 0.3).  Metric: verified tree-tokens/s (tree nodes verified per second).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Under torchrun each rank runs an independent replica on its own GPU (the path needs no exchange);
the JSON line reports the whole-job rate from the slowest rank.  ``--impl reference`` times the
fp64 CPU oracle on the host cores instead.
"""

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified tree-tokens/s per GB300 and % of roofline (HBM / bf16 TC) vs CPU oracle"
UNIT = "tree-tokens/s"
WORKLOAD = 2  # gen.configs: llama8b-b1-l2048-medusa63-typical
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--mode", default="graph", choices=["graph", "direct"],
                   help="graph: each step is one spec_round_launch of the captured round (default); "
                        "direct: the three C-ABI calls per step")
    p.add_argument("--workload", type=int, default=WORKLOAD,
                   help="gen.configs workload id (the headline metric is quoted on the default)")
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
    nodes = int(case.n_nodes.sum())
    rows = case.B * case.N
    kv_bytes = sum(2 * case.Hkv * (int(case.prefix_len[b]) + int(case.n_nodes[b])) * case.d * 2
                   for b in range(case.B))
    qo_bytes = 2 * nodes * case.Hq * case.d * 2 + nodes * case.Hq * 4
    w_bytes = case.V * case.Hd * 2
    h_bytes = rows * case.Hd * 2
    logits_bytes = rows * case.V * 4 if case.rule == "rejection" else 0
    lm_flops = 2.0 * rows * case.Hd * case.V
    attn_flops = sum(4.0 * case.d * case.Hq * int(case.n_nodes[b]) * int(case.prefix_len[b]) for b in range(case.B))
    return dict(nodes=nodes, kv_bytes=kv_bytes, qo_bytes=qo_bytes, w_bytes=w_bytes, h_bytes=h_bytes,
                logits_bytes=logits_bytes, lm_flops=lm_flops, attn_flops=attn_flops,
                lm_kernel_bytes=w_bytes + h_bytes + logits_bytes, attn_kernel_bytes=kv_bytes + qo_bytes)


def _traffic_from_profile(kernel_file):
    """DRAM bytes per launch of the LM-head kernel from the committed ncu summary, if the kernel source
    is unchanged since the counters were taken (else None)."""
    prof = os.path.join(ROOT, "profiles", "lmhead_tc_llama8b_b1_medusa63.md")
    if not os.path.exists(prof):
        return None
    text = open(prof).read()
    m_t = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    m_h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not (m_t and m_h):
        return None
    src = hashlib.sha256(open(kernel_file, "rb").read()).hexdigest()
    return int(m_t.group(1)) if src == m_h.group(1) else None


# ---- clocks -------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(gpu_index)], stdout=subprocess.PIPE,
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


def _launches_per_step(case):
    attn = 3 if case.dtype == "bf16" else 2                   # tree prep, split-KV, merge | prep, fp32 rows
    verify = 2 if case.dtype == "bf16" else 3                  # LM head (+stats) [+ fp32 stats], row finalise
    if case.rule == "rejection":
        verify += 1                                            # rejection walk
        if case.draft_to_target is not None:
            verify += 1                                        # draft-map inversion
    return attn + verify + 1                                   # + compaction


def run_native(a, rank, world, dist):
    import numpy as np
    import torch
    import tree_speculative_decoding_split_gb300 as st
    from gen import make_config_case

    st.build()
    L = st.lib()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    case = make_config_case(a.workload, seed=a.seed + rank)
    t = _device_tensors(case, dev)
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    aa, out, lse = st.attn_args(t["q"], t["k"], t["v"], t["prefix_len"], t["n_nodes"], t["parent"])
    va, outs = st.verify_args(t["hidden"], t["W"], t["tokens"], t["parent"], t["n_nodes"], case.rule, case.tau,
                              case.eps, case.delta, case.seed, t["draft"], t["map"], path_cap=case.N)
    ca, src_slot, new_len = st.compact_args(t["k"], t["v"], t["prefix_len"], outs["path"], outs["accept_len"])
    need_a = L.spec_tree_attention_workspace(ctypes.byref(aa))
    need_v = L.spec_verify_accept_workspace(ctypes.byref(va))
    ws_a = torch.empty(need_a, dtype=torch.uint8, device=dev)
    ws_v = torch.empty(need_v, dtype=torch.uint8, device=dev)
    pa, pv, pst = ctypes.c_void_p(ws_a.data_ptr()), ctypes.c_void_p(ws_v.data_ptr()), ctypes.c_void_p(status.data_ptr())
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_sink = torch.empty(1, dtype=torch.int64, device=dev)

    def l2_flush():
        # write a buffer twice the size of L2, then read it back, so that the step starts from a
        # cold L2 holding clean lines (no write-backs of the flush charged to the step)
        flush.zero_()
        torch.sum(flush.view(torch.int64), dim=0, keepdim=True, out=flush_sink)

    def step():
        c1 = L.spec_tree_attention(ctypes.byref(aa), pa, need_a, pst, sp)
        c2 = L.spec_verify_accept(ctypes.byref(va), pv, need_v, pst, sp)
        c3 = L.spec_compact_kv(ctypes.byref(ca), pst, sp)
        if c1 or c2 or c3:
            raise RuntimeError(f"C ABI returned {c1} {c2} {c3}")

    def events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)  # materialise the underlying cudaEvent_t
        return evs

    for _ in range(max(3, a.warmup)):
        l2_flush()
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status " + st.status_string(int(status.item())))

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

    rnd = None
    if a.mode == "graph":
        rnd = st.Round(aa, va, ca, dev_status=status)
        for _ in range(max(3, a.warmup)):
            l2_flush()
            rnd.launch(stream)
        torch.cuda.synchronize()

    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    # Per-kernel device times (the roofline's inputs) come from the direct calls, whose
    # library-recorded events bracket the attention and LM-head kernels; events recorded inside
    # a CUDA graph are not timable.  In graph mode the step time comes from the round's launches.
    direct_ms, attn_ms, lm_ms = timed_direct(K)
    step_ms = timed_graph(rnd, K) if rnd is not None else direct_ms
    clk = clocks.stop()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ms = statistics.fmean(step_ms)
    other_ms = statistics.fmean(direct_ms) if rnd is not None else None
    if int(status.item()) != 0:
        raise RuntimeError("device status " + st.status_string(int(status.item())))

    # ---- end to end: pinned host inputs -> device, the three calls, results -> pinned host ----
    n_tree = int(case.n_nodes.max())
    host = {}
    host["q"] = t["q"].cpu().pin_memory()
    host["hidden"] = t["hidden"].cpu().pin_memory()
    host["tokens"] = t["tokens"].cpu().pin_memory()
    host["parent"] = t["parent"].cpu().pin_memory()
    host["n_nodes"] = t["n_nodes"].cpu().pin_memory()
    host["prefix_len"] = t["prefix_len"].cpu().pin_memory()
    Lp = [int(x) for x in case.prefix_len]
    host["k_tree"] = [t["k"][b, :, Lp[b]:Lp[b] + n_tree].contiguous().cpu().pin_memory() for b in range(case.B)]
    host["v_tree"] = [t["v"][b, :, Lp[b]:Lp[b] + n_tree].contiguous().cpu().pin_memory() for b in range(case.B)]
    res_host = {k: torch.empty(outs[k].shape, dtype=torch.int32).pin_memory() for k in ("accept_len", "path", "bonus_token")}
    nl_host = torch.empty(new_len.shape, dtype=torch.int32).pin_memory()
    step_inputs = ["q", "hidden", "tokens", "parent", "n_nodes", "prefix_len"]
    if t["draft"] is not None:  # rejection sampling: the draft distributions arrive with every step
        host["draft"] = t["draft"].cpu().pin_memory()
        step_inputs.append("draft")
    h2d = sum(host[k].numel() * host[k].element_size() for k in step_inputs)
    h2d += sum(x.numel() * x.element_size() for x in host["k_tree"] + host["v_tree"])
    d2h = sum(x.numel() * 4 for x in res_host.values()) + nl_host.numel() * 4

    def e2e_step():
        for k in step_inputs:
            t[k].copy_(host[k], non_blocking=True)
        for b in range(case.B):
            t["k"][b, :, Lp[b]:Lp[b] + n_tree].copy_(host["k_tree"][b], non_blocking=True)
            t["v"][b, :, Lp[b]:Lp[b] + n_tree].copy_(host["v_tree"][b], non_blocking=True)
        if rnd is not None:
            rnd.launch(stream)
        else:
            step()
        for k in res_host:
            res_host[k].copy_(outs[k], non_blocking=True)
        nl_host.copy_(new_len, non_blocking=True)

    KE = max(10, min(K, 500))
    for _ in range(3):
        l2_flush()
        e2e_step()
    torch.cuda.synchronize()
    es, ee = events(KE), events(KE)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(KE):
        l2_flush()
        es[i].record(stream)
        e2e_step()
        ee[i].record(stream)
    torch.cuda.synchronize()
    e2e_ms = statistics.fmean(es[i].elapsed_time(ee[i]) for i in range(KE))

    ms, e2e_ms, other_agg = aggregate_ranks([ms, e2e_ms, other_ms or 0.0], dist, dev)
    other_ms = other_agg if other_ms is not None else None
    if rank != 0:
        return None

    w = _work(case)
    hbm, tc, tc_sus, peak_kind = _peaks()
    lm_avg = statistics.fmean(lm_ms)
    attn_avg = statistics.fmean(attn_ms)
    lm_achieved = w["lm_kernel_bytes"] / (lm_avg * 1e-3) / 1e9
    lm_tflops = w["lm_flops"] / (lm_avg * 1e-3) / 1e12
    lm_tc_bound = w["lm_flops"] / (tc * 1e12) > w["lm_kernel_bytes"] / (hbm * 1e9)
    # the committed counters are for the benchmark workload's LM-head kernel only
    traffic = (_traffic_from_profile(os.path.join(ROOT, "tree_speculative_decoding_split_gb300", "csrc", "lmhead.cu"))
               if a.workload == WORKLOAD else None)
    step_bytes = w["kv_bytes"] + w["qo_bytes"] + w["w_bytes"] + w["h_bytes"] + w["logits_bytes"]
    t_hbm = step_bytes / (hbm * 1e9)
    t_tc = (w["lm_flops"] + w["attn_flops"]) / (tc_sus * 1e12)
    t_ns = max((w["kv_bytes"] + w["w_bytes"]) / (hbm * 1e9), w["lm_flops"] / (tc_sus * 1e12))
    line = {
        "metric": METRIC, "value": job_rate(world, w["nodes"], ms), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, a.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": case.name, "batch": case.B, "prefix_len": [int(x) for x in case.prefix_len][:8],
                   "tree_nodes": int(case.n_nodes[0]), "q_heads": case.Hq, "kv_heads": case.Hkv, "head_dim": case.d,
                   "hidden": case.Hd, "vocab": case.V, "rule": case.rule, "eps": case.eps, "delta": case.delta,
                   "parallelism": f"replicas x{world}", "l2": "flushed before every step (256 MB write, then read)",
                   "launch": ("one CUDA-graph launch of the captured round per step (spec_round_launch)"
                              if rnd is not None else "three C-ABI calls per step")},
        "e2e": {"value": job_rate(world, w["nodes"], e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": K * _launches_per_step(case),
        "roofline": ({"kernel": "lmhead_tc_kernel (LM head GEMM + row statistics)", "bound": "tensor",
                      "achieved": lm_tflops, "peak": tc, "unit": "TFLOP/s", "frac": lm_tflops / tc,
                      "traffic": traffic, "algorithmic_flops": w["lm_flops"], "ms": lm_avg,
                      "peak_source": f"{peak_kind} bf16_tflops (burst)"} if lm_tc_bound else
                     {"kernel": "lmhead_tc_kernel (LM head GEMM + row statistics)", "bound": "hbm",
                      "achieved": lm_achieved, "peak": hbm, "unit": "GB/s", "frac": lm_achieved / hbm,
                      "traffic": traffic, "algorithmic_bytes": w["lm_kernel_bytes"], "ms": lm_avg,
                      "peak_source": f"{peak_kind} hbm_gbs"}),
        "kernels": {"tree_attention_splitkv_ms": attn_avg, "lmhead_ms": lm_avg,
                    "attention_achieved_gbs": w["attn_kernel_bytes"] / (attn_avg * 1e-3) / 1e9,
                    "attention_achieved_tflops": w["attn_flops"] / (attn_avg * 1e-3) / 1e12,
                    "attention_roofline_frac": max(w["attn_kernel_bytes"] / (hbm * 1e9),
                                                   w["attn_flops"] / (tc * 1e12)) / (attn_avg * 1e-3),
                    "lmhead_achieved_tflops": lm_tflops},
        "roofline_step": {"combined_s": t_ns, "frac_combined": t_ns / (ms * 1e-3),
                          "full_s": max(t_hbm, t_tc), "frac_full": max(t_hbm, t_tc) / (ms * 1e-3),
                          "peaks": f"{peak_kind}: hbm {hbm} GB/s, bf16 sustained {tc_sus} TFLOP/s"},
        "clocks": clk,
    }
    if world == 1:
        nxt = {}
        if a.workload == WORKLOAD:
            nxt["medusa_expand"] = _bench_medusa(st, L, dev, stream, l2_flush, events, K, case, hbm)
        nxt["eagle_dynamic_tree"] = _bench_eagle(st, L, dev, stream, l2_flush, events, K, case)
        nxt["paged_attention"] = {f"block_{bs}": _bench_paged(st, L, dev, stream, l2_flush, events, K, case, t, w, hbm, tc,
                                                              bs, attn_avg) for bs in (16, 64)}
        line["next_rows"] = nxt
    if other_ms is not None:
        line["direct_calls"] = {"ms_per_step": other_ms, "value": job_rate(world, w["nodes"], other_ms),
                                "note": "same workload, the three C-ABI calls per step instead of the graph"}
    if world == 1 and not a.no_cpu_baseline and a.workload == WORKLOAD:
        line["cpu_baseline"] = _cpu_baseline(case)
    return line


def _bench_medusa(st, L, dev, stream, l2_flush, events, K, case, hbm):
    """Static Medusa expansion at the workload's shapes: B requests, 5 heads of bf16 logits over
    the vocabulary, the workload's 63-node topology from per-head top-(3, 3, 2, 2, 1)."""
    import numpy as np
    import torch
    from gen import bf16 as BF
    topk_heads = (3, 3, 2, 2, 1)
    parent, rank = st.medusa_topology(topk_heads, int(case.n_nodes.max()))
    rng = np.random.default_rng(5)
    x = BF.f32_to_bf16_bits(rng.standard_normal((case.B, len(topk_heads), case.V)).astype(np.float32))
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

    for _ in range(3):
        l2_flush()
        call()
    n = min(K, 500)
    es, ee = events(n), events(n)
    torch.cuda.synchronize()
    for i in range(n):
        l2_flush()
        es[i].record(stream)
        call()
        ee[i].record(stream)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status " + st.status_string(int(status.item())))
    ms = statistics.fmean(es[i].elapsed_time(ee[i]) for i in range(n))
    nbytes = logits.numel() * 2
    return {"ms": ms, "steps": n, "bound": "hbm", "bytes": nbytes, "achieved_gbs": nbytes / (ms * 1e-3) / 1e9,
            "frac": nbytes / (ms * 1e-3) / 1e9 / hbm, "launches_per_call": 2,
            "shape": {"batch": case.B, "heads": len(topk_heads), "vocab": case.V, "topk": list(topk_heads),
                      "nodes": int(len(parent)), "dtype": "bf16"}}


def _bench_eagle(st, L, dev, stream, l2_flush, events, K, case):
    """Dynamic draft tree at the workload's batch: one expansion layer (frontier 8, top-8 over a
    32000-entry draft vocabulary) and the selection of an N-node tree from 8 stacked layers."""
    import numpy as np
    import torch
    B, F, k, Vd, D = case.B, 8, 8, 32000, 8
    N = int(min(case.N, 255))
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
    for l in range(1, D):
        Sn[:, l] = np.take_along_axis(Sn[:, l - 1], Pn[:, l], axis=1) - rng.exponential(1.0, (B, C))
    S = torch.from_numpy(Sn).to(dev)
    Tk = torch.from_numpy(rng.integers(0, Vd, (B, D, C)).astype(np.int32)).to(dev)
    P = torch.from_numpy(Pn).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def timed(call, n):
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
        return statistics.fmean(es[i].elapsed_time(ee[i]) for i in range(n))

    n = min(K, 300)
    layer_ms = timed(lambda: st.eagle_expand(lp, fs, k, F, dev_status=status, stream=stream), n)
    tree_ms = timed(lambda: st.eagle_tree(S, Tk, P, N, dev_status=status, stream=stream), n)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status " + st.status_string(int(status.item())))
    return {"expand_layer_ms": layer_ms, "select_tree_ms": tree_ms, "steps": n,
            "shape": {"batch": B, "frontier": F, "topk": k, "draft_vocab": Vd, "layers": D, "nodes": N},
            "note": "timed through the Python binding (argument marshalling included)"}


def _bench_paged(st, L, dev, stream, l2_flush, events, K, case, t, w, hbm, tc, bs, contiguous_ms):
    """Tree attention of the workload with its KV cache scattered over a shuffled block pool."""
    import torch
    B, Hkv, L_cap, d = t["k"].shape
    mb = (L_cap + bs - 1) // bs
    nb = B * mb
    g = torch.Generator(device="cpu").manual_seed(bs)
    table = torch.randperm(nb, generator=g).reshape(B, mb).to(torch.int32).to(dev)

    def pool_of(cache):
        padded = torch.zeros((B, Hkv, mb * bs, d), dtype=cache.dtype, device=dev)
        padded[:, :, :L_cap] = cache
        blocks = padded.view(B, Hkv, mb, bs, d).permute(0, 2, 1, 3, 4).reshape(B * mb, Hkv, bs, d)
        pool = torch.empty(blocks.shape, dtype=blocks.dtype, device=dev)
        pool[table.reshape(-1).long()] = blocks
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
    ms = statistics.fmean(eb[i].elapsed_time(ee[i]) for i in range(n))
    frac = max(w["attn_kernel_bytes"] / (hbm * 1e9), w["attn_flops"] / (tc * 1e12)) / (ms * 1e-3)
    return {"kernel_ms": ms, "contiguous_kernel_ms": contiguous_ms, "roofline_frac": frac, "steps": n,
            "pool_blocks": nb, "table_entries_per_request": mb}


# ---- oracle (CPU baseline / reference arm) ------------------------------------------------------

def _oracle_inputs(case):
    return dict(q=case.f64("q"), k=case.f64("k_cache"), v=case.f64("v_cache"), h=case.f64("hidden"),
                W=case.f32("W"))


def _oracle_step(case, x):
    import oracle
    oracle.tree_attention(x["q"], x["k"], x["v"], case.prefix_len, case.n_nodes, case.parent)
    res = oracle.verify_accept(x["h"], x["W"], case.tokens, case.parent, case.n_nodes, case.rule, case.tau, case.eps,
                               case.delta, case.seed, draft_probs=case.draft_probs,
                               draft_to_target=case.draft_to_target)
    paths = [r["path"] for r in res]
    alen = [r["accept_len"] for r in res]
    oracle.compact_kv(case.k_cache, case.v_cache, case.prefix_len, paths, alen, case.N)


def _cpu_baseline(case, budget_s=20.0):
    x = _oracle_inputs(case)
    times = []
    t_all = time.perf_counter()
    while not times or (time.perf_counter() - t_all < budget_s and len(times) < 5):
        t0 = time.perf_counter()
        _oracle_step(case, x)
        times.append(time.perf_counter() - t0)
    nodes = int(case.n_nodes.sum())
    return {"value": nodes / statistics.fmean(times), "unit": UNIT, "cores": _threads_used(), "kind": "oracle",
            "sample": f"{len(times)} full steps of the workload (all {nodes} nodes, all heads, full vocabulary)",
            "s_per_step": statistics.fmean(times)}


def run_reference(a):
    from gen import make_config_case
    case = make_config_case(a.workload, seed=a.seed)
    x = _oracle_inputs(case)
    for _ in range(a.warmup if a.warmup < 3 else 1):
        _oracle_step(case, x)
    times = []
    for _ in range(a.steps if a.steps <= 20 else 20):
        t0 = time.perf_counter()
        _oracle_step(case, x)
        times.append(time.perf_counter() - t0)
    nodes = int(case.n_nodes.sum())
    s = statistics.fmean(times)
    v = nodes / s
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": a.gpus, "steps": len(times),
            "warmup": a.warmup, "ms_per_step": s * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": case.name, "batch": case.B, "prefix_len": [int(x) for x in case.prefix_len][:8],
                       "tree_nodes": nodes, "rule": case.rule},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": _threads_used(), "kind": "oracle",
                             "sample": f"{len(times)} full steps of the workload (capped at 20 timed steps)"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


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

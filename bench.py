#!/usr/bin/env python3
"""Benchmark: tree-structured decode attention, one decode step per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long|tiny|wide|three|irreg]

One step = one tree_attn_run() of the workload (the partial-attention pass and
the log-sum-exp merge, one layer), inputs resident in HBM, L2 flushed before
every step outside the step's events: a 512 MiB memset, then a 256 MiB read,
so that the step starts from clean L2 lines (after the memset alone, the
step's cold reads would also pay for writing back the memset's dirty lines).
The default workload is the largest of the five synthetic trees: the
irregular random tree (depth 4-5, branching 1-8, node lengths log-uniform in
16-2048, ~1000 leaves each carrying 4 speculative query tokens with a causal
mask over its own last 4 tokens; 64 q / 4 kv heads, d = 128), bf16 N(0, 1)
Q/K/V in 16-token pages in shuffled order.  The other four trees are timed
the same way (fewer steps) and reported under "per_workload".  Beside the
step: "layer_chain" (eight layers back to back, each its own Q and K/V),
"append" (the step's K/V append, tree_attn_append_kv, timed alone) and
"plan_ablation" (the headline tree under other plans and the fused merge).

Metric: algorithmic HBM bytes per second (unique KV + Q + out + lse bytes of
the step / device time of the step), with ms per step beside it.  Under
torchrun each rank runs its own replica (the path has no exchange step) and
rank 0 prints one JSON line; value = bytes of all ranks / max time.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "tree-attn decode ms/step and HBM GB/s (frac of roofline) on 1 GB300"
WORKLOAD_DESC = {
    "long": "long-context tail tree, Llama-2-7B attention shape: root 4000 + 10 leaves x 400, "
            "1 decode query per leaf, 32 q / 32 kv heads, d 128, bf16, 16-token pages",
    "tiny": "root 256 + 4 leaves x 32, 4/4 heads, d 64",
    "wide": "root 2048 + 256 leaves x 64, 32/8 heads (GQA 4), d 128",
    "three": "root 1024, 16 x 512, 16 x 16 leaves x 128, 32/32 heads, d 128",
    "irreg": "irregular tree ~1000 leaves, 4 speculative tokens per leaf, 64/4 heads, d 128",
}
L2_FLUSH_BYTES = 512 << 20
L2_CLEAN_BYTES = 256 << 20


class L2Flush:
    """Evicts the step's inputs from L2 (a memset larger than L2), then reads
    a second buffer larger than L2 so that the lines left behind are clean."""

    def __init__(self, dev):
        import torch
        self.torch = torch
        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.clean = torch.zeros(L2_CLEAN_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        self.buf.zero_()
        self.torch.sum(self.clean, dim=0, out=self.sink)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def algorithmic_work(spec):
    """Bytes and FLOPs one step must move / do, whatever the plan:
    unique KV once (K and V, bf16), Q once (bf16), out (fp32) and lse (fp32)
    once; FLOPs = sum over query tokens of Hq * visible keys * 4d."""
    hq, hkv, d = spec.n_q_heads, spec.n_kv_heads, spec.head_dim
    kv = int(spec.node_kv_len.sum()) * hkv * d * 2 * 2
    qb = spec.n_queries * hq * d * 2
    ob = spec.n_queries * hq * (d + 1) * 4
    vis = 0
    for t in range(spec.n_queries):
        u = int(spec.query_node[t])
        n = int(spec.query_kv_end[t])
        x = int(spec.parent[u])
        while x >= 0:
            n += int(spec.node_kv_len[x])
            x = int(spec.parent[x])
        vis += n
    return {"bytes": kv + qb + ob, "kv_bytes": kv, "flops": 4.0 * d * hq * vis,
            "visible_pairs": vis}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


CSRC = os.path.join(ROOT, "tree_structured_decode_gb300", "csrc")


def source_hash() -> str:
    """sha256 (16 hex digits) over every source file of the library (kernels,
    planner, runtime), in name order: a profile taken on other sources does
    not describe the kernels this run times."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".cpp", ".h")):
            h.update(name.encode())
            h.update(open(os.path.join(CSRC, name), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch of the partial-attention kernel from the
    committed ncu summary of this workload, if that summary was captured on
    the current library sources; else None."""
    path = os.path.join(ROOT, "profiles", f"partial_attention_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_sha = re.search(r"library_source_sha256_16:\s*([0-9a-f]+)", txt)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.e+]+)", txt)
    if m_sha and m_b and m_sha.group(1) == source_hash():
        return float(m_b.group(1))
    return None


class NvmlClocks:
    """SM clock and clock-event (throttle) reasons polled through NVML (the
    library nvidia-smi reads) every ~2 ms on a thread while the timed steps
    run, so that even a short timed region gets many samples."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        import ctypes
        import threading

        self.ok = False
        self.samples = []
        self._stop = threading.Event()
        self._thread = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            got = False
            try:
                import torch
                uuid = str(torch.cuda.get_device_properties(torch_device).uuid)
                if not uuid.startswith("GPU-"):
                    uuid = "GPU-" + uuid
                got = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            except Exception:
                got = False
            if not got:
                idx = torch_device.index or 0
                got = lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) == 0
            if not got:
                return
            self.lib, self.h = lib, h
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 \
                else None
            self.ctypes = ctypes
            self.ok = True
        except OSError:
            return

    def _poll(self):
        c = self.ctypes
        mhz, rs = c.c_uint(), c.c_ulonglong()
        while not self._stop.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz)) == 0 and \
                    self.reasons_fn(self.h, c.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            time.sleep(0.002)

    def __enter__(self):
        import threading

        if self.ok:
            self._stop.clear()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *a):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            self._thread = None

    def result(self):
        if not self.samples:
            return None
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        sm = [m for m, _ in self.samples]
        return {"sm_mhz": float(np.median(sm)), "sm_min_mhz": float(min(sm)),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(sm), "source": "NVML, polled every ~2 ms during the timed steps"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.out = open(os.devnull, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        pass

    def result(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, val in zip(names, f[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_max_over_ranks(vals, world, device):
    """Each timing's maximum over all ranks: the slowest replica sets the
    step time of the whole job."""
    if world <= 1:
        return [float(x) for x in vals]
    import torch

    t = torch.tensor([float(x) for x in vals], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def aggregate_gbs(bytes_per_step, world, step_ms):
    """Whole-job throughput: every replica processes one step's bytes in the
    (slowest) step time."""
    return bytes_per_step * world / (step_ms * 1e-3) / 1e9


# --------------------------------------------------------------------------- ours
def time_steps(plan, q, k, v, out, lse, flush, stream, steps, warmup, clocks=None):
    """Warm up, then time `steps` steps (one event pair around each whole
    run(), L2 flushed before each outside the events); then the same steps
    again with the library's per-kernel events (they sit between the two
    kernels, so they stay out of the step time)."""
    import torch

    for _ in range(warmup):
        flush()
        plan.run(q, k, v, out=out, lse=lse)
    torch.cuda.synchronize()
    step_ms, part_ms, merge_ms = [], [], []
    if clocks is not None:
        clocks.__enter__()
    try:
        for _ in range(steps):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            plan.run(q, k, v, out=out, lse=lse)
            e1.record(stream)
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
    finally:
        if clocks is not None:
            clocks.__exit__()
    plan.profile(True)
    for _ in range(steps):
        flush()
        plan.run(q, k, v, out=out, lse=lse)
        a, b = plan.kernel_times()
        part_ms.append(a)
        merge_ms.append(b)
    plan.profile(False)
    torch.cuda.synchronize()
    return step_ms, part_ms, merge_ms


def time_layer_chain(plan, spec, dev, flush, stream, layers, iters=20, warmup=3):
    """Per-layer time of `layers` back-to-back runs of the plan, each over
    its own seeded Q and K/V pages (a decode step's layers), between one
    event pair; L2 flushed before every chain.  Within a chain each run's
    partial-attention kernel is a programmatic dependent of the previous
    run's last kernel.  Returns (ms per layer, median over iters)."""
    import torch

    data = [W.make_tensors(spec, seed=1000 + i, device=dev) for i in range(layers)]
    out = torch.empty((spec.n_queries, spec.n_q_heads, spec.head_dim), dtype=torch.float32,
                      device=dev)
    lse = torch.empty((spec.n_queries, spec.n_q_heads), dtype=torch.float32, device=dev)
    res = []
    for i in range(warmup + iters):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for q, k, v in data:
            plan.run(q, k, v, out=out, lse=lse)
        e1.record(stream)
        e1.synchronize()
        if i >= warmup:
            res.append(e0.elapsed_time(e1) / layers)
    del data
    torch.cuda.empty_cache()
    return float(np.median(res))


def time_append(plan, spec, k, v, dev, flush, stream, steps, warmup=3):
    """The decode step's K/V append (tree_attn_append_kv) for the workload's
    query tokens, timed alone on copies of the page pools (L2 flushed before
    each, one event pair around each).  Returns (median ms, bytes moved: the
    new keys and values read and written once)."""
    import torch

    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    shape = (spec.n_queries, spec.n_kv_heads, spec.head_dim)
    kn = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    vn = torch.randn(shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
    kk, vv = k.clone(), v.clone()
    res = []
    for i in range(warmup + steps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        plan.append_kv(kn, vn, kk, vv)
        e1.record(stream)
        e1.synchronize()
        if i >= warmup:
            res.append(e0.elapsed_time(e1))
    nbytes = 2 * 2 * kn.numel() * kn.element_size()
    del kk, vv, kn, vn
    torch.cuda.empty_cache()
    return float(np.median(res)), nbytes


def roofline(work, t_part, t_step, workload):
    """The partial-attention kernel against the slower of the HBM and tensor
    bounds of the step's algorithmic bytes and FLOPs (measured peaks)."""
    hbm_peak, tc_peak, peak_kind = measured_peaks()
    t_hbm = work["bytes"] / (hbm_peak * 1e9)
    t_tc = work["flops"] / (tc_peak * 1e12)
    if t_hbm >= t_tc:
        kern_gbs = work["bytes"] / (t_part * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(kern_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(kern_gbs / hbm_peak, 4)}
    else:
        tf = work["flops"] / (t_part * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": tc_peak, "unit": "TFLOP/s",
                "frac": round(tf / tc_peak, 4)}
    roof["peak_source"] = peak_kind + " (burst: the kernel is timed alone)"
    roof["traffic"] = committed_traffic(workload)
    roof["kernel"] = "partial attention pass (tree_attn_kernel)"
    roof["kernel_ms"] = round(t_part, 5)
    roof["step_roofline_frac"] = round(max(t_hbm, t_tc) * 1e3 / t_step, 4)
    return roof


def bench_workload(name, dev, flush, stream, steps, warmup, opts, clocks=None, chain_layers=0):
    """Plan and time one workload; returns its numbers and the live objects."""
    import torch

    import tree_structured_decode_gb300 as ta

    spec = W.CONFIGS[name]()
    work = algorithmic_work(spec)
    q, k, v = W.make_tensors(spec, device=dev)
    plan = ta.Plan.from_spec(spec, **opts)
    stats = plan.stats()
    out = torch.empty((spec.n_queries, spec.n_q_heads, spec.head_dim), dtype=torch.float32,
                      device=dev)
    lse = torch.empty((spec.n_queries, spec.n_q_heads), dtype=torch.float32, device=dev)
    step_ms, part_ms, merge_ms = time_steps(plan, q, k, v, out, lse, flush, stream, steps, warmup,
                                            clocks)
    chain_ms = (time_layer_chain(plan, spec, dev, flush, stream, chain_layers)
                if chain_layers > 0 else None)
    code = plan.device_status()
    return {"spec": spec, "work": work, "plan": plan, "stats": stats, "q": q, "k": k, "v": v,
            "out": out, "lse": lse, "step_ms": step_ms, "part_ms": part_ms, "merge_ms": merge_ms,
            "chain_ms": chain_ms, "device_status": code}


def chain_record(work, chain_ms, layers):
    if chain_ms is None:
        return None
    return {"layers": layers, "ms_per_layer": round(chain_ms, 5),
            "gbs": round(work["bytes"] / (chain_ms * 1e-3) / 1e9, 1)}


def bench_ours(args, rank, world, local):
    import torch

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    opts = dict(args.plan_opts)
    spec0 = W.CONFIGS[args.workload]()
    if args.edges != "greedy":  # plan ablation: every edge 0 (no joins) or 1 (join every chain)
        opts["force_edges"] = np.full(spec0.n_nodes, 1 if args.edges == "one" else 0, dtype=np.int8)
    del spec0

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = NvmlClocks(dev)
    r = bench_workload(args.workload, dev, flush, stream, args.steps, args.warmup, opts,
                       clocks if clocks.ok else None, args.chain_layers)
    if world > 1:
        torch.distributed.barrier()
    spec, work, plan, stats = r["spec"], r["work"], r["plan"], r["stats"]
    q, k, v, out, lse = r["q"], r["k"], r["v"], r["out"], r["lse"]
    launches_per_step = 1 + (1 if stats["n_merge_tokens"] > 0 else 0)

    # ---- end to end through the public API, host buffers (pinned) both ways
    hq_, hk_, hv_ = (t.cpu().pin_memory() for t in (q, k, v))
    ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dq.copy_(hq_, non_blocking=True)
        dk.copy_(hk_, non_blocking=True)
        dv.copy_(hv_, non_blocking=True)
        plan.run(dq, dk, dv, out=out, lse=lse)
        ho.copy_(out, non_blocking=True)
        hl.copy_(lse, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    del dq, dk, dv, hq_, hk_, hv_

    # ---- the step before the path: the new tokens' K/V into their pages
    t_app, app_bytes = time_append(plan, spec, k, v, dev, flush, stream, args.per_workload_steps)

    t_step = float(np.mean(r["step_ms"]))
    t_part = float(np.mean(r["part_ms"]))
    t_merge = float(np.mean(r["merge_ms"]))
    t_e2e = float(np.mean(e2e_ms))
    t_step, t_e2e, t_part = reduce_max_over_ranks([t_step, t_e2e, t_part], world, dev)
    gbs = aggregate_gbs(work["bytes"], world, t_step)
    roof = roofline(work, t_part, t_step, args.workload)
    roof["merge_ms"] = round(t_merge, 5)

    # ---- the other workloads, the same way (fewer steps)
    per = {}
    if not args.no_per_workload:
        others = [n for n in ("tiny", "long", "wide", "three", "irreg") if n != args.workload]
        for name in others:
            rr = bench_workload(name, dev, flush, stream, args.per_workload_steps,
                                min(args.warmup, 5), dict(args.plan_opts),
                                chain_layers=args.chain_layers)
            ts = float(np.mean(rr["step_ms"]))
            tp = float(np.mean(rr["part_ms"]))
            rf = roofline(rr["work"], tp, ts, name)
            per[name] = {"workload": WORKLOAD_DESC[name], "steps": args.per_workload_steps,
                         "ms_per_step": round(ts, 5),
                         "gbs_step": round(rr["work"]["bytes"] / (ts * 1e-3) / 1e9, 1),
                         "kernel_ms": round(tp, 5),
                         "merge_ms": round(float(np.mean(rr["merge_ms"])), 5),
                         "kernel_frac": rf["frac"], "bound": rf["bound"],
                         "step_frac": rf["step_roofline_frac"], "traffic": rf["traffic"],
                         "alg_bytes_per_step": rr["work"]["bytes"],
                         "n_units": rr["stats"]["n_units"],
                         "layer_chain": chain_record(rr["work"], rr["chain_ms"], args.chain_layers),
                         "device_status": rr["device_status"]}
            rr["plan"].close()
            del rr
            torch.cuda.empty_cache()

    # ---- plan ablation on this workload (the pages' "greedy grouping"
    # against fixed edge assignments, and the latency model against the
    # pages' cost proxy)
    ablation = {}
    if not args.no_ablation and args.edges == "greedy" and not args.plan_opts:
        variants = (("greedy_latency_model", {}), ("greedy_pages_proxy", {"cost_model": 1}),
                    ("every_edge_0", {"force_edges": np.zeros(spec.n_nodes, dtype=np.int8)}),
                    ("every_edge_1", {"force_edges": np.ones(spec.n_nodes, dtype=np.int8)}),
                    ("fused_merge", {"merge_mode": 1}))
        for name, opts2 in variants:
            rr = bench_workload(args.workload, dev, flush, stream, args.per_workload_steps,
                                min(args.warmup, 5), opts2)
            ablation[name] = {"ms_per_step": round(float(np.mean(rr["step_ms"])), 5),
                              "kernel_ms": round(float(np.mean(rr["part_ms"])), 5),
                              "merge_ms": round(float(np.mean(rr["merge_ms"])), 5),
                              "n_units": rr["stats"]["n_units"],
                              "n_partials": rr["stats"]["n_partials"],
                              "group_kv_tokens": rr["stats"]["group_kv_tokens"],
                              "device_status": rr["device_status"]}
            rr["plan"].close()
            del rr
            torch.cuda.empty_cache()
        best_fixed = min(ablation["every_edge_0"]["ms_per_step"], ablation["every_edge_1"]["ms_per_step"])
        ablation["greedy_speedup_over_best_fixed"] = round(
            best_fixed / ablation["greedy_latency_model"]["ms_per_step"], 3)
        ablation["steps_each"] = args.per_workload_steps

    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step, 5),
        "ms_per_step_p10_p50_p90": [round(float(x), 5)
                                    for x in np.percentile(r["step_ms"], [10, 50, 90])],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, shuffled 16-token pages)",
        "config": {"workload": WORKLOAD_DESC[args.workload], "name": args.workload,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed before every step outside the step events (512 MiB memset, then a 256 MiB read: clean lines)",
                   "alg_bytes_per_step": work["bytes"], "alg_flops_per_step": work["flops"],
                   "plan": {k: stats[k] for k in ("n_groups", "n_groups_mma", "n_units", "grid",
                                                  "n_partials", "chunk_tokens", "plan_ms")},
                   "plan_options": args.plan_opts, "edges": args.edges,
                   "library_source_sha256_16": source_hash()},
        "e2e": {"value": round(aggregate_gbs(work["bytes"], world, t_e2e), 2), "unit": "GB/s",
                "ms_per_step": round(t_e2e, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roof,
        "layer_chain": chain_record(work, r["chain_ms"], args.chain_layers),
        "append": {"ms": round(t_app, 5), "bytes": app_bytes,
                   "gbs": round(app_bytes / (t_app * 1e-3) / 1e9, 1)},
        "clocks": clocks.result() if clocks.ok else None,
        "device_status": r["device_status"],
        "per_workload": per,
        "plan_ablation": ablation,
    }
    if line["clocks"] is None:  # NVML unavailable: nvidia-smi over a repeat of the steps
        with ClockSampler(local) as clk:
            time_steps(plan, q, k, v, out, lse, flush, stream, max(args.steps, 200), 0)
            line["clocks"] = clk.result()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, q, k, v, work, args.cpu_seconds, args.workload)
    plan.close()
    return line


# --------------------------------------------------------------------------- oracle
def _oracle_sample(spec, q, k, v, budget_s):
    """Time the oracle over query tokens until ~budget_s; return
    (seconds per full step extrapolated by visible pairs, sample note, cores)."""
    import oracle

    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    vis = []
    for t in range(spec.n_queries):
        u = int(spec.query_node[t])
        n = int(spec.query_kv_end[t])
        x = int(spec.parent[u])
        while x >= 0:
            n += int(spec.node_kv_len[x])
            x = int(spec.parent[x])
        vis.append(n)
    order = list(range(spec.n_queries))
    done, pairs = 0, 0
    c0, w0 = time.process_time(), time.perf_counter()
    while done < len(order) and time.perf_counter() - w0 < budget_s:
        t = order[done]
        oracle.tree_attention_spec(spec, qc, kc, vc, tokens=[t])
        pairs += vis[t]
        done += 1
    wall = time.perf_counter() - w0
    cpu = time.process_time() - c0
    total_pairs = sum(vis)
    full_s = wall * total_pairs / max(pairs, 1)
    note = (f"{done} of {spec.n_queries} query tokens ({pairs} of {total_pairs} visible "
            f"token-keys, all heads); time scaled to the full step by visible keys")
    cores = max(1, int(round(cpu / max(wall, 1e-9))))
    return full_s, note, cores


_ONE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                   "BLIS_NUM_THREADS", "NUMEXPR_NUM_THREADS")


def _single_core_sample(workload, budget_s):
    """The oracle's seconds per full step on one core: a child process with
    every BLAS / OpenMP pool set to one thread (set before numpy loads)."""
    env = dict(os.environ)
    for name in _ONE_THREAD_ENV:
        env[name] = "1"
    cmd = [sys.executable, os.path.abspath(__file__), "--single-core-sample", workload,
           "--cpu-seconds", str(budget_s)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=budget_s * 4 + 120)
        return json.loads(r.stdout.strip().splitlines()[-1]) if r.returncode == 0 else None
    except (subprocess.TimeoutExpired, ValueError, IndexError):
        return None


def cpu_baseline(spec, q, k, v, work, budget_s, workload):
    full_s, note, cores = _oracle_sample(spec, q, k, v, budget_s)
    line = {"value": round(work["bytes"] / full_s / 1e9, 4), "unit": "GB/s", "cores": cores,
            "cores_available": len(os.sched_getaffinity(0)), "kind": "oracle", "sample": note,
            "ms_per_step": round(full_s * 1e3, 2)}
    one = _single_core_sample(workload, max(2.0, budget_s / 3))
    if one:
        line["single_core"] = {"value": round(work["bytes"] / one["full_s"] / 1e9, 4), "unit": "GB/s",
                               "ms_per_step": round(one["full_s"] * 1e3, 2), "sample": one["note"]}
    return line


def bench_reference(args, rank, world):
    if rank != 0:
        return None
    import torch

    spec = W.CONFIGS[args.workload]()
    work = algorithmic_work(spec)
    q, k, v = W.make_tensors(spec, device="cpu")
    per_step = max(2.0, min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        _oracle_sample(spec, q, k, v, per_step)
    times, notes, cores = [], None, 1
    for _ in range(args.steps):
        s, notes, cores = _oracle_sample(spec, q, k, v, per_step)
        times.append(s)
    t = float(np.mean(times))
    val = round(work["bytes"] / t / 1e9, 4)
    del torch
    return {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, shuffled 16-token pages)",
        "config": {"workload": WORKLOAD_DESC[args.workload], "name": args.workload},
        "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": notes},
        "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="irreg", choices=sorted(W.CONFIGS))
    ap.add_argument("--per-workload-steps", type=int, default=20)
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--no-ablation", action="store_true")
    ap.add_argument("--chain-layers", type=int, default=8,
                    help="layers of the per-layer chain timing (0: skip)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--single-core-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--edges", default="greedy", choices=["greedy", "zero", "one"],
                    help="edge assignment: the greedy algorithm, or every edge 0 / 1 (ablation)")
    ap.add_argument("--plan", action="append", default=[], metavar="KEY=VALUE",
                    help="planner option (tree_attn_options field), e.g. --plan gamma=16")
    args = ap.parse_args()
    args.plan_opts = {}
    for kv in args.plan:
        k, _, v = kv.partition("=")
        args.plan_opts[k] = int(v)
    args.warmup = max(3, args.warmup)
    if args.single_core_sample:  # child of cpu_baseline(): one thread everywhere
        import torch

        torch.set_num_threads(1)
        spec = W.CONFIGS[args.single_core_sample]()
        q, k, v = W.make_tensors(spec, device="cpu")
        full_s, note, _ = _oracle_sample(spec, q, k, v, args.cpu_seconds)
        print(json.dumps({"full_s": full_s, "note": note}))
        return
    rank, world, local = dist_env()
    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        line = bench_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = bench_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

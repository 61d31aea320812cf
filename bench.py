#!/usr/bin/env python3
"""Benchmark: tree-structured decode attention, one decode step per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long|tiny|wide|three|irreg]

One step = one tree_attn_run() of the workload (the partial-attention pass and
the log-sum-exp merge, one layer), inputs resident in HBM, L2 flushed before
every step outside the step's events: a 512 MiB memset, then a 256 MiB read,
so that the step starts from clean L2 lines (after the memset alone, the
step's cold reads would also pay for writing back the memset's dirty lines).  The workload is the
long-context tail tree with the Llama-2-7B attention shape (32 q heads = 32 kv
heads, d = 128, one layer): root 4000 tokens, 10 leaves of 400, one decode
query per leaf, bf16 N(0, 1) Q/K/V in 16-token pages in shuffled order.

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


def committed_traffic(kernel_src: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if the summary was taken on the current kernel source."""
    sha = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    path = os.path.join(ROOT, "profiles", f"partial_attention_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.e+]+)", txt)
    if m_sha and m_b and m_sha.group(1) == sha:
        return float(m_b.group(1))
    return None


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
def bench_ours(args, rank, world, local):
    import torch

    import tree_structured_decode_gb300 as ta

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = W.CONFIGS[args.workload]()
    work = algorithmic_work(spec)
    q, k, v = W.make_tensors(spec, device=dev)
    torch.cuda.synchronize()
    opts = dict(args.plan_opts)
    if args.edges != "greedy":  # plan ablation: every edge 0 (no joins) or 1 (join every chain)
        opts["force_edges"] = np.full(spec.n_nodes, 1 if args.edges == "one" else 0, dtype=np.int8)
    plan = ta.Plan.from_spec(spec, **opts)
    stats = plan.stats()
    out = torch.empty((spec.n_queries, spec.n_q_heads, spec.head_dim), dtype=torch.float32,
                      device=dev)
    lse = torch.empty((spec.n_queries, spec.n_q_heads), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    launches_per_step = 1 + (1 if stats["n_merge_tokens"] > 0 else 0)

    for _ in range(args.warmup):
        flush()
        plan.run(q, k, v, out=out, lse=lse)
    torch.cuda.synchronize()
    assert plan.device_status() == 0

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    step_ms, part_ms, merge_ms = [], [], []
    with ClockSampler(local) as clk:
        # the steps: one event pair around each whole run()
        for _ in range(args.steps):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            plan.run(q, k, v, out=out, lse=lse)
            e1.record(stream)
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
        # the same steps again with the library's per-kernel events (they
        # sit between the two kernels, so they are kept out of the step time)
        plan.profile(True)
        for _ in range(args.steps):
            flush()
            plan.run(q, k, v, out=out, lse=lse)
            a, b = plan.kernel_times()
            part_ms.append(a)
            merge_ms.append(b)
        plan.profile(False)
        torch.cuda.synchronize()
        clocks = clk.result()
    if world > 1:
        torch.distributed.barrier()
    code = plan.device_status()

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

    t_step = float(np.mean(step_ms))
    t_part = float(np.mean(part_ms))
    t_e2e = float(np.mean(e2e_ms))
    t_step, t_e2e, t_part = reduce_max_over_ranks([t_step, t_e2e, t_part], world, dev)
    hbm_peak, tc_peak, peak_kind = measured_peaks()
    gbs = aggregate_gbs(work["bytes"], world, t_step)
    kern_gbs = work["bytes"] / (t_part * 1e-3) / 1e9
    t_hbm = work["bytes"] / (hbm_peak * 1e9)
    t_tc = work["flops"] / (tc_peak * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(kern_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(kern_gbs / hbm_peak, 4)}
    else:
        tf = work["flops"] / (t_part * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(tf, 1), "peak": tc_peak, "unit": "TFLOP/s",
                "frac": round(tf / tc_peak, 4)}
    roof["peak_source"] = peak_kind
    roof["traffic"] = committed_traffic(
        os.path.join(ROOT, "tree_structured_decode_gb300", "csrc", "tree_attn_kernel.cu"),
        args.workload)
    roof["kernel"] = "partial attention pass"
    roof["kernel_ms"] = round(t_part, 5)
    roof["merge_ms"] = round(float(np.mean(merge_ms)), 5)
    roof["step_roofline_frac"] = round(max(t_hbm, t_tc) * 1e3 / t_step, 4)

    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step, 5),
        "ms_per_step_p10_p50_p90": [round(float(x), 5) for x in np.percentile(step_ms, [10, 50, 90])],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, shuffled 16-token pages)",
        "config": {"workload": WORKLOAD_DESC[args.workload], "name": args.workload,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed before every step outside the step events (512 MiB memset, then a 256 MiB read: clean lines)",
                   "alg_bytes_per_step": work["bytes"], "alg_flops_per_step": work["flops"],
                   "plan": {k: stats[k] for k in ("n_groups", "n_groups_mma", "n_units", "grid",
                                                  "n_partials", "chunk_tokens", "plan_ms")},
                   "plan_options": args.plan_opts, "edges": args.edges},
        "e2e": {"value": round(aggregate_gbs(work["bytes"], world, t_e2e), 2), "unit": "GB/s",
                "ms_per_step": round(t_e2e, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roof,
        "clocks": clocks,
        "device_status": code,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, q, k, v, work, args.cpu_seconds, args.workload)
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
    ap.add_argument("--workload", default="long", choices=sorted(W.CONFIGS))
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

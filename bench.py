#!/usr/bin/env python3
"""Throughput of the MoE route -> plan -> permute -> combine hot path.

One step = route_topk + plan (2 launches) + permute + combine over one batch
of a synthetic workload already resident in HBM (experts are the identity:
the combine reads the permuted buffer back).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config large]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

The default workload is the large dedup-heavy one (N=65536, E=256, K=8,
R=64, H=7168); --config picks one of the other four.

Multi-GPU runs are independent replicas of the same workload on every rank
(the path has no exchange step on one node's logical ranks): value = all
ranks' tokens / the slowest rank's time.  Under torchrun the ranks come from
the environment; a plain ``python bench.py --gpus N`` (N > 1) starts the N
ranks itself through torch.distributed.run on 127.0.0.1.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "routed tokens/s (route+plan+permute+combine)"
L2_BYTES = 129 * 1024 * 1024
BALANCED_B = 4             # redundant experts per rank in the balanced-plan timing
RANK_LAYOUT_CHANNELS = 76  # channels in the rank-layout timing (half the SMs)


# ---------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, group=None) -> float:
    """Max over ranks (identity without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def barrier(group=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier(group=group)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def algorithmic_bytes(w, P: int) -> dict:
    """HBM bytes each kernel must move at minimum (per launch)."""
    N, E, K, H, R = w.N, w.E, w.K, w.H, w.R
    NK = N * K
    return {
        "route": 4 * N * E + 8 * NK + (4 * E if w.bias else 0),
        "plan_count": 4 * NK,
        "plan_scatter": 4 * NK + 4 * NK + 4 * (NK + E * (w.alignment - 1)) + N * R + 4 * NK,
        "route_plan_fused": 4 * N * E + 8 * NK + (4 * E if w.bias else 0) + 4 * NK + 4 * NK
                      + 4 * (NK + E * (w.alignment - 1)) + N * R + 4 * NK,
        "permute": 2 * N * H + 2 * P * H + 4 * NK,
        "combine": 2 * NK * H + 2 * N * H + 8 * NK,
        # planning extensions: balanced plan (topk in, dst out, its R x E
        # matrices), tile map (counts in, two int32 per tile out), rank layout
        # (is_token_in_rank in; per-(token, rank) slots and the channel matrix out)
        "balanced": 8 * NK + 4 * (E + R * R + 3 * R * E + 3 * R * (E + BALANCED_B)),
        "tile_map": 4 * E + 8 * ((NK + E * (w.alignment - 1)) // w.alignment),
        "rank_layout": N * R + 4 * N * R + 4 * R * RANK_LAYOUT_CHANNELS,
    }


def source_hash(*names) -> str:
    h = hashlib.sha1()
    for n in names:
        with open(os.path.join(ROOT, "expert_dispatch_planning_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    source is unchanged since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[workload][kernel]
        if e.get("source_sha") != source_hash(*e["sources"]):
            return None
        return int(e["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open(os.path.join("/tmp", "moe_clocks_%d.csv" % os.getpid()), "w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.out.flush()
        self.out.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        self.out.close()
        try:
            os.remove(self.out.name)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle
def oracle_step(w, inp, n_tokens: int):
    import oracle
    logits = inp["logits"][:n_tokens]
    x = inp["x_bits"][:n_tokens]
    idx, wt = oracle.route_topk(logits, w.K, scoring=w.scoring, renormalize=w.renormalize, bias=inp["bias"],
                                n_group=w.n_group, topk_group=w.topk_group, routed_scaling=w.routed_scaling)
    p = oracle.plan(idx, w.E, w.R, w.alignment)
    perm = oracle.permute(x, p["dst"], p["zero_fill_ranges"], w.K, p["P_cap"])
    oracle.combine(perm, wt.astype(np.float32), p["dst"])


def oracle_sample_tokens(w) -> int:
    # about 0.5-1 s of single-core work per step on a server core
    return min(w.N, max(256, int(2.0e8 // (w.K * w.H + 1))))


def host_cpu():
    """nproc and the CPU model of this host (for the oracle's timing)."""
    model = platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip().lower() in ("model name", "cpu part") and v.strip():
                    model = "%s (%s %s)" % (platform.machine(), k.strip(), v.strip())
                    break
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu": model}


def cpu_baseline(w, inp, min_seconds=10.0, max_steps=40):
    n = oracle_sample_tokens(w)
    oracle_step(w, inp, n)   # warm (builds/loads the library)
    t0 = time.perf_counter()
    steps = 0
    while steps < max_steps and (steps < 2 or time.perf_counter() - t0 < min_seconds):
        oracle_step(w, inp, n)
        steps += 1
    dt = time.perf_counter() - t0
    return {"value": n * steps / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": "%d full oracle steps (route+plan+permute+combine) on the first %d of %d tokens "
                      "of the %s workload, single-threaded C" % (steps, n, w.N, w.name),
            "seconds": round(dt, 2), "host": host_cpu()}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    n_ranks = ws
    if ws > 1:
        # the ranks meet once (gloo, CPU) so that rank 0 reports the world it
        # ran in; only rank 0 then times the oracle
        import torch
        import torch.distributed as dist
        dist.init_process_group("gloo")
        t = torch.ones(1)
        dist.all_reduce(t)
        n_ranks = int(t.item())
        dist.destroy_process_group()
    if rank != 0:
        return 0
    inp = workloads.make_inputs(w, seed=0)
    n = oracle_sample_tokens(w)
    for _ in range(args.warmup):
        oracle_step(w, inp, n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, inp, n)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": n_ranks,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "first %d of %d tokens per step, single-threaded C oracle" % (n, w.N),
                         "sample_tokens": n, "host": host_cpu()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def touched_bytes(w, P: int) -> int:
    """HBM bytes one step must touch at minimum (route + permute + combine)."""
    ab = algorithmic_bytes(w, P)
    return ab["route"] + ab["permute"] + ab["combine"]


def flushes_l2(w) -> bool:
    """Workloads touching less than twice the L2 (with the fewest rows a plan
    can have, P = N*K) flush it before every timed step."""
    return touched_bytes(w, w.N * w.K) < 2 * L2_BYTES


def config_of(w):
    """The workload, identical in both arms (the driver compares the two)."""
    l2 = ("L2 flushed (256 MB memset) before each timed step, steps timed one by one"
          if flushes_l2(w) else
          "inputs larger than L2 (at least %.0f MB touched per step)" % (touched_bytes(w, w.N * w.K) / 1e6))
    return {"workload": w.describe(), "N": w.N, "E": w.E, "K": w.K, "R": w.R, "H": w.H,
            "alignment": w.alignment, "parallelism": "replicas", "l2": l2}


# ---------------------------------------------------------------- GPU arm
def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import expert_dispatch_planning_gb300 as m

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", torch.cuda.current_device())
    m.load()

    inp = workloads.make_inputs(w, seed=0)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    bias = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).to(dev)
    x = torch.from_numpy(inp["x_bits"].view(np.int16)).view(torch.bfloat16).to(dev)
    rk = dict(scoring=w.scoring, renormalize=w.renormalize, bias=bias, n_group=w.n_group,
              topk_group=w.topk_group, routed_scaling=w.routed_scaling)
    stream = torch.cuda.current_stream()
    p = m.Plan.allocate(w.N, w.E, w.K, w.R, w.alignment, device=dev)
    idx = torch.empty((w.N, w.K), dtype=torch.int32, device=dev)
    wts = torch.empty((w.N, w.K), dtype=torch.float32, device=dev)
    perm = torch.empty((p.P_cap, w.H), dtype=torch.bfloat16, device=dev)
    out = torch.empty((w.N, w.H), dtype=torch.bfloat16, device=dev)

    def step():
        # routing and plan in one call (one launch where the sizes allow)
        m.route_plan(logits, w.K, w.R, w.alignment, topk_idx=idx, topk_w=wts, out=p, **rk)
        m.permute(x, p, out=perm, early_x=True)
        m.combine(perm, wts, p, out=out)

    for _ in range(max(3, args.warmup)):
        step()
    launches_per_step = 2 + m.route_plan_launches(w.N, w.E, w.K, w.R, w.n_group)
    torch.cuda.synchronize()
    status = m.get_status(p)
    if status != 0:
        raise RuntimeError("device status %d during warm-up" % status)
    P = int(p.cu_seqlens[-1].item())

    # ---- one step, and each stage alone (10 back-to-back calls, so that a
    # graph launch does not bound a µs-scale kernel), captured as CUDA
    # graphs: the timed region replays them, so host-side launch cost is not
    # measured
    stage_reps = 10
    # the timed steps run as graphs of up to 10 steps (as a model captures
    # many MoE layers in one graph) plus one graph per leftover step
    steps_per_graph = 10
    graph_stream = torch.cuda.Stream()
    graph_stream.wait_stream(stream)
    graphs = {}
    with torch.cuda.stream(graph_stream):
        for name, fn, reps in (("step", step, 1), ("chunk", step, steps_per_graph),
                               ("route", lambda: m.route_topk(logits, w.K, topk_idx=idx, topk_w=wts, **rk), stage_reps),
                               ("plan", lambda: m.plan(idx, w.E, w.R, w.alignment, out=p), stage_reps),
                               ("route_plan_fused", lambda: m.route_plan(logits, w.K, w.R, w.alignment,
                                                                         topk_idx=idx, topk_w=wts, out=p, **rk),
                                stage_reps),
                               # standalone: no overlap with the previous call's tail
                               ("permute", lambda: m.permute(x, p, out=perm), stage_reps),
                               ("combine", lambda: m.combine(perm, wts, p, out=out), stage_reps)):
            # the one-launch route + plan is opt-in; its graph is captured with it on
            fused = name == "route_plan_fused"
            if fused:
                os.environ["MOE_ROUTE_PLAN_FUSED"] = "1"
            fn()  # warm on the capture stream
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=graph_stream):
                for _ in range(reps):
                    fn()
            graphs[name] = g
            if fused:
                os.environ.pop("MOE_ROUTE_PLAN_FUSED", None)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def timed(g, reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    # inputs smaller than twice the 129 MB L2: flush it (a 256 MB memset)
    # before every timed step and time the steps one by one
    touched = touched_bytes(w, P)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flushes_l2(w) else None

    def timed_steps(k):
        """Exactly k steps: k // 10 replays of the 10-step graph, k % 10 of the 1-step one."""
        if flush is not None:
            total = 0.0
            for _ in range(k):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graphs["step"].replay()
                e1.record(stream)
                torch.cuda.synchronize()
                total += e0.elapsed_time(e1)
            return total
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k // steps_per_graph):
            graphs["chunk"].replay()
        for _ in range(k % steps_per_graph):
            graphs["step"].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    for _ in range(max(3, args.warmup)):
        graphs["step"].replay()
    graphs["chunk"].replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[torch.cuda.current_device()]))
    with clocks:
        barrier()
        torch.cuda.synchronize()
        local_ms = timed_steps(args.steps)  # the timed region: K steps
        barrier()
        # each kernel alone, same inputs, for its achieved bandwidth
        stage_ms = {k: timed(graphs[k], args.steps) / (args.steps * stage_reps)
                    for k in ("route", "plan", "route_plan_fused", "permute", "combine")}
    ms = reduce_max(local_ms)
    assert m.get_status(p) == 0

    # ---- end to end through host buffers (pinned), copies inside the
    # region: a two-deep pipeline as a serving loop runs it -- step i's
    # host->device copies (copy stream) overlap step i-1's kernels (compute
    # stream) and step i-2's device->host copy (second copy stream); inputs
    # and outputs are double-buffered on both sides, and every step copies
    # its own inputs in and its own result out
    h_logits = [torch.from_numpy(inp["logits"]).pin_memory() for _ in range(2)]
    h_x = [torch.from_numpy(inp["x_bits"].view(np.int16)).view(torch.bfloat16).pin_memory() for _ in range(2)]
    h_out = [torch.empty((w.N, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    d_logits = [torch.empty_like(logits) for _ in range(2)]
    d_x = [torch.empty_like(x) for _ in range(2)]
    d_out = [torch.empty_like(out) for _ in range(2)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "used", "done", "out")}

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev["used"][b])        # step i-2 has consumed buffer b
            d_logits[b].copy_(h_logits[b], non_blocking=True)
            d_x[b].copy_(h_x[b], non_blocking=True)
            ev["in"][b].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(ev["in"][b])
            if i >= 2:
                s_cmp.wait_event(ev["out"][b])       # step i-2's result has left d_out[b]
            m.route_plan(d_logits[b], w.K, w.R, w.alignment, topk_idx=idx, topk_w=wts, out=p, **rk)
            m.permute(d_x[b], p, out=perm, early_x=True)
            ev["used"][b].record(s_cmp)
            m.combine(perm, wts, p, out=d_out[b])
            ev["done"][b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["done"][b])
            h_out[b].copy_(d_out[b], non_blocking=True)
            ev["out"][b].record(s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    e_steps = max(6, args.steps)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(e_steps):
        e2e_step(i)
    e1.record(s_out)          # s_out's last copy ends the region (it waits on every earlier stage)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1)) / e_steps
    if m.get_status(p) != 0:
        raise RuntimeError("device status during the end-to-end run")
    barrier()

    if rank != 0:
        if dist.is_initialized():
            dist.destroy_process_group()
        return 0

    cpu = cpu_baseline(w, inp) if ws == 1 and not args.no_cpu_baseline else None
    ms_step = ms / args.steps
    value = ws * w.N / (ms_step * 1e-3)
    ab = algorithmic_bytes(w, P)
    peak, peak_kind = measured_peaks()
    dom = "permute" if stage_ms["permute"] >= stage_ms["combine"] else "combine"
    achieved = ab[dom] / (stage_ms[dom] * 1e-3) / 1e9
    kernels = {k: {"ms": round(stage_ms[k], 5),
                   "gbs": round((ab[k] if k in ab else ab["plan_count"] + ab["plan_scatter"])
                                / (stage_ms[k] * 1e-3) / 1e9, 1)}
               for k in stage_ms}
    rp_ms = stage_ms["route"] + stage_ms["plan"]
    rp_bytes = ab["route"] + ab["plan_count"] + ab["plan_scatter"]
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w),
        "method": {"P": P, "touched_mb_per_step": round(touched / 1e6, 1),
                   "experts": "identity (combine reads the permuted rows)",
                   "launch": "CUDA graphs of 10 steps (and of 1 step for K mod 10)"
                   if flush is None else "CUDA graph of one step per timed step",
                   "permute": "early_x: x row loads overlap the plan kernel"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "traffic": committed_traffic(dom, w.name),
                     "algorithmic_bytes": ab[dom]},
        "kernels": kernels,
        "route_plan_us": round(1e3 * rp_ms, 2),
        "route_plan": {"us": round(1e3 * rp_ms, 2), "algorithmic_bytes": rp_bytes,
                       "gbs": round(rp_bytes / (rp_ms * 1e-3) / 1e9, 1),
                       "frac": round(rp_bytes / (rp_ms * 1e-3) / 1e9 / peak, 4),
                       "launches": m.route_plan_launches(w.N, w.E, w.K, w.R, w.n_group),
                       "how": "route and plan each timed alone (graphs of 10 back-to-back calls), summed"},
        "route_plan_launches": m.route_plan_launches(w.N, w.E, w.K, w.R, w.n_group),
        "cpu_baseline": cpu,
        "e2e": {"value": ws * w.N / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h_logits[0].numel() * 4 + h_x[0].numel() * 2),
                "d2h_bytes_per_step": int(h_out[0].numel() * 2), "ms_per_step": e2e_ms,
                "method": "two-deep pipeline: H2D, kernels and D2H on three streams, double-buffered"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist.is_initialized():
        dist.destroy_process_group()
    return 0


def run_stage(args, w):
    """Time one stage alone: inputs resident, K replays of a graph of 10 back-to-back calls."""
    import torch

    import expert_dispatch_planning_gb300 as m
    m.load()
    dev = torch.device("cuda", 0)
    inp = workloads.make_inputs(w, seed=0, with_x=args.stage in ("permute", "combine"))
    logits = torch.from_numpy(inp["logits"]).to(dev)
    bias = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).to(dev)
    rk = dict(scoring=w.scoring, renormalize=w.renormalize, bias=bias, n_group=w.n_group,
              topk_group=w.topk_group, routed_scaling=w.routed_scaling)
    idx, wts = m.route_topk(logits, w.K, **rk)
    p = m.plan(idx, w.E, w.R, w.alignment)
    fns = {"route": lambda: m.route_topk(logits, w.K, topk_idx=idx, topk_w=wts, **rk),
           "plan": lambda: m.plan(idx, w.E, w.R, w.alignment, out=p)}
    if args.stage == "balanced":
        # a capacity of 90% of the even share, B redundant experts per rank
        cap = int(w.N * w.K / w.R * 0.9)
        nvs = w.N * w.K + (w.E + BALANCED_B) * (w.alignment - 1)
        bp = m.plan_balanced(idx, p, w.alignment, cap, BALANCED_B, nvs)
        fns["balanced"] = lambda: m.plan_balanced(idx, p, w.alignment, cap, BALANCED_B, nvs, out=bp)
    if args.stage == "tile_map":
        tmax = max(1, p.P_cap // p.alignment)
        tout = (torch.empty(tmax, dtype=torch.int32, device=dev), torch.empty(tmax, dtype=torch.int32, device=dev),
                torch.empty(2, dtype=torch.int32, device=dev))
        fns["tile_map"] = lambda: m.tile_map(p, out=tout)
    if args.stage == "rank_layout":
        lws = m.rank_layout_workspace(w.N, w.R)
        lout = m.rank_layout(p, RANK_LAYOUT_CHANNELS, workspace=lws)
        fns["rank_layout"] = lambda: m.rank_layout(p, RANK_LAYOUT_CHANNELS, workspace=lws, out=lout)
    if args.stage in ("permute", "combine"):
        x = torch.from_numpy(inp["x_bits"].view(np.int16)).view(torch.bfloat16).to(dev)
        perm = m.permute(x, p)
        out = torch.empty_like(x)
        fns["permute"] = lambda: m.permute(x, p, out=perm)
        fns["combine"] = lambda: m.combine(perm, wts, p, out=out)
    fn = fns[args.stage]
    reps = 10  # calls per captured graph, so that graph launches do not bound µs-scale kernels
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        fn()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            for _ in range(reps):
                fn()
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(args.steps):
        g.replay()
    ev[1].record()
    torch.cuda.synchronize()
    assert m.get_status(p) == 0
    ms = ev[0].elapsed_time(ev[1]) / (args.steps * reps)
    P = int(p.cu_seqlens[-1].item())
    ab = algorithmic_bytes(w, P)
    nbytes = ab[args.stage] if args.stage in ab else ab["plan_count"] + ab["plan_scatter"]
    print(json.dumps({"stage": args.stage, "workload": w.describe(), "us_per_launch": 1e3 * ms,
                      "algorithmic_bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9}), flush=True)
    return 0


def launch_ranks(n: int, argv) -> int:
    """Start n ranks of this script on this node (torch.distributed.run,
    rendezvous on 127.0.0.1) and return the launcher's exit code."""
    import socket
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + list(argv)
    return subprocess.run(cmd).returncode


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="large", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stage", choices=["all", "route", "plan", "permute", "combine", "balanced", "tile_map",
                                        "rank_layout"], default="all",
                    help="time one step of the path alone (a profiling case, not a contract line)")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's token count N")
    return ap


def main(argv=None):
    ap = build_parser()
    args = ap.parse_args(argv)
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.stage == "all":
        if "WORLD_SIZE" not in os.environ and args.gpus > 1:
            return launch_ranks(args.gpus, sys.argv[1:] if argv is None else list(argv))
        ws = dist_env()[0]
        if ws != args.gpus:
            ap.error("--gpus %d but WORLD_SIZE=%d: launch one rank per GPU" % (args.gpus, ws))
    w = workloads.get(args.config)
    if args.tokens > 0:
        import dataclasses
        w = dataclasses.replace(w, N=args.tokens)
    if args.stage != "all":
        return run_stage(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())

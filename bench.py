"""Benchmark: MoE FusedDispatch + FusedCombine on one GB300 (per rank).

One step = one pass of the whole hot path over one batch: moe_plan (top-k,
gates, replica map, histogram, scan, slots) -> moe_dispatch (INT8 quantize +
scatter into k expert slots) -> moe_combine (gate-weighted gather-reduce),
at 4096 tokens x hidden 7168, 256 experts + 32 redundant replicas (288
physical), top-8.  Expert outputs are synthetic bf16 rows resident in the
pool's combine buffers.  Step i uses buffer set i mod 2.

Phases:
  A  300 steps serialized on one stream with CUDA events around every call:
     per-call latencies (median, p10, p90; each includes its launch gap).
  A1 50 back-to-back launches of dispatch, then of combine, on one stream
     (PDL-chained, buffer sets alternating): kernel durations without launch
     gaps; combine's gives the roofline's achieved bandwidth.
  A2 plan, plan+dispatch and combine each captured as a CUDA graph and
     replayed 200 times: median, p10, p90 per op.
  B  the K timed steps (the JSON `value`): the two buffer sets on two streams,
     so step i+1's plan overlaps step i's bandwidth-bound kernels.
  C  e2e: moe_step_host from pinned host buffers -- logits and x copied in,
     plan, dispatch, identity experts (the device stand-in for the expert
     FFNs), combine, y copied out -- on a pool of three sets and three
     streams (copies in, kernels and copy out of different steps overlap).
  D  decode latency: the 96-token decode batch (hidden 7168, 256 experts,
     top-8): plan+dispatch, combine, and the whole layer each captured in a
     CUDA graph and replayed from an idle GPU; median of the replays.

Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the only other implementation of this
path) on the host cores, on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from combine_moe_plan_gb300 import workloads as wl  # noqa: E402

FALLBACK_HBM_GBS = 6800.0


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.BENCH_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer pass (profiling runs)")
    ap.add_argument("--ep-ranks", type=int, default=8,
                    help="ranks of the expert-parallel split emulated on this GPU (0: skip that phase)")
    ap.add_argument("--ep-only", action="store_true",
                    help="run only the emulated split (profiling: with --ep-tokens, a case of a few GB)")
    ap.add_argument("--ep-tokens", type=int, default=0, help="tokens per rank of the split (0: the workload's)")
    ap.add_argument("--ep-unit-rows", type=int, default=0,
                    help="rows per transfer unit of the split (0: the emulated group's default)")
    return ap.parse_args()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    return FALLBACK_HBM_GBS, "fallback (earlier GB300 copy measurement)"


CSRC = os.path.join(ROOT, "combine_moe_plan_gb300", "csrc")


def source_closure(kernel_file: str) -> list:
    """The kernel's source file and every csrc file it includes with
    #include "...", transitively, sorted by name."""
    seen, todo = set(), [kernel_file]
    while todo:
        f = todo.pop()
        if f in seen or not os.path.exists(os.path.join(CSRC, f)):
            continue
        seen.add(f)
        for line in open(os.path.join(CSRC, f), encoding="utf-8"):
            m = re.match(r'\s*#\s*include\s+"([^"]+)"', line)
            if m:
                todo.append(m.group(1))
    return sorted(seen)


def source_hash(kernel_file: str) -> str:
    """sha256 over (name, contents) of the kernel's source closure."""
    h = hashlib.sha256()
    for f in source_closure(kernel_file):
        h.update(f.encode() + b"\0")
        h.update(open(os.path.join(CSRC, f), "rb").read())
    return h.hexdigest()


def l2_note(step_bytes: int, l2_bytes: int) -> str:
    """How the timed steps stand to L2: no flush is done, so a step's bytes
    must exceed L2 for the figures to be DRAM figures."""
    if step_bytes > l2_bytes:
        return (f"inputs larger than L2 (about {step_bytes / 1e9:.2f} GB touched per step against "
                f"{l2_bytes / 1e6:.0f} MB of L2; two buffer sets alternate); no flush")
    return (f"inputs fit in L2 ({step_bytes / 1e6:.1f} MB touched per step against {l2_bytes / 1e6:.0f} MB); "
            f"no flush: timed L2-warm, as consecutive small batches run; a latency figure, not a DRAM one")


def _traffic(kernel_file: str, kernel: str, workload: str):
    """Per-launch DRAM bytes from a committed ncu summary: only for the
    workload it was captured on, and only if the kernel's source (with
    everything it includes) has not changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    d = rec.get(kernel)
    if not d or rec.get("workload") != workload or source_hash(kernel_file) != d.get("source_sha256"):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clocks(out)


def parse_clocks(out: str):
    """Summary of nvidia-smi samples in ClockSampler.Q's column order
    (csv, noheader, nounits): the median SM clock under load (samples above
    half the largest), the largest max clock, every throttle reason seen
    Active, and the sample count; None without samples."""
    rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 9]
    if not rows:
        return None
    sm = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
    mx = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.strip() == "Active"})
    # samples under load: SM clock above the idle floor
    load = [s for s in sm if s > 0.5 * (max(sm) if sm else 1)]
    return {"sm_mhz": statistics.median(load) if load else None,
            "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(vals, device=None):
    """Element-wise max of per-rank timings (ms) over all ranks; identity
    when not distributed.  The reported time of a multi-rank run is the
    slowest rank's."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _percentiles_us(ms_list) -> list:
    """p10, median and p90 of a list of event times in ms, in microseconds."""
    v = np.sort(np.asarray(ms_list, np.float64)) * 1e3
    return [float(np.percentile(v, q)) for q in (10, 50, 90)]


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_step_fn(w: wl.Workload, inp: dict):
    """A function running the oracle over tokens [a, b) of the workload."""
    import oracle
    oracle.build()

    def run(a, b):
        ex = inp["ex_out"][: (b - a) * w.k] if "ex_out" in inp else None
        oracle.forward(inp["logits"][a:b], inp["x"][a:b], w.k, inp["rep_off"], inp["rep_ids"], w.P, ex_out=ex)
    return run


def _oracle_threads(n: int) -> int:
    import oracle
    return oracle.set_threads(n)


def _time_oracle(run, T: int, budget_s: float, max_reps: int):
    """Whole batches while they fit the budget, else a token prefix."""
    t0 = time.perf_counter()
    run(0, min(T, 64))
    per_tok = (time.perf_counter() - t0) / min(T, 64)
    n_tok = int(max(min(T, 64), min(T, budget_s / max(per_tok, 1e-9))))
    reps = max(1, min(max_reps, int(budget_s / (per_tok * n_tok))))
    t0 = time.perf_counter()
    for _ in range(reps):
        run(0, n_tok)
    return reps, n_tok, time.perf_counter() - t0


def cpu_baseline(w: wl.Workload, inp: dict, budget_s: float = 12.0) -> dict:
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload: once with its per-token loops on every core (the reported
    value), once on a single thread.  The outputs of the two are identical."""
    run = _oracle_step_fn(w, inp)
    n_thr = _oracle_threads(_host_cores())
    reps, n_tok, dt = _time_oracle(run, w.T, budget_s, 200)
    _oracle_threads(1)
    reps1, n_tok1, dt1 = _time_oracle(run, w.T, budget_s, 30)
    _oracle_threads(n_thr)
    return {"value": reps * n_tok / dt, "unit": "tokens/s", "cores": n_thr, "kind": "oracle",
            "sample": f"{reps} x the first {n_tok} tokens of {w.name} (plan+dispatch+combine, "
                      f"per-token loops on {n_thr} threads, counting sort serial)",
            "single_thread": {"value": reps1 * n_tok1 / dt1, "cores": 1,
                              "sample": f"{reps1} x the first {n_tok1} tokens"}}


def run_reference(a, w: wl.Workload):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    inp = wl.make_inputs(w)
    run = _oracle_step_fn(w, inp)
    n_thr = _oracle_threads(_host_cores())
    t0 = time.perf_counter()
    run(0, 64)
    per_tok = (time.perf_counter() - t0) / 64
    budget = 90.0  # seconds for warmup + timed steps; at least 64 tokens per step
    n_tok = int(max(min(64, w.T), min(w.T, budget / max(1, a.steps + a.warmup) / max(per_tok, 1e-9))))
    for _ in range(a.warmup):
        run(0, n_tok)
    t0 = time.perf_counter()
    for _ in range(a.steps):
        run(0, n_tok)
    dt = time.perf_counter() - t0
    v = a.steps * n_tok / dt
    sample = (f"first {n_tok} tokens of {w.name} per step (plan+dispatch+combine, "
              f"per-token loops on {n_thr} threads)")
    print(json.dumps({
        "impl": "reference", "metric": "dispatch+combine tokens/s (plan+dispatch+combine per step)",
        "value": v, "unit": "tokens/s", "n_gpus": ws, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": dt / a.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8+bf16", "data": w.describe(),
        "config": {"workload": w.name, "tokens_per_step": n_tok, "H": w.H, "E": w.E, "P": w.P, "k": w.k},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": n_thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


class _Streams:
    """One stream per buffer set: step i runs on stream i mod n, so the
    latency-bound plan of step i+1 overlaps the bandwidth-bound kernels of
    step i (the micro-batch overlap the double-buffered pool exists for).
    Each stream only ever touches its own set, so stream order alone keeps
    every set's plan -> dispatch -> combine -> next plan sequence intact."""

    def __init__(self, torch, dev, n=2):
        self.torch = torch
        self.s = [torch.cuda.Stream(device=dev) for _ in range(n)]
        self.main = torch.cuda.current_stream()

    def fork(self):
        e = self.torch.cuda.Event()
        e.record(self.main)
        for s in self.s:
            s.wait_event(e)

    def join(self):
        for s in self.s:
            e = self.torch.cuda.Event()
            e.record(s)
            self.main.wait_event(e)


def _graph_per_op(torch, pool, logits, rep_off, rep_ids, x, y, T, reps=200, warm=10) -> dict:
    """Each op of one step on buffer set 0 captured as its own CUDA graph and
    replayed `reps` times after `warm` untimed replays: GPU time per replay
    (CUDA events around it) as [p10, median, p90] in microseconds.
    "plan+dispatch" is one graph of both: the routing metadata belongs to the
    fused dispatch."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pool.plan_dispatch(logits, x, rep_off, rep_ids, buf=0, stream=s)
        pool.combine(T, y=y, buf=0, stream=s)
    torch.cuda.synchronize()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        return g

    graphs = {
        "plan": capture(lambda: pool.plan(logits, rep_off, rep_ids, buf=0, stream=s)),
        "plan+dispatch": capture(lambda: pool.plan_dispatch(logits, x, rep_off, rep_ids, buf=0, stream=s)),
        "combine": capture(lambda: pool.combine(T, y=y, buf=0, stream=s)),
    }
    torch.cuda.synchronize()
    out = {}
    for name, g in graphs.items():
        for _ in range(warm):
            g.replay()
        ts = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        out[name] = _percentiles_us(ts)
    return out


def decode_latency(dev, reps=200):
    """GPU time (median, with p10 and p90) of plan+dispatch (the routing
    metadata is part of the fused dispatch) and of combine, each replayed as
    a CUDA graph, and of the whole layer, for the 96-token decode batch."""
    import torch
    from combine_moe_plan_gb300 import moe
    w = wl.WORKLOADS["t96_h7168_e256_k8"]
    inp = wl.make_inputs(w)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2, device=dev)
    for b in range(2):
        pool.view(b)["ex_out"][: w.rows].copy_(torch.from_numpy(inp["ex_out"].view(np.int16)).view(torch.bfloat16))
    y = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(device=dev)
    # Consecutive layers of one decode step: each layer its own router
    # logits, its y the next layer's x, the two buffer sets alternating.
    n_chain = 16
    chain_logits = [torch.from_numpy(wl.make_inputs(w, seed=100 + l, with_expert_out=False)["logits"]).to(dev)
                    for l in range(n_chain)]
    chain_y = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev) for _ in range(n_chain)]

    def chain(parts="layer"):
        """16 consecutive layers: the whole layer, or only its plan, or its
        plan and dispatch (what each part adds inside a chain)."""
        xin = x
        for l in range(n_chain):
            if parts == "plan":
                pool.plan(chain_logits[l], buf=l & 1, stream=s)
                continue
            pool.plan_dispatch(chain_logits[l], xin, buf=l & 1, stream=s)
            if parts == "plan+dispatch":
                continue
            pool.combine(w.T, y=chain_y[l], buf=l & 1, stream=s)
            xin = chain_y[l]

    with torch.cuda.stream(s):
        for _ in range(3):
            pool.plan_dispatch(logits, x, stream=s)
            pool.combine(w.T, y=y, stream=s)
        chain()
    torch.cuda.synchronize()
    g_disp, g_comb, g_layer = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_disp, stream=s):
        pool.plan_dispatch(logits, x, stream=s)
    with torch.cuda.graph(g_comb, stream=s):
        pool.combine(w.T, y=y, stream=s)
    with torch.cuda.graph(g_layer, stream=s):
        pool.plan_dispatch(logits, x, stream=s)
        pool.combine(w.T, y=y, stream=s)
    g_chain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_chain, stream=s):
        chain()
    g_parts = {}
    for parts in ("plan", "plan+dispatch"):
        with torch.cuda.stream(s):
            chain(parts)
        torch.cuda.synchronize()
        g_parts[parts] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_parts[parts], stream=s):
            chain(parts)
    torch.cuda.synchronize()

    def med(fn):
        ts = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        return _percentiles_us(ts)

    pct = {"dispatch": med(g_disp.replay), "combine": med(g_comb.replay), "layer": med(g_layer.replay)}

    def queued(fn, n=100, spin=100000):
        """GPU time of one replay whose launch the host has already queued: a
        spin kernel (about 50 us by default; 20 us proved too short for the
        host to enqueue e0, the graph and e1 every time) holds the stream
        while they are enqueued, so the interval excludes the host's launch
        latency."""
        ts = []
        for _ in range(n):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(spin)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        # Event timestamps here tick in steps of about 1 us, so the median
        # sits on a step; the mean over the replays resolves finer.
        return _percentiles_us(ts) + [float(np.mean(ts)) * 1e3]

    def back_to_back(fn, n=200):
        """Mean GPU time per replay over n replays queued back to back."""
        for _ in range(3):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    layer_q = queued(g_layer.replay)
    chain_q = queued(g_chain.replay, n=50, spin=200000)
    parts_q = {k: queued(g.replay, n=50, spin=200000)[3] / n_chain for k, g in g_parts.items()}
    # The floor of a graph of three kernels that do nothing (torch adds on 16
    # floats), queued the same way: what any three-kernel graph costs.
    tiny = torch.zeros(16, device=dev)
    g_empty = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_empty, stream=s):
        for _ in range(3):
            tiny.add_(1.0)
    torch.cuda.synchronize()
    empty_q = queued(g_empty.replay)
    out = {"workload": w.name, "dispatch_us": pct["dispatch"][1], "combine_us": pct["combine"][1],
           "layer_us": pct["layer"][1], "p10_p50_p90_us": pct,
           "layer_queued_us": layer_q[1], "layer_queued_p10_p50_p90_us": layer_q[:3],
           "layer_queued_mean_us": layer_q[3],
           "layer_back_to_back_us": back_to_back(g_layer.replay),
           "empty_three_kernel_graph_queued_us": empty_q[1],
           "empty_three_kernel_graph_queued_mean_us": empty_q[3],
           "layer_in_16_layer_graph_us": chain_q[3] / n_chain,
           "parts_in_16_layer_graph_us": {"plan": parts_q["plan"], "plan+dispatch": parts_q["plan+dispatch"],
                                          "plan+dispatch+combine": chain_q[3] / n_chain},
           "note": "CUDA-graph replays from an idle GPU; dispatch = plan + dispatch (the fused "
                   "dispatch carries the routing metadata); each graph launch adds its own overhead. "
                   "layer_queued: the same layer graph with its launch already queued behind a spin "
                   "kernel (the host's launch latency excluded); layer_back_to_back: mean per replay "
                   "of 200 replays queued back to back (consecutive layers); empty_three_kernel_graph: "
                   "a graph of three do-nothing kernels queued the same way (the graph's own cost); "
                   "layer_in_16_layer_graph: one replay of 16 consecutive layers (each its own logits, "
                   "its y the next layer's x) captured as one graph and queued the same way, mean over 50 "
                   "replays divided by 16; parts_in_16_layer_graph: the same chain of the plans alone and of "
                   "the plans and dispatches, per layer. Event timestamps tick in steps of about 1 us: the "
                   "medians sit on steps, the means resolve finer"}
    if pool.check() != 0:
        raise RuntimeError("device error word set in the decode-latency pass")
    return out


def run_ours(a, w: wl.Workload):
    import torch
    import torch.distributed as dist

    from combine_moe_plan_gb300 import build as moe_build
    from combine_moe_plan_gb300 import moe

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    moe_build.build()
    moe.lib()

    # ---- inputs (seed = rank: each rank its own batch; weak scaling) ----
    inp = wl.make_inputs(w, seed=rank)
    if "ex_out" not in inp:  # identity-expert workloads: the timed combine still reads bf16 rows
        inp["ex_out"] = wl.make_expert_out(w, seed=rank)
    dev = torch.device("cuda", local)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    ex_dev = torch.from_numpy(inp["ex_out"].view(np.int16)).view(torch.bfloat16).to(dev)
    rep_off = None if inp["rep_off"] is None else torch.from_numpy(inp["rep_off"]).to(dev)
    rep_ids = None if inp["rep_ids"] is None else torch.from_numpy(inp["rep_ids"]).to(dev)
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2, device=dev)
    for b in range(2):
        pool.view(b)["ex_out"][: w.rows].copy_(ex_dev)
    del ex_dev
    ys = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    st = _Streams(torch, dev)

    def step(i, stream, ev=None):
        b = i & 1
        if ev is None:
            pool.plan_dispatch(logits, x, rep_off, rep_ids, buf=b, stream=stream)
        else:  # the same two kernels with events between them
            ev[0].record(stream)
            pool.plan(logits, rep_off, rep_ids, buf=b, stream=stream)
            ev[1].record(stream)
            # the plan is the kernel just before and x is never written here
            pool.dispatch(x, buf=b, stream=stream, after_plan=True)
            ev[2].record(stream)
        pool.combine(w.T, y=ys[b], buf=b, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    def pipelined(n, i0=0):
        st.fork()
        for i in range(i0, i0 + n):
            step(i, st.s[i & 1])
        st.join()

    pipelined(a.warmup)
    torch.cuda.synchronize()
    if pool.check() != 0:
        raise RuntimeError("device error word set during warm-up")

    # ---- phase A: serialized steps on one stream, per-kernel CUDA events ----
    n_lat = min(a.steps, 300)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_lat)]
    for i in range(n_lat):
        step(i, st.main, evs[i])
    torch.cuda.synchronize()
    per = {"plan": [], "dispatch": [], "combine": [], "step": []}
    for e in evs:
        per["plan"].append(e[0].elapsed_time(e[1]))
        per["dispatch"].append(e[1].elapsed_time(e[2]))
        per["combine"].append(e[2].elapsed_time(e[3]))
        per["step"].append(e[0].elapsed_time(e[3]))
    per_us = {k: 1e3 * statistics.median(v) for k, v in per.items()}
    per_pct = {k: _percentiles_us(v) for k, v in per.items()}

    # ---- phase A1: kernel durations without launch gaps: back-to-back
    # launches on one stream (each waits on the previous through PDL, no event
    # between them), the two buffer sets alternating so that 0.94 GB of expert
    # rows (far more than L2) are read; CUDA events around the whole batch.
    n_b2b = 50
    b2b_us = {}
    for name, launch in (("dispatch", lambda i: pool.dispatch(x, buf=i & 1, stream=st.main)),
                         ("combine", lambda i: pool.combine(w.T, y=ys[i & 1], buf=i & 1, stream=st.main))):
        for i in range(4):
            launch(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st.main)
        for i in range(n_b2b):
            launch(i)
        e1.record(st.main)
        torch.cuda.synchronize()
        b2b_us[name] = e0.elapsed_time(e1) * 1e3 / n_b2b

    # ---- phase A2: each op of a step replayed as a CUDA graph ----
    graph_us = _graph_per_op(torch, pool, logits, rep_off, rep_ids, x, ys[0], w.T)
    if pool.check() != 0:
        raise RuntimeError("device error word set during the graph replays")

    # ---- phase B (timed region): K steps, the two buffer sets on two streams ----
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    time.sleep(0.3)  # nvidia-smi's first samples
    # The GPU idled during the sleep: the W warm-up steps run again right
    # before the timed region, so that it starts on a busy GPU.
    pipelined(a.warmup)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = pool.launches()
    t_start.record(st.main)
    pipelined(a.steps, a.warmup)
    t_end.record(st.main)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop()
    n_steps = a.steps
    launches = pool.launches() - launches0
    ms = t_start.elapsed_time(t_end) / n_steps
    err = pool.check()
    if err != 0:
        raise RuntimeError(f"device error word {err:#x}")

    # ---- phase B2 (not the reported value): the same schedule over 2000
    # steps, where filling and draining the two-stream pipeline is amortized;
    # set against ms_per_step it shows what a short timed run adds.
    n_long = 2000
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st.main)
    pipelined(n_long, a.warmup + a.steps)
    e1.record(st.main)
    torch.cuda.synchronize()
    steady_us = e0.elapsed_time(e1) * 1e3 / n_long

    # ---- phase C: e2e through moe_step_host from pinned host buffers ----
    e2e_ms = float("nan")
    if not a.no_e2e:
        del pool, ys
        torch.cuda.empty_cache()
        e2e_ms = _e2e(a, w, inp, rep_off, rep_ids, dev, ws)

    # ---- phase D: decode-batch latency (CUDA graphs) ----
    decode = None if a.no_e2e else decode_latency(dev)

    # ---- phase E: the expert-parallel split, R ranks emulated on this GPU ----
    split = split_decode = None
    if a.ep_ranks > 0 and ws == 1 and not a.no_e2e:
        torch.cuda.empty_cache()
        split = ep_split(dev, w, a.ep_ranks)
        # the decode batch split the same way (one local batch of 96 tokens per rank)
        split_decode = ep_split(dev, wl.WORKLOADS["t96_h7168_e256_k8"], a.ep_ranks, reps=100)

    # ---- max over ranks ----
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], device=dev)
    if rank == 0:
        bytes_ = w.algorithmic_bytes()
        peak, peak_src = _peaks()
        achieved = bytes_["combine"] / (b2b_us["combine"] * 1e-6) / 1e9
        traffic = _traffic("combine.cu", "combine_kernel", w.name)
        tokens = w.T * ws
        out = {
            "metric": "dispatch+combine tokens/s (plan+dispatch+combine per step)",
            "value": tokens / (ms * 1e-3), "unit": "tokens/s", "n_gpus": ws, "steps": n_steps,
            "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8+bf16 (fp32 accumulate)",
            "data": w.describe(),
            "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "P": w.P, "k": w.k,
                       "group": w.group, "parallelism": f"replicas x{ws}",
                       "schedule": "two buffer sets on two streams (step i on set/stream i mod 2)",
                       "l2": l2_note(bytes_["total"],
                                     getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)
                                     or 129 * 10**6)},
            "us_per_call": {"plan": per_us["plan"], "dispatch": per_us["dispatch"],
                            "combine": per_us["combine"], "step_serialized": per_us["step"],
                            "step_pipelined": ms * 1e3, "step_pipelined_2000_steps": steady_us},
            "us_per_call_p10_p50_p90": {"plan": per_pct["plan"], "dispatch": per_pct["dispatch"],
                                        "combine": per_pct["combine"], "step_serialized": per_pct["step"]},
            "graph_replay_us_p10_p50_p90": graph_us,
            "kernel_us_back_to_back": b2b_us,
            "hbm_gbs": {"step": bytes_["total"] / (ms * 1e-3) / 1e9,
                        "step_serialized": bytes_["total"] / (per_us["step"] * 1e-6) / 1e9,
                        "dispatch": bytes_["dispatch"] / (per_us["dispatch"] * 1e-6) / 1e9,
                        "combine": bytes_["combine"] / (per_us["combine"] * 1e-6) / 1e9,
                        "step_frac_of_peak": bytes_["total"] / (ms * 1e-3) / 1e9 / peak},
            "algorithmic_bytes": bytes_,
            "roofline": {"kernel": "combine_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_src, "duration_us": b2b_us["combine"],
                         "achieved_counts": "algorithmic bytes (every expert row read once, y written once) "
                                            "per launch / mean launch duration",
                         "dram_gbs": None if traffic is None else traffic / (b2b_us["combine"] * 1e-6) / 1e9,
                         "dram_frac": None if traffic is None else traffic / (b2b_us["combine"] * 1e-6) / 1e9 / peak,
                         "dram_note": "ncu dram__bytes_read+write of one serialized launch over the same "
                                      "duration; part of y is still dirty in L2 when a launch ends under ncu "
                                      "and is written back during the next kernel, so this understates the "
                                      "steady-state DRAM traffic",
                         "duration": f"mean of {n_b2b} back-to-back launches on one stream (PDL-chained, "
                                     "buffer sets alternating: 0.94 GB of expert rows per pair), CUDA events "
                                     "around the batch"},
            "e2e": None if a.no_e2e else {
                "value": w.T * ws / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(inp["logits"].nbytes + inp["x"].nbytes),
                "d2h_bytes_per_step": int(w.T * w.H * 2), "ms_per_step": e2e_ms,
                "path": "moe_step_host: logits+x host->device, plan, dispatch, identity experts (device "
                        "stand-in for the expert FFNs), combine, y device->host; three sets on three streams"},
            "gpu_launches": int(launches),
            "clocks": clocks,
            "decode_latency": decode,
            "ep_split_emulated": split,
            "ep_split_emulated_decode": split_decode,
        }
        if not a.no_cpu_baseline and ws == 1:
            out["cpu_baseline"] = cpu_baseline(w, inp)
        print(json.dumps(out), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


def ep_split(dev, w, R, reps=20, n_b2b=20, unit_rows=0):
    """The expert-parallel split of the workload over R ranks emulated on this
    GPU (each rank its own seeded batch of w.T tokens, its own pool and a
    worst-case receive buffer): per step every rank plans and dispatches, the
    counts come to the host, libmoe's host scheduler makes both exchanges'
    LPT schedules for all R pullers, the dispatch pull (one launch, all
    pullers), the expert outputs (synthetic bf16 rows already resident in the
    receive buffers), the combine pull, and every rank's combine; the host
    schedules while the dispatch kernels run.  Reports the
    step time (tokens of all ranks per second), the two pull kernels' mean
    durations back to back with the bytes they move (read + write) against
    the HBM copy peak, and the host scheduling time."""
    import torch
    from combine_moe_plan_gb300 import ep
    kw = {"desc_kw": {"unit_rows": (unit_rows, unit_rows)}} if unit_rows else {}
    g = ep.EmulatedGroup(R, w.T, w.H, w.E, w.P, w.k, device=dev, **kw)
    inps = [wl.make_inputs(w, seed=r, with_expert_out=False) for r in range(R)]
    logits = [torch.from_numpy(i["logits"]).to(dev) for i in inps]
    xs = [torch.from_numpy(i["x"].view(np.int16)).to(dev).view(torch.bfloat16) for i in inps]
    ro = None if inps[0]["rep_off"] is None else torch.from_numpy(inps[0]["rep_off"]).to(dev)
    ri = None if inps[0]["rep_ids"] is None else torch.from_numpy(inps[0]["rep_ids"]).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    for t in g.recv_ex:
        t.copy_(torch.randn(t.shape, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16))
    s = torch.cuda.current_stream(dev)
    sched_s = []
    ys = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev) for _ in range(R)]

    cap = [t.shape[0] for t in g.recv_ex]

    def one_step(fused):
        if fused == "all":  # fused dispatch and combine: no schedule, no pull, no host round trip
            g.plan_all(logits, ro, ri)
            starts_dev, _ = g.starts_device()
            g.dispatch_fused(xs, starts_dev)
            g.combine_fused([w.T] * R, cap, starts_dev, ys=ys, recorded=True)
            return None
        ev = g.plan_dispatch(logits, xs, ro, ri)
        counts = g.counts_host(ev)
        t0 = time.perf_counter()
        disp, comb, recv_rows = g.schedules(counts)
        starts = g.recv_starts(counts) if fused else None
        sched_s.append(time.perf_counter() - t0)
        du, dc = g.upload(disp)
        cu, cc = g.upload(comb)
        g.pull_dispatch(du, dc)
        if fused:
            g.combine_fused([w.T] * R, recv_rows, starts, ys=ys)
        else:
            g.pull_combine(cu, cc)
            g.combine([w.T] * R, ys=ys)
        return (du, dc, cu, cc, starts), recv_rows, counts

    def timed_steps(fused):
        for _ in range(3):
            one_step(fused)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        sched_s.clear()
        e0.record(s)
        for _ in range(reps):
            out = one_step(fused)
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps, 1e3 * statistics.median(sched_s) if sched_s else 0.0, out

    all_fused_ms, _, _ = timed_steps("all")
    # the same fully fused step as one CUDA graph, replayed back to back
    graph = g.fused_step_graph(logits, xs, ys, ro, ri)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(reps):
        graph.replay()
    e1.record(s)
    torch.cuda.synchronize()
    graph_ms = e0.elapsed_time(e1) / reps
    del graph
    fused_ms, _, (fused_packed, _, _) = timed_steps(True)
    starts = fused_packed[4]
    step_ms, sched_ms, (packed, recv_rows, counts) = timed_steps(False)
    starts_dev, _ = g.starts_device()

    du, dc, cu, cc, _ = packed
    b2b = {}
    for name, fn in (("dispatch_pull", lambda: g.pull_dispatch(du, dc)),
                     ("combine_pull", lambda: g.pull_combine(cu, cc)),
                     ("fused_dispatch_all_ranks", lambda: g.dispatch_fused(xs, starts_dev)),
                     ("fused_combine_all_ranks", lambda: g.combine_fused([w.T] * R, cap, starts_dev, ys=ys,
                                                                         recorded=True)),
                     ("fused_combine_rows_found_all_ranks",
                      lambda: g.combine_fused([w.T] * R, recv_rows, starts, ys=ys))):
        for _ in range(3):
            fn()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(s)
        for _ in range(n_b2b):
            fn()
        a1.record(s)
        torch.cuda.synchronize()
        b2b[name] = a0.elapsed_time(a1) * 1e3 / n_b2b
    if g.check() != 0:
        raise RuntimeError("device error word set in the split pass")
    rows = int(sum(recv_rows))
    moved = {"dispatch_pull": 2 * rows * (w.H + 4 * g.Gs), "combine_pull": 2 * rows * 2 * w.H,
             "fused_combine_all_ranks": R * w.algorithmic_bytes()["combine"],
             "fused_combine_rows_found_all_ranks": R * w.algorithmic_bytes()["combine"],
             "fused_dispatch_all_ranks": R * w.algorithmic_bytes()["dispatch"]}
    peak, peak_src = _peaks()
    out = {"ranks": R, "workload_per_rank": w.name, "cores_per_puller": g.cores,
           "desc": {"fanout_cap": list(g.desc.fanout_cap), "unit_rows": list(g.desc.unit_rows),
                    "alpha_ns": list(g.desc.alpha_ns), "beta_gbs": list(g.desc.beta_gbs)},
           "value": R * w.T / (all_fused_ms * 1e-3), "unit": "tokens/s (all ranks)", "ms_per_step": all_fused_ms,
           "form": "fully fused (below), launched from the host",
           "pulled": {"value": R * w.T / (step_ms * 1e-3), "ms_per_step": step_ms,
                      "what": "counts to the host, LPT schedules for both exchanges, the dispatch pull, the "
                              "combine pull and every rank's moe_combine"},
           "fused_combine": {"value": R * w.T / (fused_ms * 1e-3), "ms_per_step": fused_ms,
                             "what": "the combine reads each copy's row in its owner's receive buffer and "
                                     "reduces locally (moe_ep_combine), instead of the combine pull and "
                                     "moe_combine"},
           "fused": {"value": R * w.T / (all_fused_ms * 1e-3), "ms_per_step": all_fused_ms,
                     "what": "window starts on the device (moe_ep_recv_start_device), every rank's tokens "
                             "quantized and written straight into the owners' receive buffers "
                             "(moe_ep_dispatch), and the fused combine: no schedule, no pull, no host round "
                             "trip",
                     "as_one_cuda_graph": {"value": R * w.T / (graph_ms * 1e-3), "ms_per_step": graph_ms}},
           "host_schedule_ms_per_step": sched_ms,
           "rows_exchanged": rows, "kernel_us_back_to_back": b2b,
           "kernel_roofline": {k: {"bytes": moved[k], "achieved_gbs": moved[k] / (b2b[k] * 1e-6) / 1e9,
                                   "peak": peak, "frac": moved[k] / (b2b[k] * 1e-6) / 1e9 / peak}
                               for k in b2b},
           "peak_source": peak_src,
           "note": "all ranks on one GPU: both exchanges move every rank's rows through local HBM (one launch "
                   "for all pullers); the step includes the counts' device-to-host copy and the host "
                   "schedules; unmeasured across GPUs"}
    del g
    torch.cuda.empty_cache()
    return out


E2E_SETS = 3


def _e2e(a, w, inp, rep_off, rep_ids, dev, ws):
    """ms per step of moe_step_host from pinned host buffers (copies inside).
    A pool of three buffer sets on three streams: one set's host copies,
    another's kernels and a third's copy back proceed together."""
    import torch
    import torch.distributed as dist
    from combine_moe_plan_gb300 import moe
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=E2E_SETS, device=dev)
    st = _Streams(torch, dev, E2E_SETS)
    h_logits = torch.from_numpy(inp["logits"]).pin_memory()
    h_x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    h_y = [torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(E2E_SETS)]

    def run(n):
        st.fork()
        for i in range(n):
            b = i % E2E_SETS
            pool.step_host(h_logits, h_x, h_y[b], None, rep_off, rep_ids, buf=b, stream=st.s[b])
        st.join()

    run(2 * E2E_SETS)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    e0.record(st.main)
    run(a.e2e_steps)
    e1.record(st.main)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / a.e2e_steps
    # the same layer run from device-resident inputs must give the same y
    x = h_x.to(dev)
    pool.plan(h_logits.to(dev), rep_off, rep_ids, buf=0)
    pool.dispatch(x, buf=0)
    pool.identity_experts(w.T, buf=0)
    y = pool.combine(w.T, buf=0)
    torch.cuda.synchronize()
    if not all(torch.equal(h, y.cpu()) for h in h_y):
        raise RuntimeError("moe_step_host output differs from the device-resident path")
    if pool.check() != 0:
        raise RuntimeError("device error word set in the e2e pass")
    return e2e_ms


def run_ep_only(a, w):
    """Only the emulated split, printed as one JSON line (a profiling aid)."""
    import torch
    from combine_moe_plan_gb300 import build as moe_build
    from combine_moe_plan_gb300 import moe
    moe_build.build()
    moe.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if a.ep_tokens:
        w = wl.small_variant(w, a.ep_tokens)
    print(json.dumps({"ep_split_emulated": ep_split(dev, w, a.ep_ranks, reps=a.steps, unit_rows=a.ep_unit_rows)}),
          flush=True)


def main():
    a = _args()
    w = wl.WORKLOADS[a.workload]
    if a.impl == "reference":
        run_reference(a, w)
    elif a.ep_only:
        run_ep_only(a, w)
    else:
        run_ours(a, w)


if __name__ == "__main__":
    main()

"""Stage timelines from the in-kernel probes of libmoe_trace.so.

The trace build stamps, for thread 0 of every CTA, %globaltimer and clock64
at each stage boundary of each kernel (include/moe_trace.h lists the stages).
This module loads that build, runs one pass of the path on the GPU, and turns
the stamps into per-stage durations across CTAs and the span of each launch
(first CTA start to last CTA end).

    python -m combine_moe_plan_gb300.trace --workload t96_h7168_e256_k8

The probes themselves live in the kernels; nothing here computes any part of
the method.
"""
from __future__ import annotations

import argparse
import ctypes
import json

import numpy as np

from combine_moe_plan_gb300 import build as moe_build
from combine_moe_plan_gb300 import moe

TRACE_CTAS, TRACE_STAGES = 8192, 12
KINDS = {
    0: ("route_tile", ["start", "top-k", "gates(pairs)", "fallback", "replicas+masks", "counts+ranks"]),
    1: ("column_scan", ["start", "end"]),
    2: ("assign", ["start", "offsets", "end"]),
    # one plan launch: the cluster kernel (6 cluster barrier passed, 7 the other
    # tiles' masks read, 8 offsets scanned, 9 copies placed) or, without
    # clusters, the ticket kernel (6 its last CTA's tail start, 7 end)
    3: ("plan_one_launch", ["start", "top-k", "gates(pairs)", "fallback", "replicas+masks", "counts+ranks",
                            "barrier|tail", "masks read|end", "offsets", "placed"]),
    4: ("dispatch", ["start", "quantized", "slots", "stored"]),
    5: ("combine", ["start", "slots", "accumulated", "stored"]),
}


def load() -> ctypes.CDLL:
    moe_build.build()
    moe.use_library(moe_build.TRACE_LIB)
    L = moe.lib()
    L.moe_trace_reset.argtypes = [ctypes.c_void_p]
    L.moe_trace_reset.restype = ctypes.c_int
    L.moe_trace_read.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    L.moe_trace_read.restype = ctypes.c_int
    return L


def reset(stream=None) -> None:
    rc = moe.lib().moe_trace_reset(moe._stream(stream))
    if rc != 0:
        raise moe.MoeError("moe_trace_reset", rc, "")


def read(kind: int):
    """(stamps uint64 [CTAs, stages, 2] as (ns, cycles), sm uint32 [CTAs])."""
    stamps = np.zeros((TRACE_CTAS, TRACE_STAGES, 2), np.uint64)
    sm = np.zeros(TRACE_CTAS, np.uint32)
    rc = moe.lib().moe_trace_read(kind, stamps.ctypes.data_as(ctypes.c_void_p), sm.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise moe.MoeError("moe_trace_read", rc, "")
    return stamps, sm


def summarize(kind: int, n_ctas: int) -> dict:
    """Per-stage durations (ns) across the first n_ctas CTAs of the last launch
    of `kind`: median and 90th percentile of (stamp[b] - stamp[a]) over CTAs
    that reached both, for consecutive stages a, b in the order they were
    reached (by median stamp: the cluster plan computes its gates, stages 2
    and 3, after stage 5), plus the launch span and the SMs used."""
    name, stages = KINDS[kind]
    st, sm = read(kind)
    ns = st[:n_ctas, :, 0].astype(np.int64)
    ran = ns[:, 0] > 0  # the stamps are cleared before each pass
    out = {"kernel": name, "ctas": int(ran.sum()), "sms": int(len(np.unique(sm[:n_ctas][ran]))), "stages": {}}
    seen = [s for s in range(len(stages)) if (ns[:, s] > 0).any()]
    order = sorted(seen, key=lambda s: (float(np.median(ns[ns[:, s] > 0, s])), s))
    for a, b in zip(order[:-1], order[1:]):
        ok = (ns[:, b] > 0) & (ns[:, a] > 0)
        if ok.any():
            d = ns[ok, b] - ns[ok, a]
            out["stages"][f"{stages[a]}->{stages[b]}"] = {
                "median_ns": float(np.median(d)), "p90_ns": float(np.percentile(d, 90)), "ctas": int(ok.sum())}
    started = ns[:, 0][ns[:, 0] > 0]
    last = ns.max(axis=1)
    if started.size:
        out["span_ns"] = float(last.max() - started.min())
        out["cta_ns_median"] = float(np.median(last[ns[:, 0] > 0] - started))
        out["first_start_ns"] = int(started.min())  # %globaltimer, common to all SMs
        out["last_end_ns"] = int(last.max())
    return out


def timeline(rows: list) -> list:
    """First start and last end of each launch in ns after the first launch's
    start (the gaps between consecutive kernels of one pass)."""
    t0 = min(r["first_start_ns"] for r in rows if "first_start_ns" in r)
    for r in rows:
        if "first_start_ns" in r:
            r["start_at_ns"] = r.pop("first_start_ns") - t0
            r["end_at_ns"] = r.pop("last_end_ns") - t0
    return rows


def run(workload: str, seed: int = 0, graph: bool = False, reps: int = 20) -> list:
    """One plan + dispatch + combine of `workload` under the trace build.
    With graph=True the three calls are captured as one CUDA graph and
    replayed `reps` times, each replay queued behind a spin kernel (so that
    it runs as it would inside a longer decode step); the stamps of every
    replay are read back and the median of each figure is reported."""
    import torch
    from combine_moe_plan_gb300 import workloads as wl
    load()
    w = wl.WORKLOADS[workload]
    inp = wl.make_inputs(w, seed=seed)
    dev = torch.device("cuda", 0)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    ro = None if inp["rep_off"] is None else torch.from_numpy(inp["rep_off"]).to(dev)
    ri = None if inp["rep_ids"] is None else torch.from_numpy(inp["rep_ids"]).to(dev)
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=1, device=dev)
    if "ex_out" in inp:
        pool.view(0)["ex_out"][: w.rows].copy_(torch.from_numpy(inp["ex_out"].view(np.int16)).view(torch.bfloat16))
    y = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream(device=dev)

    def layer():
        pool.plan(logits, ro, ri, stream=s)
        pool.dispatch(x, after_plan=True, stream=s)
        pool.combine(w.T, y=y, stream=s)

    with torch.cuda.stream(s):
        for _ in range(3):  # warm: the last pass is the one read back
            reset(s)
            layer()
    torch.cuda.synchronize()
    if pool.check() != 0:
        raise RuntimeError("device error word set")
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layer()
        torch.cuda.synchronize()
        passes = []
        for _ in range(reps):
            reset()
            torch.cuda.synchronize()
            torch.cuda._sleep(40000)
            g.replay()
            torch.cuda.synchronize()
            passes.append(_pass_rows(w))
        return _median_rows(passes)
    return _pass_rows(w)


def _median_rows(passes: list) -> list:
    """Per kernel, the median over passes of every numeric figure."""
    out = []
    for rows in zip(*passes):
        r = dict(rows[0])
        for key in ("span_ns", "cta_ns_median", "start_at_ns", "end_at_ns"):
            if key in r:
                r[key] = float(np.median([x[key] for x in rows]))
        r["stages"] = {st: {"median_ns": float(np.median([x["stages"][st]["median_ns"] for x in rows
                                                          if st in x["stages"]])),
                            "ctas": r["stages"][st]["ctas"]} for st in r["stages"]}
        r["passes"] = len(rows)
        out.append(r)
    return out


def _pass_rows(w) -> list:
    """The stamps of the last pass, per kernel, on a common time axis."""
    n_tiles = (w.T + 15) // 16  # enough for either tile size: unused CTA slots are zero and skipped
    rows = []
    one = summarize(3, 32)  # one plan launch: the cluster kernel, or the ticket kernel without clusters
    if one["ctas"] > 0:
        rows.append(one)
    else:  # the three launches
        rows += [summarize(0, n_tiles), summarize(1, (w.P + 7) // 8), summarize(2, (w.rows + 255) // 256)]
    rows.append(summarize(4, min(TRACE_CTAS, (w.T * ((w.H + 511) // 512) + 7) // 8)))
    rows.append(summarize(5, min(TRACE_CTAS, (w.T * ((w.H + 255) // 256) + 7) // 8)))
    return timeline(rows)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="t96_h7168_e256_k8")
    ap.add_argument("--graph", action="store_true", help="replay the three calls as one CUDA graph")
    a = ap.parse_args(argv)
    for r in run(a.workload, graph=a.graph):
        print(json.dumps(r))


if __name__ == "__main__":
    main()

"""Host-side multi-rank logic of bench.py, on CPU with the gloo backend
(world size 2): the reported time is the max over ranks, each rank runs its
own replica (its own seed), and the reference arm prints on rank 0 only."""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    from combine_moe_plan_gb300 import workloads as wl
    out = bench.max_over_ranks([1.0 + rank, 5.0 - rank])
    w = wl.WORKLOADS["t64_h256_e8_k2"]
    x0 = wl.make_x(w, seed=rank)[0, :4].tolist()  # each rank draws its own batch
    dist.barrier()
    q.put((rank, out, bench._dist(), x0))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, out, d, _ in res:
        assert out == [2.0, 5.0]
        assert d == (2, rank, rank)
    assert res[0][3] != res[1][3]


def _ref(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "t64_h256_e8_k2", "--steps", "2", "--warmup", "1", *args],
                          capture_output=True, text=True, env=env, timeout=300)


def test_reference_arm_rank0_only():
    r1 = _ref({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _ref({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert r0.returncode == 0, r0.stderr
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "t64_h256_e8_k2"


def test_cpu_baseline_reports_all_cores_and_single_thread():
    import bench
    import oracle
    from combine_moe_plan_gb300 import workloads as wl
    before = oracle.threads()
    w = wl.WORKLOADS["t64_h256_e8_k2"]
    d = bench.cpu_baseline(w, wl.make_inputs(w), budget_s=0.2)
    assert d["kind"] == "oracle" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cores"] == oracle.threads() >= 1
    assert d["single_thread"]["cores"] == 1 and d["single_thread"]["value"] > 0
    oracle.set_threads(before)


def test_traffic_follows_the_kernel_source_closure(monkeypatch):
    """The ncu traffic figure is keyed to its workload and to a hash over the
    kernel file and every csrc header it includes: another workload, or a
    change to any of those files, drops the figure."""
    sys.path.insert(0, ROOT)
    import bench
    assert {"combine.cu", "ptx.cuh", "moe_internal.h"} <= set(bench.source_closure("combine.cu"))
    assert "quant.cuh" in bench.source_closure("dispatch.cu")
    top = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    rec, wname = top["combine_kernel"], top["workload"]
    monkeypatch.setattr(bench, "source_hash", lambda f: rec["source_sha256"])
    assert bench._traffic("combine.cu", "combine_kernel", wname) == rec["dram_bytes_per_launch"]
    # a per-launch figure belongs to the workload it was captured on
    assert bench._traffic("combine.cu", "combine_kernel", "t96_h7168_e256_k8") is None
    monkeypatch.setattr(bench, "source_hash", lambda f: "0" * 64)
    assert bench._traffic("combine.cu", "combine_kernel", wname) is None


def test_bench_line_describes_each_workload_and_its_l2_footing():
    """The data and l2 entries of the bench line follow the workload: its own
    input distributions, and whether a step's bytes exceed L2 (no flush is
    done, so only then are the figures DRAM figures)."""
    sys.path.insert(0, ROOT)
    import bench
    from combine_moe_plan_gb300 import workloads as wl
    d = {n: w.describe() for n, w in wl.WORKLOADS.items()}
    assert "Zipf(1.2)" in d["t4096_h7168_e256p288_k8"] and "32 hot experts" in d["t4096_h7168_e256p288_k8"]
    assert "Zipf" not in d["t96_h7168_e256_k8"] and "0.1 % of elements x50" in d["t96_h7168_e256_k8"]
    assert "N(0,0.5) bf16 expert rows" in d["t16384_h2048_e64_k6"]
    assert "identity experts" in d["t64_h256_e8_k2"]
    l2 = 129 * 10**6
    big = bench.l2_note(wl.WORKLOADS["t4096_h7168_e256p288_k8"].algorithmic_bytes()["total"], l2)
    small = bench.l2_note(wl.WORKLOADS["t96_h7168_e256_k8"].algorithmic_bytes()["total"], l2)
    assert big.startswith("inputs larger than L2") and "0.83 GB" in big
    assert small.startswith("inputs fit in L2") and "not a DRAM one" in small


def test_clock_samples_are_summarised_and_throttling_is_seen():
    """The clocks entry of the bench line: median SM clock under load, the
    maximum, and every throttle reason sampled Active (a run that saw a
    hardware or thermal slowdown is not a valid measurement)."""
    sys.path.insert(0, ROOT)
    import bench
    def row(sm, reasons=("Not Active",) * 4):
        return ", ".join(["2026/12/02 12:00:00.000", "0", str(sm), "2070", "900.1", "0x0"] + list(reasons))
    idle = [row(345)] * 3
    load = [row(2070)] * 7 + [row(2055)]
    c = bench.parse_clocks("\n".join(idle + load + ["garbled line"]))
    assert c == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 11}
    hot = row(1800, ("Active", "Not Active", "Not Active", "Active"))
    c = bench.parse_clocks("\n".join(load + [hot]))
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.parse_clocks("") is None

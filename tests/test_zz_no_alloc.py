"""moe_plan_static, the entry point for callers that cannot allocate device
memory (a graph replayed from elsewhere, a plugin whose host framework owns
every allocation, a process that must not grow its footprint after start-up).

Its results must equal moe_plan's on the same inputs, on two calls in a row
(the second call reuses the shared scratch array the first one left behind),
and the oracle's: bit-exact ids, counts, offsets, slots and inverse maps,
gates within 1 fp32 ulp.
Collected last on purpose, so that a stop-at-first-failure run has already
run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_moe_plan_gb300 import moe
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import assert_gates_close, compare_plan, dev, ensure_built

pytestmark = pytest.mark.gpu

KEYS = ("topk_e", "phys", "counts", "offsets", "slot", "src_token", "src_k")


def _pool_plan(w, logits, rep_off, rep_ids):
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=1)
    pool.plan(logits, rep_off, rep_ids)
    v = pool.view(0)
    R = w.T * w.k
    out = {k: v[k].clone() for k in ("topk_e", "gates", "phys", "counts", "offsets", "slot")}
    out["src_token"] = v["src_token"][:R].clone()
    out["src_k"] = v["src_k"][:R].clone()
    assert pool.check() == 0
    return out


def _compare(got, ref, what):
    for key in KEYS:
        np.testing.assert_array_equal(got[key].cpu().numpy(), ref[key].cpu().numpy(), err_msg=f"{what}:{key}")
    assert_gates_close(got["gates"].cpu().numpy(), ref["gates"].cpu().numpy(), what)
    assert int(got["error_word"].item()) == 0


def test_plan_static_matches_plan_two_calls_in_a_row():
    ensure_built()
    cases = [wl.WORKLOADS["t4096_h7168_e256p288_k8"], wl.small_variant(wl.WORKLOADS["t16384_h2048_e64_k6"], 3000),
             wl.WORKLOADS["t96_h7168_e256_k8"], wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 1500)]
    refs, gots = [], []
    for w in cases:
        inp = wl.make_inputs(w, with_expert_out=False)
        logits = dev(inp["logits"])
        ro = None if inp["rep_off"] is None else dev(inp["rep_off"])
        ri = None if inp["rep_ids"] is None else dev(inp["rep_ids"])
        refs.append(_pool_plan(w, logits, ro, ri))
        gots.append(moe.plan_static(logits, w.k, w.P, ro, ri))  # two calls back to back
    torch.cuda.synchronize()
    for w, got, ref in zip(cases, gots, refs):
        _compare(got, ref, w.name)
        inp = wl.make_inputs(w, with_expert_out=False)
        orc = oracle.plan(inp["logits"], w.k, inp["rep_off"], inp["rep_ids"], w.P)
        compare_plan({k: v.cpu().numpy() for k, v in got.items()}, orc, f"{w.name} vs oracle")


def test_plan_static_small_batches_overlap_on_two_streams():
    """Batches of up to 512 tokens take the cluster plan, which keeps its
    scratch in shared memory: calls on two streams may overlap on the GPU and
    still give moe_plan's results (96 and 300 tokens, 20 rounds, no
    synchronization between the streams)."""
    ensure_built()
    ws = [wl.WORKLOADS["t96_h7168_e256_k8"], wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 300)]
    # Only the cluster plan keeps its scratch out of the shared array.  At 300
    # tokens it is one launch; the fallback a refused cluster takes is three.
    w300 = ws[1]
    inp300 = wl.make_inputs(w300, with_expert_out=False)
    probe = moe.Pool(w300.T, w300.H, w300.E, w300.P, w300.k, n_sets=1)
    probe.plan(dev(inp300["logits"]), dev(inp300["rep_off"]), dev(inp300["rep_ids"]))
    if probe.launches() != 1:
        pytest.skip("this device does not take the cluster plan; overlapping calls would share the array")
    args, refs = [], []
    for w in ws:
        inp = wl.make_inputs(w, with_expert_out=False)
        logits = dev(inp["logits"])
        ro = None if inp["rep_off"] is None else dev(inp["rep_off"])
        ri = None if inp["rep_ids"] is None else dev(inp["rep_ids"])
        args.append((w, logits, ro, ri))
        refs.append(_pool_plan(w, logits, ro, ri))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[], []]
    torch.cuda.synchronize()
    for _ in range(20):
        for i, (w, logits, ro, ri) in enumerate(args):
            with torch.cuda.stream(streams[i]):
                outs[i].append(moe.plan_static(logits, w.k, w.P, ro, ri, stream=streams[i]))
    torch.cuda.synchronize()
    for i, (w, _, _, _) in enumerate(args):
        for r, got in enumerate(outs[i]):
            _compare(got, refs[i], f"{w.name} round {r}")


def test_plan_static_rejects_oversized_scratch():
    ensure_built()
    L = moe.lib()
    p = ctypes.c_void_p(1 << 41)  # never dereferenced: the size check comes first
    # 2^20 tokens x 4096 experts needs far more than the 4 MiB scratch array
    rc = L.moe_plan_static(p, 1 << 20, 1024, 4096, 8, p, p, p, p, p, p, p, p, p, p, p, None)
    assert rc == -2

"""moe_plan_dispatch (plan and dispatch as one call) against the oracle.

The call launches the plan's kernels and then the dispatch kernel in its
early form, which loads and quantizes x while the plan runs; the plan being
the kernel just before it makes that safe.  Every batch size and plan form is
covered (the cluster plan up to 512 tokens, the three launches beyond, the
ticket kernel when clusters are refused: tests/test_gpu_no_cluster.py re-runs
this file with MOE_PLAN_NO_CLUSTER=1).  The bar is the plan's and the
dispatch's: bit-exact ids, slots, inverse maps, codes and scales; gates within
1 fp32 ulp; y within 1 bf16 ulp.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from combine_moe_plan_gb300 import moe
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import (Run, assert_y_close, compare_plan, dev, dev_bf16, ensure_built, f32_bits,
                            host_u16)

pytestmark = pytest.mark.gpu

CLUSTERS = os.environ.get("MOE_PLAN_NO_CLUSTER") != "1"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check(w, inp, run, ex_out=None):
    ref = oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"], w.P, ex_out=ex_out)
    compare_plan(run.plan_host(), ref, w.name)
    R, G = run.T * w.k, w.G
    np.testing.assert_array_equal(run.v["codes"][:R].cpu().numpy(), ref["codes"], err_msg="codes")
    np.testing.assert_array_equal(f32_bits(run.v["scales"][:R, :G].cpu().numpy()), f32_bits(ref["scales"]),
                                  err_msg="scales")
    assert_y_close(host_u16(run.y), ref["y"], w.name)
    assert run.err == 0


def _custom(T, H, E, P, k, logits, rep_off=None, rep_ids=None, seed=0, T_max=None, pool=None):
    w = wl.Workload("custom", T=T, H=H, E=E, P=P, k=k)
    rng = np.random.default_rng(seed)
    x = wl.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    inp = {"logits": np.ascontiguousarray(logits, np.float32), "x": x, "rep_off": rep_off, "rep_ids": rep_ids}
    ex = wl.f32_to_bf16_bits(rng.standard_normal((T * k, H)).astype(np.float32))
    run = Run(w, inp, ex_out=ex, T_max=T_max, pool=pool, fused=True)
    _check(w, inp, run, ex_out=ex)
    return run


SMALL = [("t64_h256_e8_k2", 64), ("t96_h7168_e256_k8", 96), ("t4096_h7168_e256p288_k8", 300),
         ("t16384_h2048_e64_k6", 1000), ("t30720_h7168_e256_k8", 200), ("t4096_h7168_e256p288_k8", 512)]


@pytest.mark.parametrize("name,T", SMALL)
def test_workloads(name, T):
    w = wl.small_variant(wl.WORKLOADS[name], T)
    inp = wl.make_inputs(w)
    ex = inp.get("ex_out")  # None where the workload's experts are the identity
    run = Run(w, inp, ex_out=ex, fused=True)
    _check(w, inp, run, ex_out=ex)
    inp = wl.make_inputs(w, seed=7, with_expert_out=False)
    run = Run(w, inp, fused=True)
    _check(w, inp, run)
    np.testing.assert_array_equal(host_u16(run.v["ex_out"][: w.rows]),
                                  oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"],
                                                 w.P)["ex_out"], err_msg="identity experts")


@pytest.mark.parametrize("H", [256, 7168])
def test_switch_points_on_one_pool(H):
    """The cluster plan's tiles of 8 tokens up to 64, 16 up to 128, 32 up to
    512 (non-portable clusters beyond 256), the three launches from 513 on:
    every switch point on one pool, in both orders, with the bench workload's
    replica map."""
    rng = np.random.default_rng(31)
    E, P, k = 256, 288, 8
    inp = wl.make_inputs(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 513))
    pool = moe.Pool(513, H, E, P, k, n_sets=2)
    for T in (1, 8, 9, 64, 65, 128, 129, 256, 257, 512, 513, 512, 257, 129, 65, 9, 1, 33):
        _custom(T, H, E, P, k, inp["logits"][:T], rep_off=inp["rep_off"], rep_ids=inp["rep_ids"],
                seed=int(rng.integers(1 << 30)), T_max=513, pool=pool)


@pytest.mark.parametrize("T,H", [(96, 16384), (300, 16384), (512, 16384), (100, 640), (6, 65536)])
def test_long_rows_and_a_partial_segment(T, H):
    """Rows of 32 and 128 segments of 512 elements; H = 640 ends in a partial
    segment."""
    rng = np.random.default_rng(T + H)
    _custom(T, H, 64, 64, 6, rng.standard_normal((T, 64)), seed=T)


@pytest.mark.parametrize("T", [60, 100, 300])
def test_maximum_shapes(T):
    """E = 1024, P = 4096 (four replicas per expert), k = 32: the largest
    shared-memory footprint for each tile size (8, 16, 32 tokens)."""
    rng = np.random.default_rng(40 + T)
    E, P = 1024, 4096
    off = np.arange(0, P + 1, 4, dtype=np.int32)
    ids = rng.permutation(P).astype(np.int32)
    _custom(T, 128, E, P, 32, rng.standard_normal((T, E)), rep_off=off, rep_ids=ids, seed=T)


def test_same_buffers_as_the_two_calls():
    """Every buffer the two calls write (plan outputs, dispatch rows and
    scales) is written the same, byte for byte, by the one call."""
    w = wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 200)
    inp = wl.make_inputs(w, with_expert_out=False)
    a = Run(w, inp)
    b = Run(w, inp, fused=True)
    R = w.rows
    for key in ("topk_e", "gates", "phys", "slot"):
        assert torch.equal(a.v[key][: w.T], b.v[key][: w.T]), key
    for key in ("src_token", "src_k", "codes", "scales", "ex_out"):
        assert torch.equal(a.v[key][:R], b.v[key][:R]), key
    for key in ("counts", "offsets"):
        assert torch.equal(a.v[key], b.v[key]), key
    assert torch.equal(a.y, b.y)


@pytest.mark.parametrize("T", [1, 96, 512, 513])
def test_launches(T):
    """The plan's kernels (one cluster launch up to 512 tokens; without
    clusters the ticket kernel up to 128 tokens; else three) and the
    dispatch kernel."""
    w = wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], T)
    inp = wl.make_inputs(w, with_expert_out=False)
    pool = moe.Pool(T, 256, w.E, w.P, w.k)
    x_host = np.ascontiguousarray(inp["x"][:, :256])
    lg, x = dev(inp["logits"]), dev_bf16(x_host)
    ro, ri = dev(inp["rep_off"]), dev(inp["rep_ids"])
    n0 = pool.launches()
    pool.plan_dispatch(lg, x, ro, ri)
    n = pool.launches() - n0
    if T <= 512 and CLUSTERS:
        assert n == 2
    elif T <= 128:
        assert n == 2
    else:
        assert n == 4
    ref = oracle.forward(inp["logits"], x_host, w.k, inp["rep_off"], inp["rep_ids"], w.P)
    np.testing.assert_array_equal(pool.view(0)["codes"][: T * w.k].cpu().numpy(), ref["codes"])
    assert pool.check() == 0


def test_empty_batch():
    pool = moe.Pool(8, 256, 16, 16, 2)
    v = pool.view(0)
    v["counts"].fill_(7)
    v["offsets"].fill_(7)
    pool.plan_dispatch(torch.empty((0, 16), dtype=torch.float32, device="cuda"),
                       torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"))
    y = pool.combine(0)
    assert y.shape == (0, 256) and pool.check() == 0
    assert not v["counts"].any() and not v["offsets"].any()


def test_bad_replica_map_sets_the_error_word():
    """An id outside [0, P) in the replica map is reported in the error word,
    no row is written out of range, and the pool is usable after the error is
    cleared."""
    E, P, k, T, H = 4, 6, 2, 40, 128
    off = dev(np.array([0, 2, 3, 5, 6], np.int32))
    ids = dev(np.array([0, 4, 1, 2, 99, 3], np.int32))
    pool = moe.Pool(T, H, E, P, k)
    logits = dev(np.random.default_rng(8).standard_normal((T, E)).astype(np.float32))
    x = dev_bf16(wl.f32_to_bf16_bits(np.ones((T, H), np.float32)))
    pool.plan_dispatch(logits, x, off, ids)
    pool.combine(T)
    err = pool.check()
    assert err & moe.DEVERR_REPLICA
    assert err & moe.DEVERR_SLOT
    pool.clear_error()
    assert pool.check() == 0
    _custom(T, H, E, P, k, np.random.default_rng(9).standard_normal((T, E)),
            rep_off=np.array([0, 2, 3, 5, 6], np.int32), rep_ids=np.array([0, 4, 1, 2, 5, 3], np.int32), seed=3,
            pool=pool)


def test_two_streams_two_sets():
    """Two batches on two streams and two buffer sets, launched back to back
    several times: each set's results are its own batch's."""
    w = wl.small_variant(wl.WORKLOADS["t96_h7168_e256_k8"], 96)
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2)
    inps = [wl.make_inputs(w, seed=50 + b, with_expert_out=False) for b in range(2)]
    lg = [dev(i["logits"]) for i in inps]
    xs = [dev_bf16(i["x"]) for i in inps]
    ys = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(5):
        for b in range(2):
            with torch.cuda.stream(streams[b]):
                pool.plan_dispatch(lg[b], xs[b], buf=b, stream=streams[b])
                pool.identity_experts(w.T, buf=b, stream=streams[b])
                pool.combine(w.T, y=ys[b], buf=b, stream=streams[b])
    torch.cuda.synchronize()
    for b in range(2):
        ref = oracle.forward(inps[b]["logits"], inps[b]["x"], w.k, None, None, w.P)
        np.testing.assert_array_equal(pool.view(b)["codes"][: w.rows].cpu().numpy(), ref["codes"])
        assert_y_close(host_u16(ys[b]), ref["y"], f"set {b}")
    assert pool.check() == 0

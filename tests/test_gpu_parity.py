"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bar: bit-exact for top-k experts, physical experts, counts, offsets, slots,
inverse maps, INT8 codes and fp32 scales; gates within 1 fp32 ulp (fp64
softmax rounded once on both sides, so in practice identical); combine output
within 1 bf16 ulp (identical unless a gate differed).
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_plan_gb300 import moe
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import (Run, assert_y_close, compare_plan, dev, dev_bf16, ensure_built, f32_bits,
                            host_u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


# Oracle-sized variants of every workload: several 32-token tiles plus a
# ragged tail (or the workload's own T where it is already small).
SMALL = [("t64_h256_e8_k2", 64), ("t96_h7168_e256_k8", 96), ("t4096_h7168_e256p288_k8", 300),
         ("t16384_h2048_e64_k6", 1000), ("t30720_h7168_e256_k8", 200)]


def _check_all(w, inp, run, ex_out=None):
    ref = oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"], w.P, ex_out=ex_out)
    compare_plan(run.plan_host(), ref, w.name)
    R, G = run.T * w.k, w.G
    np.testing.assert_array_equal(run.v["codes"][:R].cpu().numpy(), ref["codes"], err_msg="codes")
    np.testing.assert_array_equal(f32_bits(run.v["scales"][:R, :G].cpu().numpy()), f32_bits(ref["scales"]),
                                  err_msg="scales")
    if ex_out is None:
        np.testing.assert_array_equal(host_u16(run.v["ex_out"][:R]), ref["ex_out"], err_msg="identity experts")
    nd = assert_y_close(host_u16(run.y), ref["y"], w.name)
    assert run.err == 0
    return nd


@pytest.mark.parametrize("name,T", SMALL)
def test_small_parity_generated_experts(name, T):
    w = wl.small_variant(wl.WORKLOADS[name], T)
    inp = wl.make_inputs(w)
    ex = inp.get("ex_out")
    run = Run(w, inp, ex_out=ex)
    _check_all(w, inp, run, ex_out=ex)


@pytest.mark.parametrize("name,T", SMALL)
def test_small_parity_identity_experts_roundtrip(name, T):
    w = wl.small_variant(wl.WORKLOADS[name], T)
    inp = wl.make_inputs(w, with_expert_out=False)
    run = Run(w, inp)
    _check_all(w, inp, run)
    # round trip: y recovers x within the INT8 bound plus two bf16 roundings
    x = wl.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    y = wl.bf16_bits_to_f32(host_u16(run.y)).astype(np.float64)
    _, s = oracle.quantize(inp["x"])
    scale = np.repeat(s.astype(np.float64), 128, axis=1)
    bound = scale * (0.5 + 2.0 ** -12) + 2.0 ** -7 * (np.abs(x) + 0.5 * scale) + 127 * scale * 2.0 ** -20
    assert np.all(np.abs(y - x) <= bound)


def test_full_bench_workload_parity():
    """The bench workload at full size (4096 x 7168, 288 physical experts,
    top-8), compared in full."""
    w = wl.WORKLOADS["t4096_h7168_e256p288_k8"]
    inp = wl.make_inputs(w)
    run = Run(w, inp, ex_out=inp["ex_out"])
    _check_all(w, inp, run, ex_out=inp["ex_out"])
    # replicas carry traffic: every physical slot of a hot expert got tokens
    counts = run.plan_host()["counts"]
    assert (counts[w.E:] > 0).all()


def test_full_16384_ten_iterations_double_buffered():
    """16384 x 2048, 64 experts, top-6: 10 back-to-back iterations alternating
    the two buffer sets (buf = i & 1) with no host sync in between; every
    iteration's output checked against the oracle."""
    w = wl.WORKLOADS["t16384_h2048_e64_k6"]
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2)
    runs = []
    for i in range(w.iterations):
        inp = wl.make_inputs(w, seed=i)
        logits, x, ex = dev(inp["logits"]), dev_bf16(inp["x"]), dev_bf16(inp["ex_out"])
        buf = i & 1
        pool.plan(logits, buf=buf)
        pool.dispatch(x, buf=buf)
        y = pool.combine(w.T, ex_out=ex, buf=buf)
        runs.append((inp, y, (logits, x, ex)))
    assert pool.check() == 0
    for i, (inp, y, _) in enumerate(runs):
        pl = oracle.plan(inp["logits"], w.k)
        y_ref = oracle.combine(inp["ex_out"], pl["slot"], pl["gates"])
        assert_y_close(host_u16(y), y_ref, f"iteration {i}")
    # the last two iterations' metadata and dispatch rows are still in the sets
    for i in (w.iterations - 2, w.iterations - 1):
        inp = runs[i][0]
        v = pool.view(i & 1)
        ref = oracle.plan(inp["logits"], w.k)
        np.testing.assert_array_equal(v["slot"].cpu().numpy(), ref["slot"])
        codes, scales = oracle.dispatch(inp["x"], ref["slot"])
        np.testing.assert_array_equal(v["codes"][:w.rows].cpu().numpy(), codes)


def test_full_30720_in_full():
    """Global decode batch 30720 x 7168, 256 experts, top-8, buffers sized for
    the worst case: plan metadata, every dispatch row (codes and scales) and
    every combine output compared in full with the oracle."""
    w = wl.WORKLOADS["t30720_h7168_e256_k8"]
    inp = wl.make_inputs(w)
    run = Run(w, inp, ex_out=inp["ex_out"])
    ref = oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"], w.P, ex_out=inp["ex_out"])
    compare_plan(run.plan_host(), ref, w.name)
    R = w.T * w.k
    assert np.array_equal(run.v["codes"][:R].cpu().numpy(), ref["codes"]), "codes"
    assert np.array_equal(f32_bits(run.v["scales"][:R, :w.G].cpu().numpy()), f32_bits(ref["scales"])), "scales"
    assert_y_close(host_u16(run.y), ref["y"], w.name)
    assert run.err == 0


def test_largest_batch_the_pool_takes():
    """T = 2^20 tokens, the largest batch a pool takes (hidden 128, 64
    experts with 16 replicas, top-8: 8.4 M copies, 32,768 route tiles):
    the whole plan, every dispatch row and every combine output compared in
    full with the oracle, through moe_plan_dispatch."""
    T, H, E, k = 1 << 20, 128, 64, 8
    rng = np.random.default_rng(77)
    hot = rng.choice(E, size=16, replace=False)
    off, ids, nxt = [0], [], E
    for e in range(E):
        mine = [e] + ([nxt] if e in hot else [])
        nxt += e in hot
        ids += mine
        off.append(off[-1] + len(mine))
    P = nxt
    rep_off, rep_ids = np.array(off, np.int32), rng.permutation(P)[np.array(ids)].astype(np.int32)
    w = wl.Workload("custom", T=T, H=H, E=E, P=P, k=k)
    inp = {"logits": rng.standard_normal((T, E), dtype=np.float32),
           "x": wl.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32)),
           "rep_off": rep_off, "rep_ids": rep_ids}
    run = Run(w, inp, n_sets=1, fused=True)
    _check_all(w, inp, run)


# ------------------------------------------------------------ edge cases --

def _custom(T, H, E, P, k, logits, x=None, rep_off=None, rep_ids=None, seed=0, T_max=None, pool=None):
    w = wl.Workload("custom", T=T, H=H, E=E, P=P, k=k)
    rng = np.random.default_rng(seed)
    if x is None:
        x = wl.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    inp = {"logits": np.ascontiguousarray(logits, np.float32), "x": x, "rep_off": rep_off, "rep_ids": rep_ids}
    ex = wl.f32_to_bf16_bits(rng.standard_normal((T * k, H)).astype(np.float32))
    run = Run(w, inp, ex_out=ex, T_max=T_max, pool=pool)
    _check_all(w, inp, run, ex_out=ex)
    run2 = Run(w, inp, T_max=T_max, pool=pool)
    _check_all(w, inp, run2)
    return run


# The three ways to run a batch's plan and dispatch: moe_plan + moe_dispatch
# ("wait": x read after the wait), moe_plan + moe_dispatch_after_plan, and
# moe_plan_dispatch (the two as one call).
MODES = ["wait", "after_plan", "fused"]


def _plan_dispatch(pool, mode, logits, ro, ri, x, buf, stream):
    if mode == "fused":
        pool.plan_dispatch(logits, x, ro, ri, buf=buf, stream=stream)
    else:
        pool.plan(logits, ro, ri, buf=buf, stream=stream)
        pool.dispatch(x, buf=buf, stream=stream, after_plan=(mode == "after_plan"))


def test_single_token():
    _custom(1, 256, 8, 8, 2, np.random.default_rng(1).standard_normal((1, 8)))


def test_k_equals_E_and_k1():
    rng = np.random.default_rng(2)
    _custom(70, 128, 8, 8, 8, rng.standard_normal((70, 8)))
    _custom(70, 384, 16, 16, 1, rng.standard_normal((70, 16)))


def test_ties_and_signed_zero():
    rng = np.random.default_rng(3)
    vals = np.array([-1.0, -0.0, 0.0, 0.5, 0.5, 2.0], np.float32)
    _custom(97, 256, 40, 40, 5, rng.choice(vals, size=(97, 40)))


def test_everyone_on_one_expert():
    """Worst-case capacity: all tokens pick expert 0 first."""
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((300, 64)).astype(np.float32)
    lg[:, 0] += 100.0
    run = _custom(300, 512, 64, 64, 4, lg)
    assert run.plan_host()["counts"][0] == 300


def test_max_experts_and_max_k():
    rng = np.random.default_rng(5)
    _custom(65, 128, 1024, 1024, 32, rng.standard_normal((65, 1024)))


def test_max_experts_with_replica_map():
    """E = 1024 logical experts (1025 CSR offsets) with 76 replicas, P = 1100."""
    E, P, k, T = 1024, 1100, 8, 70
    rng = np.random.default_rng(9)
    hot = rng.choice(E, size=P - E, replace=False)
    off = np.zeros(E + 1, np.int32)
    ids = []
    extra = E
    for e in range(E):
        mine = [e]
        if e in set(hot.tolist()):
            mine.append(extra)
            extra += 1
        ids += mine
        off[e + 1] = off[e] + len(mine)
    ids = np.array(ids, np.int32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[:, hot] += 2.0
    _custom(T, 128, E, P, k, lg, rep_off=off, rep_ids=ids)


def test_three_replicas_and_zero_groups():
    """Expert 0 has three physical replicas; some activation groups are all zero."""
    E, P = 6, 9
    off = np.array([0, 3, 4, 5, 7, 8, 9], np.int32)   # expert 0: 3 replicas, expert 3: 2
    ids = np.array([0, 6, 8, 1, 2, 3, 7, 4, 5], np.int32)
    rng = np.random.default_rng(6)
    lg = rng.standard_normal((130, E)).astype(np.float32)
    lg[:, 0] += 3.0
    x = rng.standard_normal((130, 384)).astype(np.float32)
    x[5, :] = 0.0
    x[7, 128:256] = -0.0
    _custom(130, 384, E, P, 3, lg, x=wl.f32_to_bf16_bits(x), rep_off=off, rep_ids=ids)


def test_pool_reuse_smaller_T_and_ragged_tail():
    """A pool sized for 256 tokens serves a 256-token call, then a 33-token
    call (one full tile plus one token) on the same set."""
    rng = np.random.default_rng(7)
    pool = moe.Pool(256, 256, 32, 32, 4, n_sets=2)
    _custom(256, 256, 32, 32, 4, rng.standard_normal((256, 32)), pool=pool)
    _custom(33, 256, 32, 32, 4, rng.standard_normal((33, 32)), pool=pool)


def test_outlier_workload_scales():
    """The decode-batch workload's x50 outliers dominate their groups' scales."""
    w = wl.WORKLOADS["t96_h7168_e256_k8"]
    inp = wl.make_inputs(w)
    run = Run(w, inp, ex_out=inp["ex_out"])
    s = run.v["scales"][:w.rows, :w.G].cpu().numpy()
    assert s.max() > 20 * np.median(s)


# --------------------------------------------------------- error reporting --

def test_device_error_word_bad_replica_map():
    """A replica map with an id outside [0, P) is caught by the kernel's own
    bounds check: the error word says so and nothing is written out of range."""
    E, P, k, T, H = 4, 6, 2, 40, 128
    off = dev(np.array([0, 2, 3, 5, 6], np.int32))
    ids = dev(np.array([0, 4, 1, 2, 99, 3], np.int32))  # 99 is out of range
    pool = moe.Pool(T, H, E, P, k)
    logits = dev(np.random.default_rng(8).standard_normal((T, E)).astype(np.float32))
    x = dev_bf16(wl.f32_to_bf16_bits(np.ones((T, H), np.float32)))
    pool.plan(logits, off, ids)
    pool.dispatch(x)
    pool.combine(T)
    err = pool.check()
    assert err & moe.DEVERR_REPLICA
    assert err & moe.DEVERR_SLOT
    pool.clear_error()
    assert pool.check() == 0


def test_device_error_word_duplicate_physical_id():
    E, P, k, T, H = 4, 4, 2, 64, 128
    off = dev(np.array([0, 1, 2, 3, 4], np.int32))
    ids = dev(np.array([0, 0, 2, 3], np.int32))  # experts 0 and 1 share a slot
    pool = moe.Pool(T, H, E, P, k)
    lg = np.zeros((T, E), np.float32)
    lg[:, :2] = 5.0  # every token picks experts 0 and 1
    pool.plan(dev(lg), off, ids)
    pool.dispatch(dev_bf16(wl.f32_to_bf16_bits(np.ones((T, H), np.float32))))
    pool.combine(T)
    assert pool.check() & moe.DEVERR_DUPLICATE


def test_launch_count():
    w = wl.small_variant(wl.WORKLOADS["t64_h256_e8_k2"], 64)
    inp = wl.make_inputs(w, with_expert_out=False)
    pool = moe.Pool(64, w.H, w.E, w.P, w.k)
    n0 = pool.launches()
    Run(w, inp, pool=pool)
    # a 64-token plan is one launch (the cluster plan); then dispatch, identity experts, combine
    assert pool.launches() - n0 == 4
    # a 1056-token plan (33 tiles) takes the three-launch path
    big = wl.small_variant(wl.WORKLOADS["t64_h256_e8_k2"], 1056)
    inp = wl.make_inputs(big, with_expert_out=False)
    pool = moe.Pool(big.T, big.H, big.E, big.P, big.k)
    n0 = pool.launches()
    Run(big, inp, pool=pool)
    assert pool.launches() - n0 == 6
    _check_all(big, inp, Run(big, inp, pool=pool))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("T", [40, 96, 200, 512, 1000])
def test_step_captures_in_a_cuda_graph(T, mode):
    """plan -> dispatch -> combine (PDL launches) captured once in a CUDA graph
    and replayed on new input contents gives the oracle's results: 40, 96, 200
    and 512 tokens (cluster plans of 5 CTAs of 8 tokens, 6 of 16, 7 of 32 and
    16 of 32) and 1000 (the three launches), with plan and dispatch in each of
    the three forms."""
    w = wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], T)
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2)
    inp0 = wl.make_inputs(w, seed=0)
    logits, x, ex = dev(inp0["logits"]), dev_bf16(inp0["x"]), dev_bf16(inp0["ex_out"])
    ro, ri = dev(inp0["rep_off"]), dev(inp0["rep_ids"])
    y = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # warm
        _plan_dispatch(pool, mode, logits, ro, ri, x, 1, s)
        pool.combine(w.T, y=y, ex_out=ex, buf=1, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _plan_dispatch(pool, mode, logits, ro, ri, x, 1, s)
        pool.combine(w.T, y=y, ex_out=ex, buf=1, stream=s)
    for seed in (3, 4, 5):
        inp = wl.make_inputs(w, seed=seed)
        logits.copy_(dev(inp["logits"]))
        x.copy_(dev_bf16(inp["x"]))
        ex.copy_(dev_bf16(inp["ex_out"]))
        ro.copy_(dev(inp["rep_off"]))  # the replica map follows the seed's popularity ranking
        ri.copy_(dev(inp["rep_ids"]))
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"], w.P,
                             ex_out=inp["ex_out"])
        np.testing.assert_array_equal(pool.view(1)["slot"].cpu().numpy(), ref["slot"])
        np.testing.assert_array_equal(pool.view(1)["codes"][:w.rows].cpu().numpy(), ref["codes"])
        assert_y_close(host_u16(y), ref["y"], f"graph replay seed {seed}")
    assert pool.check() == 0


def test_empty_batch_and_maximum_sizes():
    """T = 0 is a no-op with empty windows; P = 4096 (4 replicas per expert)
    and H = 65536 go through the whole path."""
    pool = moe.Pool(8, 256, 16, 16, 2)
    v = pool.view(0)
    v["counts"].fill_(7)
    v["offsets"].fill_(7)
    pool.plan(torch.empty((0, 16), dtype=torch.float32, device="cuda"))
    pool.dispatch(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"))
    y = pool.combine(0)
    assert y.shape == (0, 256) and pool.check() == 0
    assert not v["counts"].any() and not v["offsets"].any()
    ref = oracle.place(np.zeros((0, 2), np.int32), 16)
    assert ref["offsets"].tolist() == [0] * 17
    with pytest.raises(moe.MoeError):
        pool.dispatch(torch.empty((1, 256), dtype=torch.bfloat16, device="cuda"))

    rng = np.random.default_rng(10)
    E, P = 1024, 4096
    off = np.arange(0, P + 1, 4, dtype=np.int32)
    ids = rng.permutation(P).astype(np.int32)
    _custom(40, 128, E, P, 4, rng.standard_normal((40, E)), rep_off=off, rep_ids=ids)
    _custom(6, 65536, 8, 8, 2, rng.standard_normal((6, 8)))


@pytest.mark.parametrize("k", list(range(1, 13)))
def test_combine_every_batch_width(k):
    """Combine keeps min(k, 8) copies in flight (one kernel per width); every
    k from 1 to 12, so each width and k > 8 (a partial second batch) run, at
    H = 384 (the second 256-element segment is half full)."""
    rng = np.random.default_rng(300 + k)
    E = max(16, k)
    _custom(45, 384, E, E, k, rng.standard_normal((45, E)), seed=k)


@pytest.mark.parametrize("E", [8, 16, 32, 64, 100, 128, 200, 512])
@pytest.mark.parametrize("k", [2, 6, 12])
def test_route_lane_segments(E, k):
    """The three-launch route kernel gives each token 8, 16 or 32 lanes
    (the fewest that keep at most 8 logits a lane and a lane per gate);
    1100 tokens (35 tiles) over expert counts and k that select every
    (lanes, logits-per-lane) variant, checked in full against the oracle."""
    if k > E:
        pytest.skip("k > E")
    rng = np.random.default_rng(1000 * k + E)
    _custom(1100, 128, E, E, k, rng.standard_normal((1100, E)), seed=E + k)


@pytest.mark.parametrize("T", [64, 1100])
def test_non_finite_logits_keep_a_valid_placement(T):
    """NaN and +-Inf logits and activations are outside the method's domain
    (the oracle rejects them; gates, codes and y are unspecified), but both
    plan paths must still pick k distinct experts per token in range, place
    every copy exactly once, set no device error bit, and leave the pool
    usable: a finite batch right after matches the oracle."""
    rng = np.random.default_rng(77)
    E, k, H = 64, 6, 256
    logits = rng.standard_normal((T, E)).astype(np.float32)
    flat = logits.reshape(-1)
    pos = rng.choice(flat.size, size=flat.size // 20, replace=False)
    flat[pos[0::3]] = np.nan
    flat[pos[1::3]] = np.inf
    flat[pos[2::3]] = -np.inf
    pool = moe.Pool(T, H, E, E, k, n_sets=1)
    xf = rng.standard_normal((T, H)).astype(np.float32)
    xf[rng.random((T, H)) < 0.01] = np.nan  # non-finite activations too: codes and scales unspecified
    xf[rng.random((T, H)) < 0.01] = np.inf
    x = dev_bf16(wl.f32_to_bf16_bits(xf))
    pool.plan(dev(logits))
    pool.dispatch(x)
    pool.combine(T)
    assert pool.check() == 0
    v = pool.view(0)
    topk = v["topk_e"][:T].cpu().numpy()
    assert topk.min() >= 0 and topk.max() < E
    assert all(len(set(r)) == k for r in topk.tolist())
    slots = v["slot"][:T].cpu().numpy()
    assert sorted(slots.ravel().tolist()) == list(range(T * k))
    finite = rng.standard_normal((T, E)).astype(np.float32)
    _custom(T, H, E, E, k, finite, pool=pool, T_max=T)


def test_step_host_matches_oracle():
    """moe_step_host: logits and x from pinned host memory, plan, dispatch,
    expert outputs from the host (or the identity stand-in), combine, y back
    to the host.  Four steps alternate the two sets on two streams with their
    own inputs; every y and plan is checked against the oracle."""
    w = wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 300)
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    steps = []
    for i in range(4):
        inp = wl.make_inputs(w, seed=40 + i)
        h_logits = torch.from_numpy(inp["logits"]).pin_memory()
        h_x = torch.from_numpy(inp["x"].view(np.int16)).pin_memory()
        h_ex = torch.from_numpy(inp["ex_out"][: w.T * w.k].view(np.int16)).pin_memory() if i % 2 else None
        h_y = torch.empty((w.T, w.H), dtype=torch.int16).pin_memory()
        ro, ri = dev(inp["rep_off"]), dev(inp["rep_ids"])
        steps.append((inp, h_logits, h_x, h_ex, h_y, ro, ri))
    for i, (inp, h_logits, h_x, h_ex, h_y, ro, ri) in enumerate(steps[:2]):
        pool.step_host(h_logits, h_x, h_y, h_ex, ro, ri, buf=i, stream=streams[i])
    torch.cuda.synchronize()
    for i, (inp, h_logits, h_x, h_ex, h_y, ro, ri) in enumerate(steps):
        if i >= 2:
            pool.step_host(h_logits, h_x, h_y, h_ex, ro, ri, buf=i % 2, stream=streams[i % 2])
            torch.cuda.synchronize()
        ex = None if h_ex is None else inp["ex_out"][: w.T * w.k]
        ref = oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"], w.P, ex_out=ex)
        assert_y_close(h_y.numpy().view(np.uint16), ref["y"], f"step {i}")
        v = pool.view(i % 2)
        np.testing.assert_array_equal(v["slot"][: w.T].cpu().numpy(), ref["slot"])
    assert pool.check() == 0


def test_plan_at_32_and_33_tiles():
    """1024 tokens (32 tiles) and 1025 (33 tiles, a ragged tail of one token)
    through the three launches on one pool, one after the other."""
    rng = np.random.default_rng(12)
    E, P, k, H = 256, 288, 8, 256
    w = wl.WORKLOADS["t4096_h7168_e256p288_k8"]
    inp = wl.make_inputs(wl.small_variant(w, 1025))
    pool = moe.Pool(1025, H, E, P, k, n_sets=2)
    for T in (1024, 1025, 1024):
        _custom(T, H, E, P, k, inp["logits"][:T], rep_off=inp["rep_off"], rep_ids=inp["rep_ids"],
                seed=int(rng.integers(1 << 30)), T_max=1025, pool=pool)


def test_plan_path_switch_at_cluster_sizes():
    """The cluster plan takes tiles of 8 tokens up to 64 tokens, 16 up to 128
    and 32 up to 512; up to 256 tokens the cluster is portable (at most 8
    CTAs), 257 to 512 need the non-portable size; 513 tokens and more take the
    three launches (and without clusters, 129 tokens and more).  Every switch
    point (1, 8, 9, 64, 65, 128, 129, 256, 257, 512, 513 tokens) on one pool,
    one after the other, in both orders, with the bench workload's replica
    map."""
    rng = np.random.default_rng(13)
    E, P, k, H = 256, 288, 8, 256
    inp = wl.make_inputs(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 513))
    pool = moe.Pool(513, H, E, P, k, n_sets=2)
    for T in (1, 8, 9, 64, 65, 128, 129, 256, 257, 512, 513, 512, 257, 256, 129, 128, 65, 64, 9, 8, 1, 33, 32):
        _custom(T, H, E, P, k, inp["logits"][:T], rep_off=inp["rep_off"], rep_ids=inp["rep_ids"],
                seed=int(rng.integers(1 << 30)), T_max=513, pool=pool)


def test_plan_mid_size_tiles():
    """513 to 2048 tokens whose tokens take a whole warp route in 16-token
    tiles (512-thread CTAs); beyond 2048, 32-token tiles again.  Every switch
    point and a ragged tail of each tile size on one pool sized for 3000
    tokens, one after the other in both orders; then a pool sized for 700
    tokens, whose tile-count scratch holds ceil(700 / 16) columns."""
    rng = np.random.default_rng(14)
    E, P, k, H = 256, 288, 8, 256
    inp = wl.make_inputs(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 3000))
    pool = moe.Pool(3000, H, E, P, k, n_sets=2)
    for T in (513, 527, 528, 1000, 2047, 2048, 2049, 3000, 2048, 1025, 512, 513):
        _custom(T, H, E, P, k, inp["logits"][:T], rep_off=inp["rep_off"], rep_ids=inp["rep_ids"],
                seed=int(rng.integers(1 << 30)), T_max=3000, pool=pool)
    pool = moe.Pool(700, H, E, P, k, n_sets=1)
    for T in (700, 513, 699):
        _custom(T, H, E, P, k, inp["logits"][:T], rep_off=inp["rep_off"], rep_ids=inp["rep_ids"],
                seed=int(rng.integers(1 << 30)), T_max=700, pool=pool)


def test_three_launch_plan_at_maximum_shapes():
    """More than 32 tiles (so the route / column-scan / assign kernels run)
    at the largest shapes the API takes: E = 1024, P = 4096 (four replicas per
    expert), k = 32 -- the route kernel's largest shared-memory footprint."""
    rng = np.random.default_rng(11)
    E, P = 1024, 4096
    off = np.arange(0, P + 1, 4, dtype=np.int32)
    ids = rng.permutation(P).astype(np.int32)
    _custom(1100, 128, E, P, 32, rng.standard_normal((1100, E)), rep_off=off, rep_ids=ids)


@pytest.mark.parametrize("T", [60, 100, 300])
def test_cluster_plan_at_maximum_shapes(T):
    """The cluster plan at the largest shapes the API takes (E = 1024, P =
    4096 with four replicas per expert, k = 32), for each tile size: 60 tokens
    (8 CTAs of 8), 100 (7 of 16), 300 (10 of 32, non-portable) -- its largest
    shared-memory footprint (about 85 KB a CTA) and 32 keys a lane."""
    rng = np.random.default_rng(20 + T)
    E, P = 1024, 4096
    off = np.arange(0, P + 1, 4, dtype=np.int32)
    ids = rng.permutation(P).astype(np.int32)
    _custom(T, 128, E, P, 32, rng.standard_normal((T, E)), rep_off=off, rep_ids=ids, seed=T)


@pytest.mark.parametrize("mode", MODES)
def test_bench_schedule_two_streams_full_size(mode):
    """The bench's timed schedule at the bench workload's full size: steps
    alternate the two buffer sets on two streams, launched back to back, each
    step with its own inputs and output buffer; every step's result is
    checked against the oracle.  The bench's own form is moe_plan_dispatch
    ("fused")."""
    w = wl.WORKLOADS["t4096_h7168_e256p288_k8"]
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    steps = []
    for i in range(6):
        inp = wl.make_inputs(w, seed=100 + i)
        steps.append((inp, dev(inp["logits"]), dev_bf16(inp["x"]), dev_bf16(inp["ex_out"]),
                      dev(inp["rep_off"]), dev(inp["rep_ids"]),
                      torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")))
    torch.cuda.synchronize()
    ev = torch.cuda.Event()
    ev.record()
    for s in streams:
        s.wait_event(ev)
    for i, (_, logits, x, ex, ro, ri, y) in enumerate(steps):
        s, b = streams[i & 1], i & 1
        _plan_dispatch(pool, mode, logits, ro, ri, x, b, s)
        pool.combine(w.T, y=y, ex_out=ex, buf=b, stream=s)
    torch.cuda.synchronize()
    assert pool.check() == 0
    for i, (inp, *_, y) in enumerate(steps):
        pl = oracle.plan(inp["logits"], w.k, inp["rep_off"], inp["rep_ids"], w.P)
        assert_y_close(host_u16(y), oracle.combine(inp["ex_out"], pl["slot"], pl["gates"]), f"step {i}")
    # the last step of each set left its plan and dispatch rows in the set
    for i in (4, 5):
        inp = steps[i][0]
        v = pool.view(i & 1)
        pl = oracle.plan(inp["logits"], w.k, inp["rep_off"], inp["rep_ids"], w.P)
        np.testing.assert_array_equal(v["slot"].cpu().numpy(), pl["slot"])
        codes, _ = oracle.dispatch(inp["x"], pl["slot"])
        np.testing.assert_array_equal(v["codes"][:w.rows].cpu().numpy(), codes)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name,T", [("t96_h7168_e256_k8", 96), ("t4096_h7168_e256p288_k8", 300),
                                    ("t16384_h2048_e64_k6", 1000), ("t16384_h2048_e64_k6", 2000)])
def test_layers_chained_on_one_stream(name, T, mode):
    """Six layers back to back on one stream, each layer's y the next layer's x,
    the two buffer sets alternating, no synchronization in between; then the
    same chain captured once as a CUDA graph and replayed.  Every layer's y
    equals the oracle run layer after layer on its own outputs.  With
    after_plan, dispatch reads x before its wait for the plan, so this checks
    that the previous layer's combine has finished writing x by then (the
    plan in between waits for it); moe_plan_dispatch does the same in one
    call.
    The plan forms covered: cluster (96 tokens as 6 CTAs of 16, 300 as 10 of
    32) and three launches (1000 and 2000 tokens, 8-lane segments at 64
    experts); the test run without clusters adds the ticket kernel."""
    w = wl.small_variant(wl.WORKLOADS[name], T)
    L = 6
    layers = [wl.make_inputs(w, seed=10 + l, with_expert_out=False) for l in range(L)]
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2)
    x0 = dev_bf16(layers[0]["x"])
    lg = [dev(inp["logits"]) for inp in layers]
    ro = [None if inp["rep_off"] is None else dev(inp["rep_off"]) for inp in layers]
    ri = [None if inp["rep_ids"] is None else dev(inp["rep_ids"]) for inp in layers]
    ys = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(L)]

    refs, x = [], layers[0]["x"]
    for l, inp in enumerate(layers):
        refs.append(oracle.forward(inp["logits"], x, w.k, inp["rep_off"], inp["rep_ids"], w.P)["y"])
        x = refs[-1]

    s = torch.cuda.Stream()

    def chain():
        xin = x0
        for l in range(L):
            b = l & 1
            _plan_dispatch(pool, mode, lg[l], ro[l], ri[l], xin, b, s)
            pool.identity_experts(w.T, buf=b, stream=s)
            pool.combine(w.T, y=ys[l], buf=b, stream=s)
            xin = ys[l]

    def fill_nan():
        for y in ys:
            y.view(torch.int16).fill_(-1)  # 0xffff: a NaN that no layer produces
        torch.cuda.synchronize()

    fill_nan()
    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    for l in range(L):
        assert_y_close(host_u16(ys[l]), refs[l], f"{name} T={T} layer {l}")
    assert pool.check() == 0

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    for _ in range(2):
        fill_nan()
        g.replay()
        torch.cuda.synchronize()
        for l in range(L):
            assert_y_close(host_u16(ys[l]), refs[l], f"{name} T={T} graph layer {l}")
    assert pool.check() == 0


def test_handworked_cases_on_the_gpu():
    """The hand-worked fixtures (tests/golden/handworked.json: every output
    derived by hand from the method's definitions) checked against the CUDA
    path directly, not through the oracle: routing, placement, codes, scales
    and, through the identity experts, y."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "handworked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        T, H, E, P, k = c["T"], c["H"], c["E"], c["P"], c["k"]
        pool = moe.Pool(T, H, E, P, k, n_sets=1)
        ro = dev(np.array(c["rep_off"], np.int32)) if "rep_off" in c else None
        ri = dev(np.array(c["rep_ids"], np.int32)) if "rep_ids" in c else None
        pool.plan(dev(np.array(c["logits"], np.float32)), ro, ri)
        v = pool.view(0)
        R = T * k
        for key in ("topk_e", "gates", "phys", "slot"):
            np.testing.assert_array_equal(v[key][:T].cpu().numpy(), np.array(c[key]), err_msg=f"{c['name']}:{key}")
        for key in ("counts", "offsets"):
            np.testing.assert_array_equal(v[key].cpu().numpy(), np.array(c[key]), err_msg=f"{c['name']}:{key}")
        for key in ("src_token", "src_k"):
            np.testing.assert_array_equal(v[key][:R].cpu().numpy(), np.array(c[key]), err_msg=f"{c['name']}:{key}")
        if "x_head" in c:
            x = np.zeros((T, H), np.float32)
            for t, head in enumerate(c["x_head"]):
                x[t, :len(head)] = head
            pool.dispatch(dev_bf16(wl.f32_to_bf16_bits(x)))
            pool.identity_experts(T)
            y = wl.bf16_bits_to_f32(host_u16(pool.combine(T)))
            codes = v["codes"][:R].cpu().numpy()
            scales = v["scales"][:R, :H // 128].cpu().numpy()
            for t in range(T):
                head = c["codes_head"][t]
                for j in range(k):
                    r = c["slot"][t][j]
                    np.testing.assert_array_equal(codes[r, :len(head)], head, err_msg=f"{c['name']} codes t{t}")
                    assert not codes[r, len(head):].any()
                    assert scales[r].tolist() == c["scales"][t]
                np.testing.assert_array_equal(y[t, :len(c["y_head"][t])], c["y_head"][t], err_msg=f"{c['name']} y t{t}")
                assert not y[t, len(c["y_head"][t]):].any()
        assert pool.check() == 0

"""The expert-parallel split on one GPU, R ranks emulated as R pools and R
receive buffers, against the oracle's split (oracle.ep_forward), through the
C ABI.

Bar: receive buffers (INT8 codes, fp32 scales) and returned expert rows
bit-exact, y within 1 bf16 ulp (identical in practice: the split only moves
rows), device error word clear.  Every pull runs as one launch over all R
pullers, so no rank's kernel waits on another's.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_plan_gb300 import ep
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import assert_y_close, dev, dev_bf16, ensure_built, f32_bits, host_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _inputs(w, R, Ts=None, seed0=0):
    Ts = Ts or [w.T] * R
    out = []
    for r in range(R):
        wr = wl.dataclasses.replace(w, T=Ts[r])
        out.append(wl.make_inputs(wr, seed=seed0 + r, with_expert_out=False))
    return out


def _check(g, inps, w, recv_rows, ys, counts, ref=None, recv_ex_out=None, fused=False):
    R = g.R
    rep_off, rep_ids = inps[0]["rep_off"], inps[0]["rep_ids"]
    if ref is None:
        ref = oracle.ep_forward([i["logits"] for i in inps], [i["x"] for i in inps], w.k, w.P, rep_off, rep_ids,
                                recv_ex_out=recv_ex_out)
    np.testing.assert_array_equal(counts, ref["counts"])
    for d in range(R):
        n = recv_rows[d]
        assert n == ref["recv_codes"][d].shape[0]
        np.testing.assert_array_equal(g.recv_codes[d][:n].cpu().numpy(), ref["recv_codes"][d], err_msg=f"codes {d}")
        np.testing.assert_array_equal(f32_bits(g.recv_scales[d][:n, :w.G].cpu().numpy()),
                                      f32_bits(ref["recv_scales"][d]), err_msg=f"scales {d}")
    for s in range(R):
        rows = int(counts[s].sum())
        if not fused:  # the fused combine reads the owners' rows in place: nothing comes back to the pool
            np.testing.assert_array_equal(host_u16(g.views[s]["ex_out"][:rows]), ref["ex_out"][s],
                                          err_msg=f"ex_out {s}")
        assert_y_close(host_u16(ys[s]), ref["y"][s], f"y of rank {s}")
    assert g.check() == 0


def _group(w, R, **kw):
    return ep.EmulatedGroup(R, max(w.T, 1), w.H, w.E, w.P, w.k, **kw)


def _run(g, inps, recv_ex_out=None, fused=False, fused_dispatch=False):
    logits = [dev(i["logits"]) for i in inps]
    xs = [dev_bf16(i["x"]) for i in inps]
    ro = None if inps[0]["rep_off"] is None else dev(inps[0]["rep_off"])
    ri = None if inps[0]["rep_ids"] is None else dev(inps[0]["rep_ids"])
    rex = None if recv_ex_out is None else [dev_bf16(a) for a in recv_ex_out]
    ys, counts, recv_rows = g.step(logits, xs, ro, ri, recv_ex_out=rex, fused_combine=fused,
                                   fused_dispatch=fused_dispatch)
    torch.cuda.synchronize()
    return ys, counts, recv_rows


@pytest.mark.parametrize("mode", ["pull", "fused_combine", "fused"])
@pytest.mark.parametrize("R,T,cores,cap,S", [(1, 96, 4, (8, 8), (64, 64)), (2, 150, 3, (1, 1), (5, 7)),
                                             (3, 77, 8, (2, 1), (16, 3)), (4, 64, 16, (8, 8), (1, 1)),
                                             (5, 41, 2, (1, 1), (3, 3))])
def test_split_small_identity_experts(R, T, cores, cap, S, mode):
    """The bench workload's experts (288 physical, 32 replicas) at small
    batches: many small units, caps that bind, single-row units; both
    exchanges pulled, or the combine fused (rows read in place), or both
    fused (rows written straight into the owners' buffers, window starts
    computed on the device)."""
    w = wl.dataclasses.replace(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], T), H=1024)
    inps = _inputs(w, R)
    g = _group(w, R, cores=cores, desc_kw=dict(fanout_cap=cap, unit_rows=S))
    fused = mode != "pull"
    ys, counts, recv_rows = _run(g, inps, fused=fused, fused_dispatch=mode == "fused")
    _check(g, inps, w, recv_rows, ys, counts, fused=fused)


@pytest.mark.parametrize("mode", ["pull", "fused"])
def test_split_at_the_largest_group(mode):
    """MOE_EP_MAX_RANKS = 64 ranks of 16 tokens over the bench workload's 288
    physical experts (four or five experts a rank; the pointer tables, the
    device window starts over 64 x 288 counts and the schedules at their
    largest group)."""
    R = 64
    w = wl.dataclasses.replace(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 16), H=256)
    inps = _inputs(w, R)
    g = _group(w, R)
    ys, counts, recv_rows = _run(g, inps, fused=mode == "fused", fused_dispatch=mode == "fused")
    _check(g, inps, w, recv_rows, ys, counts, fused=mode == "fused")


def test_split_generated_expert_rows_and_ragged_batches():
    """Receivers' expert outputs are seeded bf16 rows; the ranks' batches
    differ in size, one rank's batch is empty."""
    w = wl.dataclasses.replace(wl.WORKLOADS["t16384_h2048_e64_k6"], T=300)
    R = 4
    Ts = [300, 0, 123, 31]
    inps = _inputs(w, R, Ts)
    ref0 = oracle.ep_forward([i["logits"] for i in inps], [i["x"] for i in inps], w.k, w.P)
    rng = np.random.default_rng(5)
    rex = [wl.f32_to_bf16_bits(rng.standard_normal((c.shape[0], w.H)).astype(np.float32))
           for c in ref0["recv_codes"]]
    g = ep.EmulatedGroup(R, 300, w.H, w.E, w.P, w.k, cores=6)
    ys, counts, recv_rows = _run(g, inps, rex)
    _check(g, inps, w, recv_rows, ys, counts, recv_ex_out=rex)
    ys, counts, recv_rows = _run(g, inps, rex, fused=True)
    _check(g, inps, w, recv_rows, ys, counts, recv_ex_out=rex, fused=True)
    ys, counts, recv_rows = _run(g, inps, rex, fused=True, fused_dispatch=True)
    _check(g, inps, w, recv_rows, ys, counts, recv_ex_out=rex, fused=True)


def test_split_more_ranks_than_experts_and_one_hot_expert():
    """Six ranks over four experts (two ranks own none), and every token of
    every rank routed to the same top-2 experts (one window holds all rows)."""
    w = wl.Workload("tiny", T=40, H=256, E=4, P=4, k=2)
    R = 6
    inps = _inputs(w, R)
    for i in inps:
        i["logits"][:, :] = -5.0
        i["logits"][:, 1] = 4.0
        i["logits"][:, 2] = 3.0
    g = _group(w, R, cores=3)
    for fused, fd in ((False, False), (True, False), (True, True)):
        ys, counts, recv_rows = _run(g, inps, fused=fused, fused_dispatch=fd)
        assert sorted(recv_rows) == [0, 0, 0, 0, R * w.T, R * w.T]
        _check(g, inps, w, recv_rows, ys, counts, fused=fused)


def test_split_full_bench_shape_eight_ranks():
    """Eight ranks of the bench workload (4096 tokens x 7168, 256 experts + 32
    replicas, top-8) with the default group cost model: every receive buffer,
    every returned row and every y compared in full; then the fused combine,
    and the fused dispatch with it (receive buffers filled with a pattern
    first, so that every row must be written by it), whose y must equal the
    pulled-back one bit for bit."""
    w = wl.WORKLOADS["t4096_h7168_e256p288_k8"]
    R = 8
    inps = _inputs(w, R)
    g = _group(w, R)
    ys, counts, recv_rows = _run(g, inps)
    ref = oracle.ep_forward([i["logits"] for i in inps], [i["x"] for i in inps], w.k, w.P, inps[0]["rep_off"],
                            inps[0]["rep_ids"])
    _check(g, inps, w, recv_rows, ys, counts, ref=ref)
    ys_pulled = [y.clone() for y in ys]
    for fd in (False, True):
        for t in g.recv_codes:  # the fused dispatch must write every row itself
            t.fill_(0x55)
        ys, counts, recv_rows = _run(g, inps, fused=True, fused_dispatch=fd)
        _check(g, inps, w, recv_rows, ys, counts, ref=ref, fused=True)
        for a, b in zip(ys, ys_pulled):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_one_puller_per_launch_equals_all_pullers():
    """A rank of a real group pulls only its own lists (first_puller = its
    rank, n_pullers = 1): R such launches build the same receive buffers."""
    w = wl.dataclasses.replace(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 200), H=512)
    R = 3
    inps = _inputs(w, R)
    g = _group(w, R, cores=5)
    _, _, recv_rows = _run(g, inps)
    want = [g.recv_codes[d][:recv_rows[d]].clone() for d in range(R)]
    counts = g.counts()
    for d in range(R):
        g.recv_codes[d].zero_()
        s = ep.schedule(g.desc, 0, d, counts, w.H + 4 * g.Gs)
        u, c = g.upload(ep.pack_schedules([s]))
        ep.pull(u, c, R, g.cores, d, 1, g.disp_planes, g.error_word)
    torch.cuda.synchronize()
    for d in range(R):
        assert torch.equal(g.recv_codes[d][:recv_rows[d]], want[d])
        assert int(g.recv_codes[d][recv_rows[d]:].abs().sum().item()) == 0  # nothing written past the rows
    assert g.check() == 0


def test_bad_units_are_skipped_and_reported():
    """A unit past the end of its destination buffer, one past its source
    buffer and one naming a peer outside the group are skipped by the
    kernel's own bounds checks and reported in the error word; the valid unit
    beside them still lands."""
    R, rows, H = 2, 64, 256
    src = [torch.arange(rows * H, dtype=torch.int32, device="cuda").to(torch.int8).view(rows, H) for _ in range(R)]
    dst = [torch.zeros((rows, H), dtype=torch.int8, device="cuda") for _ in range(R)]
    pl = ep.plane(src, dst, H)
    units = np.array([(1, 0, 0, 8), (0, 0, rows - 2, 4), (1, rows - 1, 0, 2), (5, 0, 0, 1)], ep.UNIT)
    u = torch.from_numpy(units.view(np.int32).reshape(-1, 4).copy()).cuda()
    core_off = torch.tensor([[0, 4], [4, 4]], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.pull(u, core_off, R, 1, 0, R, [pl], err)
    torch.cuda.synchronize()
    assert int(err.item()) == ep.DEVERR_UNIT
    assert torch.equal(dst[0][:8], src[1][:8])
    assert int(dst[0][8:].abs().sum().item()) == 0 and int(dst[1].abs().sum().item()) == 0


def test_fused_combine_rejects_rows_outside_the_owners_buffers():
    """recv_start tables that point past an owner's rows: the fused combine
    skips those tokens and reports MOE_DEVERR_UNIT; no access outside."""
    w = wl.dataclasses.replace(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 64), H=256)
    R = 2
    inps = _inputs(w, R)
    g = _group(w, R, cores=2)
    _, counts, recv_rows = _run(g, inps)
    starts = g.recv_starts(counts)
    starts[0].fill_(1 << 30)  # every expert window of rank 0 far past the end
    y = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    ep.combine(g.pools[0], w.T, g.recv_ex, recv_rows, starts[0], y)
    err = g.pools[0].check()
    assert err & ep.DEVERR_UNIT
    assert int((y.view(torch.int16) != 0).sum().item()) == 0


def test_recorded_rows_outside_the_owners_buffers_are_rejected():
    """Recorded copy rows that are -1, name an owner outside the group, or
    point past an owner's rows: the fused combine skips those tokens'
    segments and reports MOE_DEVERR_UNIT; every other token is the oracle's."""
    w = wl.dataclasses.replace(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 64), H=256)
    R = 2
    inps = _inputs(w, R)
    g = _group(w, R)
    ys, counts, recv_rows = _run(g, inps, fused=True, fused_dispatch=True)
    _check(g, inps, w, recv_rows, ys, counts, fused=True)
    rec = g.copy_rows[0].view(w.T, w.k)
    good = rec.clone()
    rec[3, 0] = -1
    rec[5, 1] = (R + 3) << 40                      # no such owner
    rec[7, 2] = (1 << 40) + g.recv_ex[1].shape[0]  # one row past owner 1's buffer
    y = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    cap = [t.shape[0] for t in g.recv_ex]
    ep.combine(g.pools[0], w.T, g.recv_ex, cap, None, y, copy_row=g.copy_rows[0])
    assert g.pools[0].check() & ep.DEVERR_UNIT
    bad = {3, 5, 7}
    yh = host_u16(y)
    assert not yh[sorted(bad)].any()
    keep = [t for t in range(w.T) if t not in bad]
    np.testing.assert_array_equal(yh[keep], host_u16(ys[0])[keep])
    g.pools[0].clear_error()
    rec.copy_(good)


def test_device_window_starts_equal_the_host_ones():
    """moe_ep_recv_start_device against moe_ep_recv_start and the rows each
    rank receives, at the bench shape and at a group with P < R."""
    for w, R in ((wl.WORKLOADS["t4096_h7168_e256p288_k8"], 8), (wl.Workload("tiny", T=30, H=128, E=4, P=4, k=2), 6)):
        w = wl.small_variant(w, min(w.T, 500))
        inps = _inputs(w, R)
        g = _group(w, R, cores=2)
        g.plan_all([dev(i["logits"]) for i in inps], None if inps[0]["rep_off"] is None else dev(inps[0]["rep_off"]),
                   None if inps[0]["rep_ids"] is None else dev(inps[0]["rep_ids"]))
        starts, rows = g.starts_device()
        counts = g.counts()
        want = np.stack([ep.recv_start(counts, s) for s in range(R)])
        np.testing.assert_array_equal(starts.cpu().numpy(), want)
        np.testing.assert_array_equal(rows.cpu().numpy(), [int(ep.layout(counts, d)[0][-1]) for d in range(R)])


def test_fused_split_as_one_cuda_graph():
    """The fully fused step needs nothing from the host, so it is captured
    once as a CUDA graph and replayed on new batches written into the same
    input tensors: every replay's y against the oracle's split with the
    expert outputs the receive buffers hold (seeded rows, fixed)."""
    w = wl.dataclasses.replace(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 200), H=512)
    R = 4
    g = _group(w, R, cores=8)
    inps = _inputs(w, R, seed0=0)
    logits = [dev(i["logits"]) for i in inps]
    xs = [dev_bf16(i["x"]) for i in inps]
    ro, ri = dev(inps[0]["rep_off"]), dev(inps[0]["rep_ids"])
    ys = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    rng = np.random.default_rng(9)
    fixed = [wl.f32_to_bf16_bits(rng.standard_normal((t.shape[0], w.H)).astype(np.float32)) for t in g.recv_ex]
    for t, a in zip(g.recv_ex, fixed):
        t.copy_(dev_bf16(a))
    graph = g.fused_step_graph(logits, xs, ys, ro, ri)
    for seed0 in (10, 20, 30):
        new = _inputs(w, R, seed0=seed0)
        for r in range(R):
            logits[r].copy_(dev(new[r]["logits"]))
            xs[r].copy_(dev_bf16(new[r]["x"]))
        ro.copy_(dev(new[0]["rep_off"]))
        ri.copy_(dev(new[0]["rep_ids"]))
        for t, a in zip(g.recv_ex, fixed):  # the experts' outputs: the same rows in place every replay
            t.copy_(dev_bf16(a))
        graph.replay()
        torch.cuda.synchronize()
        counts = g.counts()
        layouts = [ep.layout(counts, d) for d in range(R)]
        rex = [fixed[d][:int(layouts[d][0][-1])] for d in range(R)]
        ref = oracle.ep_forward([i["logits"] for i in new], [i["x"] for i in new], w.k, w.P, new[0]["rep_off"],
                                new[0]["rep_ids"], recv_ex_out=rex)
        for d in range(R):
            n = int(layouts[d][0][-1])
            np.testing.assert_array_equal(g.recv_codes[d][:n].cpu().numpy(), ref["recv_codes"][d])
        for r in range(R):
            assert_y_close(host_u16(ys[r]), ref["y"][r], f"replay {seed0} rank {r}")
    assert g.check() == 0


def test_fused_dispatch_rejects_rows_outside_the_owners_buffers():
    """Window starts past an owner's rows: the fused dispatch skips those
    copies, reports MOE_DEVERR_UNIT and writes nothing outside."""
    w = wl.dataclasses.replace(wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 64), H=256)
    R = 2
    inps = _inputs(w, R)
    g = _group(w, R, cores=2)
    g.plan_all([dev(i["logits"]) for i in inps], dev(inps[0]["rep_off"]), dev(inps[0]["rep_ids"]))
    starts, _ = g.starts_device()
    starts[0].fill_(1 << 30)
    for t in g.recv_codes:
        t.zero_()
    cap = [t.shape[0] for t in g.recv_codes]
    ep.dispatch(g.pools[0], dev_bf16(inps[0]["x"]), g.recv_codes, g.recv_scales, cap, starts[0])
    err = g.pools[0].check()
    assert err & ep.DEVERR_UNIT
    assert all(int(t.abs().sum().item()) == 0 for t in g.recv_codes)


@pytest.mark.parametrize("fused", [False, True])
def test_handworked_split_on_the_gpu(fused):
    """The split worked by hand in tests/golden/ep_handworked.json, pulled and
    fused: every owner receives the rows the fixture names, in its order (a
    token's scale names it), the device window starts are the fixture's, and
    every rank's y is the oracle's."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "ep_handworked.json")))
    R, E, P, k, H = g["R"], g["E"], g["P"], g["k"], g["H"]
    logits = [np.array(a, np.float32) for a in g["logits"]]
    xs = []
    for s in range(R):
        x = np.zeros((len(g["logits"][s]), H), np.float32)
        x[:, 0] = [1 + 4 * s + t for t in range(x.shape[0])]
        xs.append(wl.f32_to_bf16_bits(x))
    grp = ep.EmulatedGroup(R, 3, H, E, P, k, cores=2)
    ys, counts, recv_rows = grp.step([dev(a) for a in logits], [dev_bf16(a) for a in xs],
                                     fused_combine=fused, fused_dispatch=fused)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(counts, g["counts"])
    assert list(recv_rows) == g["recv_rows"]
    for d in range(R):
        want = np.array([np.float32(1 + 4 * s + t) / np.float32(127) for s, t in g["received"][d]], np.float32)
        got = grp.recv_scales[d][:recv_rows[d], 0].cpu().numpy()
        np.testing.assert_array_equal(got.view(np.int32), want.view(np.int32))
    starts, rows = grp.starts_device()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(starts.cpu().numpy(), g["recv_start"])
    assert rows.cpu().tolist() == g["recv_rows"]
    ref = oracle.ep_forward(logits, xs, k, P)
    for s in range(R):
        assert_y_close(host_u16(ys[s]), ref["y"][s], f"rank {s}")
    assert grp.check() == 0

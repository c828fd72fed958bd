"""The host side of a rank in a real expert-parallel group, as separate
processes on CPU with the gloo backend (world sizes 2 and 3).

Each rank draws its own batch and, since there is no GPU here, takes its plan
and its dispatch rows from the oracle (the stand-in for moe_plan /
moe_dispatch on its device).  What is under test is the product's host path:
ep.gather_counts (one all-gather of every rank's counts over the process
group) and ep.rank_schedules (libmoe's layout and LPT schedules).  The
schedules must equal the oracle's; executed on the host against every peer's
rows (exchanged here by all-gathers that stand in for peer memory), the
dispatch units must rebuild the oracle's receive buffer of the rank and the
combine units its returned rows, and the rank's combine its local y.  The
fused form's addressing (ep.recv_start, each copy written straight to its
owner's row, the combine reading it there) must give the same receive buffer
and the same y.
"""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_units(units, core_off, src_planes, dst):
    """Execute a schedule on the host: every core's units in list order."""
    for c in range(len(core_off) - 1):
        for u in units[core_off[c]:core_off[c + 1]]:
            q, s, d, n = (int(v) for v in (u["peer"], u["src_row"], u["dst_row"], u["rows"]))
            dst[d:d + n] = src_planes[q][s:s + n]


def _all_gather_rows(torch, dist, a):
    """Every rank's array (rows may differ): pad to the largest, all-gather, cut."""
    R = dist.get_world_size()
    n = torch.tensor([a.shape[0]], dtype=torch.int64)
    ns = [torch.zeros(1, dtype=torch.int64) for _ in range(R)]
    dist.all_gather(ns, n)
    m = max(int(v.item()) for v in ns)
    pad = np.zeros((m,) + a.shape[1:], a.dtype)
    pad[:a.shape[0]] = a
    t = torch.from_numpy(pad.view(np.uint8).reshape(m, -1).copy())
    outs = [torch.zeros_like(t) for _ in range(R)]
    dist.all_gather(outs, t)
    return [o.numpy().view(a.dtype).reshape((m,) + a.shape[1:])[:int(ns[r].item())] for r, o in enumerate(outs)]


def _worker(rank, ws, port, q):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
        sys.path.insert(0, ROOT)
        import torch
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=ws)
        import oracle
        from combine_moe_plan_gb300 import ep
        from combine_moe_plan_gb300 import workloads as wl

        base = wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 40 + 7 * rank)
        w = wl.dataclasses.replace(base, H=256)
        Ts = [40 + 7 * r for r in range(ws)]
        rep_off, rep_ids = wl.make_replica_map(w)
        inp = wl.make_inputs(w, seed=rank, with_expert_out=False)
        pl = oracle.plan(inp["logits"], w.k, rep_off, rep_ids, w.P)
        codes, scales = oracle.dispatch(inp["x"], pl["slot"])
        Gs = (w.G + 3) // 4 * 4
        scales_s = np.zeros((scales.shape[0], Gs), np.float32)
        scales_s[:, :w.G] = scales

        # the product's host path
        counts_all = ep.gather_counts(torch.from_numpy(pl["counts"].copy()))
        desc = ep.make_desc(ws, w.P, 5, fanout_cap=(1, 2), unit_rows=(3, 4), alpha_ns=(1, 3), beta_gbs=(3000, 700))
        sch = ep.rank_schedules(desc, counts_all, rank, w.H, Gs)

        # every rank's counts arrived, in rank order
        want_counts = []
        for r in range(ws):
            wr = wl.dataclasses.replace(w, T=Ts[r])
            ir = wl.make_inputs(wr, seed=r, with_expert_out=False)
            want_counts.append(oracle.plan(ir["logits"], w.k, rep_off, rep_ids, w.P)["counts"])
        np.testing.assert_array_equal(counts_all, np.stack(want_counts))

        # the schedules are the oracle's
        for key, direction, rb in (("dispatch", 0, w.H + 4 * Gs), ("combine", 1, 2 * w.H)):
            ref = oracle.ep_schedule(direction, rank, counts_all, 5, [1, 2], [3, 4], [1, 3], [3000, 700], rb)
            np.testing.assert_array_equal(sch[key]["core_off"], ref["core_off"])
            np.testing.assert_array_equal(sch[key]["units"].view(np.int32), ref["units"].view(np.int32))

        # dispatch pull, executed against every peer's rows
        peers_codes = _all_gather_rows(torch, dist, codes)
        peers_scales = _all_gather_rows(torch, dist, scales_s)
        n_recv = int(sch["expert_off"][-1])
        recv_codes = np.zeros((n_recv, w.H), np.int8)
        recv_scales = np.zeros((n_recv, Gs), np.float32)
        u, co = sch["dispatch"]["units"], sch["dispatch"]["core_off"]
        _run_units(u, co, peers_codes, recv_codes)
        _run_units(u, co, peers_scales, recv_scales)
        np.testing.assert_array_equal(recv_codes, oracle.ep_gather(peers_codes, counts_all, rank))
        np.testing.assert_array_equal(recv_scales[:, :w.G].view(np.int32),
                                      oracle.ep_gather([s[:, :w.G] for s in peers_scales], counts_all,
                                                       rank).view(np.int32))

        # experts on the receive rows, then the combine pull and the local combine
        recv_ex = oracle.identity_experts(recv_codes, recv_scales[:, :w.G])
        peers_ex = _all_gather_rows(torch, dist, recv_ex)
        ex_out = np.zeros((int(counts_all[rank].sum()), w.H), np.uint16)
        _run_units(sch["combine"]["units"], sch["combine"]["core_off"], peers_ex, ex_out)
        loc = oracle.forward(inp["logits"], inp["x"], w.k, rep_off, rep_ids, w.P)
        np.testing.assert_array_equal(ex_out, loc["ex_out"])
        y = oracle.combine(ex_out, pl["slot"], pl["gates"])
        np.testing.assert_array_equal(y, loc["y"])

        # the fused form: this rank's window starts in every owner's buffer
        # from every rank's counts (the product's host call), each copy
        # written straight to row start[p] + slot - offsets[p] of its owner,
        # and the combine reading each copy's expert row there
        starts = np.asarray(ep.recv_start(counts_all, rank), np.int64)
        slot_f, phys_f = pl["slot"].reshape(-1).astype(np.int64), pl["phys"].reshape(-1).astype(np.int64)
        owner_f = (phys_f * ws) // w.P
        dst_f = starts[phys_f] + slot_f - pl["offsets"][phys_f].astype(np.int64)
        meta = _all_gather_rows(torch, dist, np.stack([owner_f, dst_f], 1))
        payload = _all_gather_rows(torch, dist, codes[slot_f])
        recv_fused = np.full((n_recv, w.H), 0x55, np.int8)
        for mr, pr in zip(meta, payload):
            mine = mr[:, 0] == rank
            recv_fused[mr[mine, 1]] = pr[mine]
        np.testing.assert_array_equal(recv_fused, recv_codes)
        rows_f = np.stack([peers_ex[int(o)][int(d)] for o, d in zip(owner_f, dst_f)]) if len(dst_f) else \
            np.zeros((0, w.H), np.uint16)
        ex_f = np.zeros_like(ex_out)
        ex_f[slot_f] = rows_f
        np.testing.assert_array_equal(oracle.combine(ex_f, pl["slot"], pl["gates"]), loc["y"])

        # what each rank pulls from a peer is what that peer's window holds for it
        pulled = np.zeros(ws, np.int64)
        for x in sch["dispatch"]["units"]:
            pulled[int(x["peer"])] += int(x["rows"])
        first, cnt = ep.experts(ws, w.P, rank)
        np.testing.assert_array_equal(pulled, counts_all[:, first:first + cnt].sum(axis=1))
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # report to the parent instead of hanging it
        import traceback
        q.put((rank, traceback.format_exc() + repr(e)))


@pytest.mark.parametrize("ws", [2, 3])
def test_rank_host_path_gloo(ws):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    for rank, msg in res:
        assert msg == "ok", f"rank {rank}: {msg}"
    for p in procs:
        assert p.exitcode == 0

"""ctypes binding of libmoe's expert-parallel split (include/moe_ep.h), and
the group drivers built on it.

Argument marshalling and plumbing only: the transfer schedule is libmoe's
host code (C++), every data movement runs in libmoe's CUDA kernels, and
torch supplies device memory, streams and, for a group spread over
processes, torch.distributed (the all-gather of the per-expert counts every
rank needs to lay out and schedule its pulls).

  EmulatedGroup   R ranks on one GPU: R pools, R receive buffers, each
                  exchange one moe_ep_pull launch for all R pullers.
  gather_counts,  the host side of a rank in a real group: every rank's
  rank_schedules  counts by one all-gather, then this rank's dispatch and
                  combine schedules.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import moe

MAX_RANKS = 64
DEVERR_UNIT = 0x8
HEADER = os.path.join(os.path.dirname(moe.HEADER), "moe_ep.h")

i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p

UNIT = np.dtype([("peer", np.int32), ("src_row", np.int32), ("dst_row", np.int32), ("rows", np.int32)])


class EpDesc(ctypes.Structure):
    _fields_ = [("R", i32), ("P", i32), ("cores", i32), ("fanout_cap", i32 * 2), ("unit_rows", i32 * 2),
                ("alpha_ns", i64 * 2), ("beta_gbs", i64 * 2)]


class Plane(ctypes.Structure):
    _fields_ = [("src", vp * MAX_RANKS), ("dst", vp * MAX_RANKS), ("src_rows", i64 * MAX_RANKS),
                ("dst_rows", i64 * MAX_RANKS), ("row_bytes", i64)]


_bound = False


def lib():
    global _bound
    L = moe.lib()
    if not _bound:
        pp = ctypes.POINTER
        sig = {
            "moe_ep_experts": [i32, i32, i32, pp(i32), pp(i32)],
            "moe_ep_layout": [i32, i32, vp, i32, vp, vp],
            "moe_ep_max_units": [pp(EpDesc), i64, pp(i32)],
            "moe_ep_schedule": [pp(EpDesc), i32, i32, vp, i64, vp, i32, pp(i32), vp, pp(i64)],
            "moe_ep_schedule_group": [pp(EpDesc), i32, vp, i64, vp, i32, pp(i32), vp, vp],
            "moe_ep_pull": [vp, vp, i32, i32, i32, i32, i32, pp(Plane), i32, vp, vp],
            "moe_dequant_rows": [vp, vp, i32, i32, i32, vp, vp],
            "moe_ep_recv_start": [i32, i32, vp, i32, vp],
            "moe_ep_recv_start_device": [i32, i32, pp(vp), vp, vp, vp],
            "moe_ep_dispatch": [vp, vp, i32, ctypes.c_int, i32, pp(vp), pp(vp), pp(i64), vp, vp, vp],
            "moe_ep_combine": [vp, i32, ctypes.c_int, i32, pp(vp), pp(i64), vp, vp, vp, vp],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        _bound = True
    return L


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != moe.MOE_OK:
        raise moe.MoeError(name, rc, lib().moe_status_str(rc).decode())


def _np_ptr(a):
    return a.ctypes.data_as(vp)


def make_desc(R, P, cores, fanout_cap=None, unit_rows=(64, 64), alpha_ns=(1, 2), beta_gbs=(6000, 900)):
    """A group and its cost model: tier 0 = the puller's own memory, tier 1 = a
    peer's.  The defaults model one GB300 (about 6 TB/s to its own HBM) and
    NVLink (about 900 GB/s per direction to a peer).  The default fan-out cap
    leaves the puller's own memory unlimited and lets ceil(cores / R) cores
    work on one peer per stripe: R peers x that cap cover every core.  (A cap
    with R * H_t < cores leaves cores that never receive a unit: at most
    R * H_t cores can hold a unit in any stripe.)"""
    if fanout_cap is None:
        fanout_cap = (cores, max(1, -(-cores // max(R, 1))))
    return EpDesc(R, P, cores, (i32 * 2)(*fanout_cap), (i32 * 2)(*unit_rows), (i64 * 2)(*alpha_ns),
                  (i64 * 2)(*beta_gbs))


def experts(R, P, d):
    """(first, count): rank d owns physical experts first .. first+count-1."""
    first, count = i32(), i32()
    _call("moe_ep_experts", R, P, d, ctypes.byref(first), ctypes.byref(count))
    return first.value, count.value


def layout(counts, d):
    """Receive layout of rank d from every rank's counts [R, P] (host):
    (expert_off [n_d + 1], chunk_row [R, n_d])."""
    counts = np.ascontiguousarray(counts, np.int32)
    R, P = counts.shape
    _, nd = experts(R, P, d)
    off = np.zeros(nd + 1, np.int32)
    chunk = np.zeros((R, nd), np.int32)
    _call("moe_ep_layout", R, P, _np_ptr(counts), d, _np_ptr(off), _np_ptr(chunk))
    return off, chunk


def max_units(desc, rows):
    n = i32()
    _call("moe_ep_max_units", ctypes.byref(desc), int(rows), ctypes.byref(n))
    return n.value


def schedule(desc, direction, puller, counts, row_bytes, cap_units=None):
    """The LPT transfer schedule of one puller (host): dict with units (UNIT
    records grouped by core), core_off [cores + 1] and makespan (ps)."""
    counts = np.ascontiguousarray(counts, np.int32)
    if cap_units is None:
        cap_units = max_units(desc, int(counts.sum()))
    units = np.zeros(max(1, cap_units), UNIT)
    core_off = np.zeros(desc.cores + 1, np.int32)
    n, ms = i32(), i64()
    _call("moe_ep_schedule", ctypes.byref(desc), direction, puller, _np_ptr(counts), int(row_bytes), _np_ptr(units),
          cap_units, ctypes.byref(n), _np_ptr(core_off), ctypes.byref(ms))
    return {"units": units[:n.value].copy(), "core_off": core_off, "makespan": ms.value}


def schedule_group(desc, direction, counts, row_bytes):
    """The schedules of all R pullers, packed by libmoe (host threads):
    (units [n, 4] int32, core_off [R, cores + 1] int32 absolute, makespans [R])."""
    counts = np.ascontiguousarray(counts, np.int32)
    cap = desc.R * max_units(desc, int(counts.sum()))
    units = np.empty(max(1, cap), UNIT)
    core_off = np.zeros((desc.R, desc.cores + 1), np.int32)
    ms = np.zeros(desc.R, np.int64)
    n = i32()
    _call("moe_ep_schedule_group", ctypes.byref(desc), direction, _np_ptr(counts), int(row_bytes), _np_ptr(units),
          cap, ctypes.byref(n), _np_ptr(core_off), _np_ptr(ms))
    return units[:n.value].view(np.int32).reshape(-1, 4).copy(), core_off, ms


def plane(src, dst, row_bytes, src_rows=None, dst_rows=None) -> Plane:
    """A plane from per-rank device tensors (None for ranks taking no part);
    rows default to each tensor's first dimension."""
    p = Plane()
    for q, t in enumerate(src):
        if t is not None:
            p.src[q] = t.data_ptr()
            p.src_rows[q] = t.shape[0] if src_rows is None else src_rows[q]
    for r, t in enumerate(dst):
        if t is not None:
            p.dst[r] = t.data_ptr()
            p.dst_rows[r] = t.shape[0] if dst_rows is None else dst_rows[r]
    p.row_bytes = int(row_bytes)
    return p


def pull(units, core_off, R, cores, first_puller, n_pullers, planes, error_word, stream=None):
    """moe_ep_pull.  units: device int32 tensor [n, 4] (UNIT records);
    core_off: device int32 tensor [n_pullers, cores + 1] of absolute indices."""
    arr = (Plane * len(planes))(*planes)
    _call("moe_ep_pull", units.data_ptr() if units.numel() else None, core_off.data_ptr(), units.shape[0], R, cores,
          first_puller, n_pullers, arr, len(planes), error_word.data_ptr(), moe._stream(stream))


def recv_start(counts, s):
    """First row of rank s's window of every physical expert in its owner's
    receive buffer (host int32 [P])."""
    counts = np.ascontiguousarray(counts, np.int32)
    R, P = counts.shape
    out = np.zeros(P, np.int32)
    _call("moe_ep_recv_start", R, P, _np_ptr(counts), s, _np_ptr(out))
    return out


def recv_start_device(counts_dev, recv_start_dev, recv_rows_dev=None, stream=None):
    """moe_ep_recv_start_device: every rank's window starts [R, P] (and rows
    received [R]) from the ranks' device counts, computed on the device."""
    R = len(counts_dev)
    P = counts_dev[0].shape[0]
    ptrs = (vp * R)(*[t.data_ptr() for t in counts_dev])
    _call("moe_ep_recv_start_device", R, P, ptrs, recv_start_dev.data_ptr(),
          None if recv_rows_dev is None else recv_rows_dev.data_ptr(), moe._stream(stream))


def dispatch(pool, x, recv_codes, recv_scales, recv_rows, recv_start_dev, buf=0, stream=None, copy_row=None):
    """moe_ep_dispatch: the rank's tokens quantized and written straight into
    the owners' receive buffers; with copy_row (device int64 [T, k]) where
    each copy went is recorded for moe_ep_combine."""
    R = len(recv_codes)
    cp = (vp * R)(*[None if t is None else t.data_ptr() for t in recv_codes])
    sp = (vp * R)(*[None if t is None else t.data_ptr() for t in recv_scales])
    rows = (i64 * R)(*[int(r) for r in recv_rows])
    _call("moe_ep_dispatch", pool.handle, x.data_ptr() if x.numel() else None, x.shape[0], buf, R, cp, sp, rows,
          recv_start_dev.data_ptr(), None if copy_row is None else copy_row.data_ptr(), moe._stream(stream))


def combine(pool, T, recv_ex, recv_rows, recv_start_dev, y, buf=0, stream=None, copy_row=None):
    """moe_ep_combine: rank's y [T, H] straight from the owners' receive buffers
    (recv_ex: per-rank bf16 device tensors, recv_rows: rows each holds); with
    copy_row, the rows its moe_ep_dispatch recorded (recv_start_dev may then be
    None)."""
    R = len(recv_ex)
    ptrs = (vp * R)(*[None if t is None else t.data_ptr() for t in recv_ex])
    rows = (i64 * R)(*[int(r) for r in recv_rows])
    _call("moe_ep_combine", pool.handle, int(T), buf, R, ptrs, rows,
          None if recv_start_dev is None else recv_start_dev.data_ptr(),
          None if copy_row is None else copy_row.data_ptr(), y.data_ptr(), moe._stream(stream))


def dequant_rows(codes, scales, rows, out, stream=None):
    """moe_dequant_rows: out[:rows] = bf16(codes * scale) (identity experts on any buffer)."""
    _call("moe_dequant_rows", codes.data_ptr(), scales.data_ptr(), int(rows), codes.shape[1], scales.shape[1],
          out.data_ptr(), moe._stream(stream))


def pack_schedules(scheds):
    """Concatenate per-puller schedules into one host array each: units [n, 4]
    int32 and core_off [n_pullers, cores + 1] int32 with absolute indices."""
    base, us, offs = 0, [], []
    for s in scheds:
        us.append(s["units"])
        offs.append(s["core_off"] + base)
        base += len(s["units"])
    units = np.concatenate(us) if base else np.zeros(0, UNIT)
    return units.view(np.int32).reshape(-1, 4), np.stack(offs).astype(np.int32)


# ---------------------------------------------- a rank of a real group --

def gather_counts(counts, group=None) -> np.ndarray:
    """Every rank's counts [R, P] on the host, by one all-gather of this
    rank's counts (an int32 tensor [P] on the process group's device)."""
    import torch.distributed as dist
    R = dist.get_world_size(group)
    out = [torch.empty_like(counts) for _ in range(R)]
    dist.all_gather(out, counts.contiguous(), group=group)
    return torch.stack(out).cpu().numpy()


def rank_schedules(desc, counts_all, rank, H, scale_stride):
    """This rank's two schedules from every rank's counts: dispatch (it pulls
    its experts' INT8 rows and scales) and combine (it pulls its bf16 rows
    back), plus its receive layout."""
    disp = schedule(desc, 0, rank, counts_all, H + 4 * scale_stride)
    comb = schedule(desc, 1, rank, counts_all, 2 * H)
    off, chunk = layout(counts_all, rank)
    return {"dispatch": disp, "combine": comb, "expert_off": off, "chunk_row": chunk}


# ------------------------------------------- a group emulated on one GPU --

class EmulatedGroup:
    """R ranks of an expert-parallel group on one GPU.  Rank r has its own
    pool (moe.Pool, one buffer set), a receive buffer sized for the worst case
    (every rank sending every row to r: R * T_max * k rows) and a stream of its
    own, on which its kernels run (forked from the caller's stream and joined
    back to it).  Pulled exchanges run as one moe_ep_pull launch over all R
    pullers; the fused forms run each rank's moe_ep_dispatch and
    moe_ep_combine on its own stream.

    Every peer buffer is in this GPU's memory, so by default both tiers of the
    cost model are the local one (alpha 1 ns, 6000 GB/s) and no fan-out cap
    binds: the schedules then balance the bytes the cores really move.  Pass
    desc_kw to schedule for another machine's tiers instead."""

    LOCAL_TIERS = dict(alpha_ns=(1, 1), beta_gbs=(6000, 6000))

    def __init__(self, R, T_max, H, E, P, k, cores=None, desc_kw=None, device="cuda"):
        self.R, self.T_max, self.H, self.E, self.P, self.k = R, T_max, H, E, P, k
        self.device = torch.device(device)
        if cores is None:
            sms = torch.cuda.get_device_properties(self.device).multi_processor_count
            cores = max(1, (4 * sms) // R)  # one wave of 512-thread CTAs over all pullers
        self.cores = cores
        kw = dict(self.LOCAL_TIERS, fanout_cap=(cores, cores))
        kw.update(desc_kw or {})
        self.desc = make_desc(R, P, cores, **kw)
        self.pools = [moe.Pool(T_max, H, E, P, k, n_sets=1, device=device) for _ in range(R)]
        self.views = [p.view(0) for p in self.pools]
        self.Gs = self.views[0]["scales"].shape[1]
        cap = R * T_max * k
        self.recv_codes = [torch.empty((cap, H), dtype=torch.int8, device=device) for _ in range(R)]
        self.recv_scales = [torch.empty((cap, self.Gs), dtype=torch.float32, device=device) for _ in range(R)]
        self.recv_ex = [torch.empty((cap, H), dtype=torch.bfloat16, device=device) for _ in range(R)]
        # where each rank's fused dispatch sent each copy (owner * 2^40 + row), for its fused combine
        self.copy_rows = [torch.empty((T_max * k,), dtype=torch.int64, device=device) for _ in range(R)]
        self.error_word = torch.zeros(1, dtype=torch.int32, device=device)
        self._counts_host = torch.zeros((R, P), dtype=torch.int32).pin_memory()
        self._starts = torch.empty((R, P), dtype=torch.int32, device=device)
        self._rows = torch.empty(R, dtype=torch.int32, device=device)
        self.disp_planes = [plane([v["codes"] for v in self.views], self.recv_codes, H),
                            plane([v["scales"] for v in self.views], self.recv_scales, 4 * self.Gs)]
        self.comb_planes = [plane(self.recv_ex, [v["ex_out"] for v in self.views], 2 * H)]
        # one stream per rank (created here, never inside a capture)
        self._rank_streams = [torch.cuda.Stream(device=self.device) for _ in range(R)]

    def _per_rank(self, stream, fn):
        """fn(r, s_r) for every rank r, each on its own stream s_r forked from
        `stream` and joined back to it: the emulated ranks' kernels run side
        by side, as the ranks of a real group do on their own GPUs."""
        s = stream or torch.cuda.current_stream(self.device)
        fork = torch.cuda.Event()
        fork.record(s)
        out = []
        for r, st in enumerate(self._rank_streams):
            st.wait_event(fork)
            out.append(fn(r, st))
        for st in self._rank_streams:
            s.wait_stream(st)
        return out

    def plan_dispatch(self, logits, xs, rep_off=None, rep_ids=None, stream=None):
        """Every rank's plan, the counts on their way to the host, then every
        rank's dispatch.  Returns an event that completes once the counts are
        in host memory (read them with counts_host()): the host can schedule
        while the dispatch kernels run."""
        s = stream or torch.cuda.current_stream(self.device)
        self.plan_all(logits, rep_off, rep_ids, s)
        with torch.cuda.stream(s):
            for r, v in enumerate(self.views):
                self._counts_host[r].copy_(v["counts"], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(s)
        # the kernel before each dispatch is not its own plan: the default form
        self._per_rank(s, lambda r, st: self.pools[r].dispatch(xs[r], stream=st))
        return ev

    def counts_host(self, ev) -> np.ndarray:
        """Every rank's counts [R, P], once `ev` (from plan_dispatch) completed."""
        ev.synchronize()
        return self._counts_host.numpy().copy()

    def counts(self) -> np.ndarray:
        """Every rank's counts [R, P] on the host (synchronizes)."""
        return torch.stack([v["counts"] for v in self.views]).cpu().numpy()

    def schedules(self, counts):
        """Host schedules of both exchanges for all R pullers, packed:
        (dispatch units, core_off), (combine units, core_off), recv rows."""
        H, Gs = self.H, self.Gs
        disp = schedule_group(self.desc, 0, counts, H + 4 * Gs)[:2]  # each on libmoe's worker threads
        comb = schedule_group(self.desc, 1, counts, 2 * H)[:2]
        owner = (np.arange(self.P, dtype=np.int64) * self.R) // self.P
        recv_rows = np.bincount(owner, weights=counts.sum(axis=0), minlength=self.R).astype(np.int64).tolist()
        return disp, comb, [int(v) for v in recv_rows]

    def upload(self, packed, stream=None):
        """Host schedule arrays -> device tensors, copied on `stream`."""
        units, core_off = packed
        s = stream or torch.cuda.current_stream(self.device)
        with torch.cuda.stream(s):
            u = torch.from_numpy(units).pin_memory().to(self.device, non_blocking=True)
            c = torch.from_numpy(core_off).pin_memory().to(self.device, non_blocking=True)
        return u, c

    def pull_dispatch(self, units, core_off, stream=None):
        pull(units, core_off, self.R, self.cores, 0, self.R, self.disp_planes, self.error_word, stream)

    def pull_combine(self, units, core_off, stream=None):
        pull(units, core_off, self.R, self.cores, 0, self.R, self.comb_planes, self.error_word, stream)

    def identity_experts(self, recv_rows, stream=None):
        def one(d, st):
            if recv_rows[d]:
                dequant_rows(self.recv_codes[d], self.recv_scales[d], recv_rows[d], self.recv_ex[d], st)
        self._per_rank(stream, one)

    def _outputs(self, T_list, stream):
        """Every rank's y [T, H], allocated on `stream` (the one they are
        handed back on)."""
        with torch.cuda.stream(stream or torch.cuda.current_stream(self.device)):
            return [torch.empty((T, self.H), dtype=torch.bfloat16, device=self.device) for T in T_list]

    def combine(self, T_list, ys=None, stream=None):
        ys = ys or self._outputs(T_list, stream)
        self._per_rank(stream, lambda r, st: self.pools[r].combine(T_list[r], y=ys[r], stream=st))
        return ys

    def recv_starts(self, counts, stream=None):
        """Every rank's recv_start table [R, P] on the device (copied on `stream`)."""
        tab = np.stack([recv_start(counts, s) for s in range(self.R)])
        s = stream or torch.cuda.current_stream(self.device)
        with torch.cuda.stream(s):
            return torch.from_numpy(tab).pin_memory().to(self.device, non_blocking=True)

    def combine_fused(self, T_list, recv_rows, starts, ys=None, stream=None, recorded=False):
        """Every rank's y straight from the owners' receive buffers (no
        combine pull): moe_ep_combine per rank.  With `recorded`, each copy's
        row is the one the rank's fused dispatch recorded (dispatch_fused);
        otherwise it is found from the plan and the window starts."""
        ys = ys or self._outputs(T_list, stream)
        self._per_rank(stream, lambda r, st: combine(self.pools[r], T_list[r], self.recv_ex, recv_rows, starts[r],
                                                      ys[r], stream=st,
                                                      copy_row=self.copy_rows[r] if recorded else None))
        return ys

    def plan_all(self, logits, rep_off=None, rep_ids=None, stream=None):
        """Every rank's plan.  The plans are independent and latency-bound, so
        they run side by side on R streams forked from `stream` and joined
        back to it (as the ranks of a real group plan at the same time)."""
        self._per_rank(stream, lambda r, st: self.pools[r].plan(logits[r], rep_off, rep_ids, stream=st))

    def starts_device(self, stream=None):
        """Every rank's window starts [R, P] and rows received [R], computed on
        the device from the plans' counts (moe_ep_recv_start_device)."""
        recv_start_device([v["counts"] for v in self.views], self._starts, self._rows, stream)
        return self._starts, self._rows

    def dispatch_fused(self, xs, starts, stream=None):
        """Every rank's fused dispatch into the owners' receive buffers,
        recording where each copy went (copy_rows)."""
        cap = [t.shape[0] for t in self.recv_codes]
        self._per_rank(stream, lambda r, st: dispatch(self.pools[r], xs[r], self.recv_codes, self.recv_scales, cap,
                                                       starts[r], stream=st, copy_row=self.copy_rows[r]))

    def step(self, logits, xs, rep_off=None, rep_ids=None, recv_ex_out=None, stream=None, fused_combine=False,
             fused_dispatch=False):
        """The whole split path: plan + dispatch on every rank, counts to the
        host, schedules, the dispatch pull, the experts (identity experts on
        the receive buffers unless recv_ex_out[d] gives each receiver's bf16
        rows), the combine pull, and every rank's combine -- or, with
        fused_combine, every rank's moe_ep_combine straight from the owners'
        receive buffers instead of the combine pull and moe_combine.  With
        fused_dispatch (which implies fused_combine) the window starts are
        computed on the device and every rank's moe_ep_dispatch writes its rows
        straight into the owners' buffers: no schedule, no pull and no host
        round trip (only the identity experts read the rows received back).
        Returns the per-rank y, the counts and the rows each rank received."""
        if fused_dispatch:
            return self._step_fused(logits, xs, rep_off, rep_ids, recv_ex_out, stream)
        ev = self.plan_dispatch(logits, xs, rep_off, rep_ids, stream)
        counts = self.counts_host(ev)
        disp, comb, recv_rows = self.schedules(counts)
        du, dc = self.upload(disp, stream)
        cu, cc = self.upload(comb, stream)
        self.pull_dispatch(du, dc, stream)
        if recv_ex_out is None:
            self.identity_experts(recv_rows, stream)
        else:
            for d in range(self.R):
                self.recv_ex[d][:recv_rows[d]].copy_(recv_ex_out[d])
        T_list = [lg.shape[0] for lg in logits]
        if fused_combine:
            ys = self.combine_fused(T_list, recv_rows, self.recv_starts(counts, stream), stream=stream)
        else:
            self.pull_combine(cu, cc, stream)
            ys = self.combine(T_list, stream=stream)
        return ys, counts, recv_rows

    def _step_fused(self, logits, xs, rep_off, rep_ids, recv_ex_out, stream):
        self.plan_all(logits, rep_off, rep_ids, stream)
        starts, rows_dev = self.starts_device(stream)
        self.dispatch_fused(xs, starts, stream)
        recv_rows = [int(v) for v in rows_dev.cpu().tolist()] if recv_ex_out is None else None
        if recv_ex_out is None:
            self.identity_experts(recv_rows, stream)
        else:
            for d in range(self.R):
                self.recv_ex[d][:recv_ex_out[d].shape[0]].copy_(recv_ex_out[d])
        cap = [t.shape[0] for t in self.recv_ex]
        T_list = [lg.shape[0] for lg in logits]
        ys = self.combine_fused(T_list, cap, starts, stream=stream, recorded=True)
        counts = self.counts()
        if recv_rows is None:
            recv_rows = [int(v) for v in rows_dev.cpu().tolist()]
        return ys, counts, recv_rows

    def fused_step_graph(self, logits, xs, ys, rep_off=None, rep_ids=None, stream=None):
        """The fully fused step (plans, device window starts, fused dispatch,
        fused combine into ys) captured once as a CUDA graph: it reads no
        counts on the host, so one replay runs the whole split.  The expert
        outputs are whatever the receive buffers hold.  Replays read the
        current contents of logits, xs and the replica map."""
        s = stream or torch.cuda.Stream(device=self.device)
        cap = [t.shape[0] for t in self.recv_ex]
        T_list = [lg.shape[0] for lg in logits]

        def body():
            self.plan_all(logits, rep_off, rep_ids, s)
            starts, _ = self.starts_device(s)
            self.dispatch_fused(xs, starts, s)
            self.combine_fused(T_list, cap, starts, ys=ys, stream=s, recorded=True)

        with torch.cuda.stream(s):
            body()  # warm (module loads, attributes) outside the capture
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            body()
        return g

    def check(self) -> int:
        """Synchronize; the pull error word OR every pool's error word."""
        torch.cuda.synchronize(self.device)
        w = int(self.error_word.item())
        for p in self.pools:
            w |= p.check()
        return w

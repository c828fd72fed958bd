"""CPU oracle for MoE FusedDispatch / FusedCombine (numpy front end).

TEST INFRASTRUCTURE ONLY: tests, the smoke check and the bench's CPU-baseline
leg are the only callers.  The product path (the CUDA library and its Python
binding) never imports this package, and this package imports nothing from
the product.  The arithmetic lives in ``moe_oracle.c`` (plain loops); this
file compiles it with gcc and marshals numpy arrays.

Every step follows the CloudMatrix384 write-up, section "FusedDispatch and
FusedCombine" (routing metadata, early INT8 quantization with a scale,
token-level load -> quantize/address -> write, expert output return), with the
placement order of the StrataCL analysis, section 3.5 (token placement ->
expert-window aggregation).  The expert-parallel split over R ranks
(``moe_oracle_ep.c``: ownership, receive layout, pull exchanges, and the
transfer schedule of section 3.5 -- peer-window partition into units, LPT
under a per-peer fan-out cap) is wrapped by the ``ep_*`` functions below.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SRC_EP = os.path.join(_HERE, "moe_oracle_ep.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {0: "ok", -1: "bad argument", -2: "malformed replica map",
          -3: "token routed twice to one physical expert", -4: "non-finite input"}


class OracleError(RuntimeError):
    pass


_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc, ISO C11, no FP
    contraction), with OpenMP for the per-token loops where gcc has it."""
    os.makedirs(_LIBDIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_SRC_EP))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        r = subprocess.run(["gcc", *_FLAGS, "-fopenmp", "-o", tmp, _SRC, _SRC_EP, "-lm"], capture_output=True)
        if r.returncode != 0:  # no OpenMP runtime: the same loops, serial
            subprocess.run(["gcc", *_FLAGS, "-o", tmp, _SRC, _SRC_EP, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            lib.orc_route.argtypes = [P, i32, i32, i32, P, P, i32, P, P, P]
            lib.orc_place.argtypes = [P, i32, i32, i32, P, P, P, P, P]
            lib.orc_quantize.argtypes = [P, i32, i32, P, P]
            lib.orc_dispatch.argtypes = [P, i32, i32, i32, P, i32, P, P]
            lib.orc_identity_experts.argtypes = [P, P, i32, i32, P]
            lib.orc_combine.argtypes = [P, i32, i32, i32, P, P, i32, P]
            lib.orc_combine_tokens.argtypes = [P, i32, i32, i32, P, P, P, i32, P]
            lib.orc_f32_to_bf16_array.argtypes = [P, ctypes.c_int64, P]
            lib.orc_set_threads.argtypes = [ctypes.c_int]
            lib.orc_set_threads.restype = ctypes.c_int
            for f in ("orc_route", "orc_place", "orc_quantize", "orc_dispatch",
                      "orc_identity_experts", "orc_combine", "orc_combine_tokens"):
                getattr(lib, f).restype = ctypes.c_int
            lib.orc_f32_to_bf16_array.restype = None
            i64 = ctypes.c_int64
            lib.orc_ep_owner.argtypes = [i32, i32, i32]
            lib.orc_ep_owner.restype = i32
            lib.orc_ep_layout.argtypes = [P, i32, i32, i32, P, P, P]
            lib.orc_ep_gather.argtypes = [P, i64, P, i32, i32, i32, P]
            lib.orc_ep_return.argtypes = [P, i64, P, i32, i32, i32, P]
            lib.orc_ep_schedule.argtypes = [i32, i32, P, i32, i32, i32, P, P, P, P, i64, i32, P, P, P, P, P]
            for f in ("orc_ep_layout", "orc_ep_gather", "orc_ep_return", "orc_ep_schedule"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def set_threads(n: int = 0) -> int:
    """Threads for the per-token loops (n < 1: keep the current setting).
    Returns the count now in force (1 when built without OpenMP)."""
    return int(_load().orc_set_threads(int(n)))


def threads() -> int:
    return set_threads(0)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc):
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"error {rc}"))


def route(logits, k, rep_off=None, rep_ids=None, P=None):
    """Top-k + gates + replica pick.  Returns (topk_e, gates, phys), each [T, k]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    P = E if P is None else P
    rep_off, rep_ids = _c(rep_off, np.int32), _c(rep_ids, np.int32)
    topk_e = np.empty((T, k), np.int32)
    gates = np.empty((T, k), np.float32)
    phys = np.empty((T, k), np.int32)
    _check(_load().orc_route(_p(logits), T, E, k, _p(rep_off), _p(rep_ids), P,
                             _p(topk_e), _p(gates), _p(phys)))
    return topk_e, gates, phys


def place(phys, P):
    """Counting sort into expert windows.  Returns dict of counts, offsets,
    slot [T,k], src_token [T*k], src_k [T*k]."""
    phys = _c(phys, np.int32)
    T, k = phys.shape
    out = {"counts": np.empty(P, np.int32), "offsets": np.empty(P + 1, np.int32),
           "slot": np.empty((T, k), np.int32), "src_token": np.empty(T * k, np.int32),
           "src_k": np.empty(T * k, np.int32)}
    _check(_load().orc_place(_p(phys), T, k, P, _p(out["counts"]), _p(out["offsets"]),
                             _p(out["slot"]), _p(out["src_token"]), _p(out["src_k"])))
    return out


def plan(logits, k, rep_off=None, rep_ids=None, P=None):
    topk_e, gates, phys = route(logits, k, rep_off, rep_ids, P)
    P = logits.shape[1] if P is None else P
    out = place(phys, P)
    out.update(topk_e=topk_e, gates=gates, phys=phys)
    return out


def quantize(x):
    """Per-token, per-128 group INT8 quantization.  Returns (codes [T,H], scales [T,G])."""
    x = _c(x, np.uint16)
    T, H = x.shape
    codes = np.empty((T, H), np.int8)
    scales = np.empty((T, H // 128), np.float32)
    _check(_load().orc_quantize(_p(x), T, H, _p(codes), _p(scales)))
    return codes, scales


def dispatch(x, slot, rows=None):
    """Quantize and scatter into slot rows.  Returns (codes [R,H], scales [R,G]).
    Rows no token lands in keep the fill value (codes 0, scales NaN)."""
    x = _c(x, np.uint16)
    slot = _c(slot, np.int32)
    T, H = x.shape
    k = slot.shape[1]
    R = T * k if rows is None else rows
    codes = np.zeros((R, H), np.int8)
    scales = np.full((R, H // 128), np.nan, np.float32)
    _check(_load().orc_dispatch(_p(x), T, H, k, _p(slot), R, _p(codes), _p(scales)))
    return codes, scales


def identity_experts(codes, scales):
    codes = _c(codes, np.int8)
    scales = _c(scales, np.float32)
    R, H = codes.shape
    out = np.empty((R, H), np.uint16)
    _check(_load().orc_identity_experts(_p(codes), _p(scales), R, H, _p(out)))
    return out


def combine(ex_out, slot, gates):
    ex_out = _c(ex_out, np.uint16)
    slot = _c(slot, np.int32)
    gates = _c(gates, np.float32)
    R, H = ex_out.shape
    T, k = slot.shape
    y = np.empty((T, H), np.uint16)
    _check(_load().orc_combine(_p(ex_out), R, H, k, _p(slot), _p(gates), T, _p(y)))
    return y


def combine_tokens(ex_out, slot, gates, tokens):
    """Combine only the listed tokens (rows of y in the order given)."""
    ex_out = _c(ex_out, np.uint16)
    slot = _c(slot, np.int32)
    gates = _c(gates, np.float32)
    tok = _c(tokens, np.int32)
    R, H = ex_out.shape
    k = slot.shape[1]
    y = np.empty((len(tok), H), np.uint16)
    _check(_load().orc_combine_tokens(_p(ex_out), R, H, k, _p(slot), _p(gates), _p(tok),
                                      len(tok), _p(y)))
    return y


def f32_to_bf16(a):
    a = _c(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    _load().orc_f32_to_bf16_array(_p(a), a.size, _p(out))
    return out


def forward(logits, x, k, rep_off=None, rep_ids=None, P=None, ex_out=None):
    """The whole path: plan, dispatch, experts (identity unless ex_out is
    given), combine.  Returns a dict with every intermediate."""
    out = plan(logits, k, rep_off, rep_ids, P)
    codes, scales = dispatch(x, out["slot"])
    if ex_out is None:
        ex_out = identity_experts(codes, scales)
    out.update(codes=codes, scales=scales, ex_out=ex_out,
               y=combine(ex_out, out["slot"], out["gates"]))
    return out


# ------------------------------------------------- expert-parallel split --

EP_UNIT = np.dtype([("peer", np.int32), ("src_row", np.int32), ("dst_row", np.int32), ("rows", np.int32)])


def ep_owner(p, R, P) -> int:
    """Rank that owns physical expert p: floor(p * R / P)."""
    return int(_load().orc_ep_owner(int(p), int(R), int(P)))


def ep_layout(counts, d):
    """Receive layout of rank d from every rank's counts [R, P]: returns
    (expert_off [n_d + 1], chunk_row [R, n_d]); expert_off[-1] is the number
    of rows d receives."""
    counts = _c(counts, np.int32)
    R, P = counts.shape
    n = ctypes.c_int32()
    off = np.zeros(P + 1, np.int32)
    chunk = np.zeros(R * P, np.int32)
    _check(_load().orc_ep_layout(_p(counts), R, P, int(d), ctypes.byref(n), _p(off), _p(chunk)))
    nd = n.value
    return off[:nd + 1].copy(), chunk[:R * nd].reshape(R, nd).copy()


def _planes(arrs):
    arrs = [np.ascontiguousarray(a) for a in arrs]
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return arrs, ptrs


def _row_bytes(a):
    """Bytes per row from the shape (an empty array's strides may be 0)."""
    return int(a.dtype.itemsize * int(np.prod(a.shape[1:], dtype=np.int64)))


def ep_gather(pools, counts, d):
    """Dispatch exchange of one plane: pools[s] is rank s's plane [rows, ...]
    (expert-major windows); returns rank d's receive plane."""
    counts = _c(counts, np.int32)
    R, P = counts.shape
    arrs, ptrs = _planes(pools)
    row_bytes = _row_bytes(arrs[0])
    off, _ = ep_layout(counts, d)
    out = np.zeros((int(off[-1]),) + arrs[0].shape[1:], arrs[0].dtype)
    _check(_load().orc_ep_gather(ptrs, row_bytes, _p(counts), R, P, int(d), _p(out)))
    return out


def ep_return(recvs, counts, s, rows):
    """Combine exchange of one plane: recvs[d] is rank d's receive plane;
    returns rank s's pool plane with `rows` rows (rows no copy lands in are 0)."""
    counts = _c(counts, np.int32)
    R, P = counts.shape
    arrs, ptrs = _planes(recvs)
    row_bytes = _row_bytes(arrs[0])
    out = np.zeros((rows,) + arrs[0].shape[1:], arrs[0].dtype)
    _check(_load().orc_ep_return(ptrs, row_bytes, _p(counts), R, P, int(s), _p(out)))
    return out


def ep_schedule(direction, puller, counts, C, cap, unit_rows, alpha_ns, beta_gbs, row_bytes, max_units=None):
    """LPT transfer schedule of one puller.  Returns dict with units (EP_UNIT
    records grouped by core), cost [n] (ps), core_off [C+1], makespan (ps)."""
    counts = _c(counts, np.int32)
    R, P = counts.shape
    if max_units is None:
        max_units = int(R * P + counts.sum() // max(1, min(unit_rows)) + 1)
    units = np.zeros(max_units, EP_UNIT)
    cost = np.zeros(max_units, np.int64)
    core_off = np.zeros(C + 1, np.int32)
    n = ctypes.c_int32()
    ms = ctypes.c_int64()
    a = [np.ascontiguousarray(v, t) for v, t in ((cap, np.int32), (unit_rows, np.int32), (alpha_ns, np.int64),
                                                 (beta_gbs, np.int64))]
    _check(_load().orc_ep_schedule(int(direction), int(puller), _p(counts), R, P, int(C), *[_p(v) for v in a],
                                   int(row_bytes), int(max_units), _p(units), _p(cost), ctypes.byref(n),
                                   _p(core_off), ctypes.byref(ms)))
    return {"units": units[:n.value].copy(), "cost": cost[:n.value].copy(), "core_off": core_off,
            "makespan": ms.value}


def ep_forward(logits_list, x_list, k, P=None, rep_off=None, rep_ids=None, recv_ex_out=None):
    """The whole path split over R = len(logits_list) ranks: each rank plans
    and dispatches its own batch into its own pool, the owners gather their
    experts' rows (codes and scales), the experts run on the receive buffers
    (identity experts unless recv_ex_out[d] gives bf16 rows), the rows return
    to their sources, and each rank combines its own tokens.  Returns a dict
    with per-rank lists: plan, codes, scales, counts [R, P], recv_codes,
    recv_scales, recv_ex_out, ex_out (returned rows), y."""
    R = len(logits_list)
    E = logits_list[0].shape[1]
    P = E if P is None else P
    plans = [plan(lg, k, rep_off, rep_ids, P) for lg in logits_list]
    disp = [dispatch(x, pl["slot"]) for x, pl in zip(x_list, plans)]
    counts = np.stack([pl["counts"] for pl in plans])
    recv_codes = [ep_gather([c for c, _ in disp], counts, d) for d in range(R)]
    recv_scales = [ep_gather([s for _, s in disp], counts, d) for d in range(R)]
    if recv_ex_out is None:
        recv_ex_out = [identity_experts(c, s) for c, s in zip(recv_codes, recv_scales)]
    ex_out = [ep_return(recv_ex_out, counts, s, int(plans[s]["offsets"][-1])) for s in range(R)]
    y = [combine(ex_out[s], plans[s]["slot"], plans[s]["gates"]) for s in range(R)]
    return {"plan": plans, "codes": [c for c, _ in disp], "scales": [s for _, s in disp], "counts": counts,
            "recv_codes": recv_codes, "recv_scales": recv_scales, "recv_ex_out": recv_ex_out,
            "ex_out": ex_out, "y": y}

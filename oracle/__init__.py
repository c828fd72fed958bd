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
expert-window aggregation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
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
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        r = subprocess.run(["gcc", *_FLAGS, "-fopenmp", "-o", tmp, _SRC, "-lm"], capture_output=True)
        if r.returncode != 0:  # no OpenMP runtime: the same loops, serial
            subprocess.run(["gcc", *_FLAGS, "-o", tmp, _SRC, "-lm"], check=True)
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

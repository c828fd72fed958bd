"""ctypes binding of libmoe (include/moe.h).

Argument marshalling only: torch tensors supply device pointers and the
current stream; every step of the path runs in libmoe's CUDA kernels.  The
library must have been built (``__graft_entry__.build()`` or
``python -m combine_moe_plan_gb300.build``); if it is missing, loading raises
``LibraryMissing`` -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "moe.h")

MOE_OK = 0
STATUS = {0: "MOE_OK", -1: "MOE_ERR_NULL", -2: "MOE_ERR_SIZE", -3: "MOE_ERR_ALIGN", -4: "MOE_ERR_BUF",
          -5: "MOE_ERR_WORKSPACE", -6: "MOE_ERR_CUDA", -7: "MOE_ERR_DEVICE", -8: "MOE_ERR_REPLICA",
          -9: "MOE_ERR_STATE"}
DEVERR_REPLICA, DEVERR_DUPLICATE, DEVERR_SLOT = 0x1, 0x2, 0x4


class LibraryMissing(ImportError):
    pass


class MoeError(RuntimeError):
    def __init__(self, fn, rc, msg):
        super().__init__(f"{fn}: {STATUS.get(rc, rc)} ({msg})")
        self.rc = rc


class Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T_max", "H", "E", "P", "k", "group", "n_sets")]


class View(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("codes", "scales", "ex_out", "topk_e", "phys", "gates", "slot",
                                              "src_token", "src_k", "counts", "offsets", "error_word")] + \
               [("rows", ctypes.c_int32), ("scale_stride", ctypes.c_int32)]


_lib = None
_lib_path = LIB_PATH


def use_library(path: str) -> None:
    """Choose which build of the library this process loads (e.g. the trace
    build, libmoe_trace.so).  Must be called before the first call into it."""
    global _lib_path
    if _lib is not None and path != _lib_path:
        raise RuntimeError(f"{_lib_path} is already loaded in this process")
    _lib_path = path


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_lib_path):
        raise LibraryMissing(f"{_lib_path} is not built; run combine_moe_plan_gb300.build.build()")
    L = ctypes.CDLL(_lib_path)
    vp, i32, pp = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER
    sig = {
        "moe_pool_bytes": [pp(Desc), pp(ctypes.c_size_t)],
        "moe_pool_init": [pp(Desc), vp, ctypes.c_size_t, pp(vp)],
        "moe_pool_destroy": [vp],
        "moe_pool_view": [vp, ctypes.c_int, pp(View)],
        "moe_pool_clear_error": [vp, vp],
        "moe_pool_check": [vp, vp, pp(i32)],
        "moe_pool_launches": [vp, pp(ctypes.c_uint64)],
        "moe_replica_check": [vp, vp, i32, i32],
        "moe_plan": [vp, vp, i32, vp, vp, ctypes.c_int, vp],
        "moe_dispatch": [vp, vp, i32, ctypes.c_int, vp],
        "moe_dispatch_after_plan": [vp, vp, i32, ctypes.c_int, vp],
        "moe_plan_dispatch": [vp, vp, i32, vp, vp, vp, ctypes.c_int, vp],
        "moe_identity_experts": [vp, i32, ctypes.c_int, vp],
        "moe_combine": [vp, vp, vp, i32, ctypes.c_int, vp],
        "moe_step_host": [vp, vp, vp, vp, vp, i32, vp, vp, ctypes.c_int, vp],
        "moe_plan_static": [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    L.moe_status_str.argtypes = [ctypes.c_int]
    L.moe_status_str.restype = ctypes.c_char_p
    _lib = L
    return L


def header_functions(path: str = HEADER) -> list[str]:
    """Names of every function a header (default include/moe.h) declares."""
    src = open(path).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != MOE_OK:
        raise MoeError(name, rc, lib().moe_status_str(rc).decode())
    return rc


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def pool_bytes(T_max, H, E, P, k, n_sets=2) -> int:
    d = Desc(T_max, H, E, P, k, 128, n_sets)
    n = ctypes.c_size_t()
    _call("moe_pool_bytes", ctypes.byref(d), ctypes.byref(n))
    return n.value


def replica_check(rep_off, rep_ids, E, P) -> int:
    """Host check of a CSR replica map (numpy or CPU tensors); returns the status."""
    import numpy as np
    off = np.ascontiguousarray(rep_off, np.int32)
    ids = np.ascontiguousarray(rep_ids, np.int32)
    return lib().moe_replica_check(off.ctypes.data_as(ctypes.c_void_p), ids.ctypes.data_as(ctypes.c_void_p),
                                   E, P)


class Pool:
    """A static dispatch/combine buffer pool over one device workspace.

    The workspace is one torch uint8 tensor of ``pool_bytes`` bytes; views
    into it (codes, scales, ex_out, plan metadata) are exposed as tensors."""

    def __init__(self, T_max, H, E, P, k, n_sets=2, device="cuda", stream=None):
        self.desc = Desc(T_max, H, E, P, k, 128, n_sets)
        self.T_max, self.H, self.E, self.P, self.k, self.n_sets = T_max, H, E, P, k, n_sets
        self.nbytes = pool_bytes(T_max, H, E, P, k, n_sets)
        self.workspace = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        h = ctypes.c_void_p()
        _call("moe_pool_init", ctypes.byref(self.desc), _ptr(self.workspace), self.nbytes, ctypes.byref(h))
        self.handle = h
        _call("moe_pool_clear_error", self.handle, _stream(stream))

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _lib is not None:
            _lib.moe_pool_destroy(h)
            self.handle = None

    # -- views ---------------------------------------------------------------
    def view(self, buf=0) -> dict:
        v = View()
        _call("moe_pool_view", self.handle, buf, ctypes.byref(v))
        base = self.workspace.data_ptr()
        R, H, T, k, P = v.rows, self.H, self.T_max, self.k, self.P

        def t(addr, dtype, shape):
            n = 1
            for s in shape:
                n *= s
            nb = n * torch.empty((), dtype=dtype).element_size()
            off = addr - base
            return self.workspace[off:off + nb].view(dtype).view(*shape)

        return {
            "codes": t(v.codes, torch.int8, (R, H)),
            "scales": t(v.scales, torch.float32, (R, v.scale_stride)),
            "ex_out": t(v.ex_out, torch.bfloat16, (R, H)),
            "topk_e": t(v.topk_e, torch.int32, (T, k)),
            "phys": t(v.phys, torch.int32, (T, k)),
            "gates": t(v.gates, torch.float32, (T, k)),
            "slot": t(v.slot, torch.int32, (T, k)),
            "src_token": t(v.src_token, torch.int32, (R,)),
            "src_k": t(v.src_k, torch.int32, (R,)),
            "counts": t(v.counts, torch.int32, (P,)),
            "offsets": t(v.offsets, torch.int32, (P + 1,)),
            "error_word": t(v.error_word, torch.int32, (1,)),
        }

    # -- calls ---------------------------------------------------------------
    def plan(self, logits, rep_off=None, rep_ids=None, buf=0, stream=None):
        T = logits.shape[0]
        _call("moe_plan", self.handle, _ptr(logits), T, _ptr(rep_off), _ptr(rep_ids), buf, _stream(stream))
        return T

    def dispatch(self, x, buf=0, stream=None, after_plan=False):
        """moe_dispatch; with ``after_plan`` moe_dispatch_after_plan, which
        reads x before waiting for the kernel just before it: only right after
        this set's plan on the same stream, with x written before that plan."""
        fn = "moe_dispatch_after_plan" if after_plan else "moe_dispatch"
        _call(fn, self.handle, _ptr(x), x.shape[0], buf, _stream(stream))

    def plan_dispatch(self, logits, x, rep_off=None, rep_ids=None, buf=0, stream=None):
        """moe_plan_dispatch: plan and dispatch as one call; the dispatch
        reads x while the plan runs, which the call makes safe."""
        T = logits.shape[0]
        if x.shape[0] != T:
            raise ValueError("logits and x must have the same number of tokens")
        _call("moe_plan_dispatch", self.handle, _ptr(logits), T, _ptr(rep_off), _ptr(rep_ids), _ptr(x), buf,
              _stream(stream))
        return T

    def identity_experts(self, T, buf=0, stream=None):
        _call("moe_identity_experts", self.handle, T, buf, _stream(stream))

    def combine(self, T, y=None, ex_out=None, buf=0, stream=None):
        if y is None:
            y = torch.empty((T, self.H), dtype=torch.bfloat16, device=self.workspace.device)
        _call("moe_combine", self.handle, _ptr(ex_out), _ptr(y), T, buf, _stream(stream))
        return y

    def step_host(self, h_logits, h_x, h_y, h_ex_out=None, rep_off=None, rep_ids=None, buf=0, stream=None):
        """Whole layer from host tensors (pinned for asynchronous copies)."""
        _call("moe_step_host", self.handle, _ptr(h_logits), _ptr(h_x), _ptr(h_ex_out), _ptr(h_y),
              h_x.shape[0], _ptr(rep_off), _ptr(rep_ids), buf, _stream(stream))

    def clear_error(self, stream=None):
        _call("moe_pool_clear_error", self.handle, _stream(stream))

    def check(self, stream=None) -> int:
        """Synchronize and return the device error word (0 = clean)."""
        w = ctypes.c_int32()
        rc = lib().moe_pool_check(self.handle, _stream(stream), ctypes.byref(w))
        if rc not in (MOE_OK, -7):
            raise MoeError("moe_pool_check", rc, lib().moe_status_str(rc).decode())
        return w.value

    def launches(self) -> int:
        n = ctypes.c_uint64()
        _call("moe_pool_launches", self.handle, ctypes.byref(n))
        return n.value


def plan_static(logits, k, P=None, rep_off=None, rep_ids=None, out=None, stream=None) -> dict:
    """moe_plan_static: routing metadata into caller-owned tensors, with no
    device allocation inside the library (its scratch is a fixed 4 MiB array
    in the library's device image).  ``out`` may hold preallocated tensors
    (topk_e, gates, phys, counts, offsets, slot, src_token, src_k,
    error_word); missing ones are allocated here by torch, outside the call."""
    T, E = logits.shape
    P = E if P is None else P
    dev = logits.device
    shapes = {"topk_e": ((T, k), torch.int32), "gates": ((T, k), torch.float32), "phys": ((T, k), torch.int32),
              "counts": ((P,), torch.int32), "offsets": ((P + 1,), torch.int32), "slot": ((T, k), torch.int32),
              "src_token": ((T * k,), torch.int32), "src_k": ((T * k,), torch.int32),
              "error_word": ((1,), torch.int32)}
    out = dict(out or {})
    for name, (shape, dtype) in shapes.items():
        if name not in out:
            out[name] = (torch.zeros if name == "error_word" else torch.empty)(shape, dtype=dtype, device=dev)
    _call("moe_plan_static", _ptr(logits), T, E, P, k, _ptr(rep_off), _ptr(rep_ids),
          *[_ptr(out[n]) for n in ("topk_e", "gates", "phys", "counts", "offsets", "slot", "src_token", "src_k",
                                    "error_word")], _stream(stream))
    return out

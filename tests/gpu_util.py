"""Shared helpers for the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C ABI, and compare with the oracle."""
import numpy as np
import torch

from combine_moe_plan_gb300 import build as moe_build
from combine_moe_plan_gb300 import moe


def ensure_built():
    moe_build.build()
    moe.lib()


def dev_bf16(a_u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).cuda().view(torch.bfloat16)


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def f32_bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, np.float32).view(np.int32)


def ulp_dist_f32(a, b) -> np.ndarray:
    """Distance in binary32 ulps between finite values (ordered-integer map)."""
    def ordered(x):
        i = f32_bits(x).astype(np.int64)
        return np.where(i < 0, -(i & 0x7FFFFFFF), i)
    return np.abs(ordered(a) - ordered(b))


def ulp_dist_bf16(a_u16, b_u16) -> np.ndarray:
    def ordered(x):
        i = np.asarray(x, np.uint16).astype(np.int64)
        return np.where(i >= 0x8000, -(i & 0x7FFF), i)
    return np.abs(ordered(a_u16) - ordered(b_u16))


def assert_gates_close(g_gpu, g_ref, what=""):
    """Gates are exp/sum/divide in fp64 rounded once to fp32 on both sides; the
    two fp64 exp implementations may differ by an fp64 ulp, so a value that sits
    within ~2^-50 of an fp32 rounding midpoint may round the other way: allow
    1 fp32 ulp on at most a handful of entries."""
    d = ulp_dist_f32(g_gpu, g_ref)
    assert d.max() <= 1, f"{what}: gate differs by {d.max()} ulp"
    assert (d > 0).sum() <= max(2, d.size // 100000), f"{what}: {(d > 0).sum()} gates differ"


def assert_y_close(y_gpu, y_ref, what=""):
    """Combine output within 1 bf16 ulp (identical unless a gate differed)."""
    d = ulp_dist_bf16(y_gpu, y_ref)
    assert d.shape == np.shape(y_ref), f"{what}: shape {d.shape} against {np.shape(y_ref)}"
    if d.size == 0:  # an empty batch
        return 0
    assert d.max() <= 1, f"{what}: y differs by {d.max()} bf16 ulp"
    return int((d > 0).sum())


class Run:
    """One pass of the CUDA path over a workload's seeded inputs."""

    def __init__(self, w, inp, T_max=None, n_sets=2, ex_out=None, buf=0, pool=None, fused=False):
        self.w = w
        T = inp["logits"].shape[0]
        self.T = T
        self.pool = pool or moe.Pool(T_max or T, w.H, w.E, w.P, w.k, n_sets=n_sets)
        self.logits = dev(inp["logits"])
        self.x = dev_bf16(inp["x"])
        self.rep_off = None if inp["rep_off"] is None else dev(inp["rep_off"])
        self.rep_ids = None if inp["rep_ids"] is None else dev(inp["rep_ids"])
        self.buf = buf
        p = self.pool
        if fused:  # moe_plan_dispatch
            p.plan_dispatch(self.logits, self.x, self.rep_off, self.rep_ids, buf=buf)
        else:
            p.plan(self.logits, self.rep_off, self.rep_ids, buf=buf)
            p.dispatch(self.x, buf=buf)
        self.v = p.view(buf)
        if ex_out is None:
            p.identity_experts(T, buf=buf)
            self.y = p.combine(T, buf=buf)
        else:
            self.ex = dev_bf16(ex_out)
            self.y = p.combine(T, ex_out=self.ex, buf=buf)
        self.err = p.check()

    def plan_host(self):
        T, k, R = self.T, self.w.k, self.T * self.w.k
        v = self.v
        return {"topk_e": v["topk_e"][:T].cpu().numpy(), "gates": v["gates"][:T].cpu().numpy(),
                "phys": v["phys"][:T].cpu().numpy(), "slot": v["slot"][:T].cpu().numpy(),
                "counts": v["counts"].cpu().numpy(), "offsets": v["offsets"].cpu().numpy(),
                "src_token": v["src_token"][:R].cpu().numpy(), "src_k": v["src_k"][:R].cpu().numpy()}


def compare_plan(gpu, ref, what=""):
    for key in ("topk_e", "phys", "counts", "offsets", "slot", "src_token", "src_k"):
        np.testing.assert_array_equal(gpu[key], ref[key], err_msg=f"{what}: {key}")
    assert_gates_close(gpu["gates"], ref["gates"], what)

"""moe_dispatch reads x only after waiting for the kernel before it.

A foreign kernel (tests/pdl_writer.cu, built here with nvcc) is enqueued
between moe_plan and moe_dispatch on the same stream.  It is launched with
programmatic dependent launch, lets its dependents start at once, and only
after a delay overwrites x with another batch.  moe_dispatch, the default
call, must quantize the new x: its codes and scales equal the oracle's for
the new activations, bit for bit.  moe_dispatch_after_plan is the opt-in that
reads x before the wait; its precondition excludes exactly this sequence, so
it is not run here.  moe_plan_dispatch reads both the logits and x after its
wait: foreign kernels that overwrite both right before it are covered too.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from combine_moe_plan_gb300 import moe
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import dev, dev_bf16, ensure_built, f32_bits

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def writer(tmp_path_factory):
    ensure_built()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("pdlw") / "libpdl_writer.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    "-cudart", "static", os.path.join(ROOT, "tests", "pdl_writer.cu"), "-o", out], check=True)
    L = ctypes.CDLL(out)
    L.pdl_write.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong,
                            ctypes.c_void_p]
    L.pdl_write.restype = ctypes.c_int
    return L


@pytest.mark.parametrize("name,T", [("t96_h7168_e256_k8", 96), ("t4096_h7168_e256p288_k8", 300)])
def test_foreign_kernel_writing_x_between_plan_and_dispatch(writer, name, T):
    w = wl.small_variant(wl.WORKLOADS[name], T)
    inp_old = wl.make_inputs(w, seed=0, with_expert_out=False)
    inp_new = wl.make_inputs(w, seed=1, with_expert_out=False)
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=1)
    logits = dev(inp_old["logits"])
    ro = None if inp_old["rep_off"] is None else dev(inp_old["rep_off"])
    ri = None if inp_old["rep_ids"] is None else dev(inp_old["rep_ids"])
    x = dev_bf16(inp_old["x"])
    x_new = dev_bf16(inp_new["x"])
    ref = oracle.plan(inp_old["logits"], w.k, inp_old["rep_off"], inp_old["rep_ids"], w.P)
    codes, scales = oracle.dispatch(inp_new["x"], ref["slot"])
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for rnd in range(5):
            x.copy_(dev_bf16(inp_old["x"]))  # back to the old batch before every round
            pool.plan(logits, ro, ri, stream=s)
            rc = writer.pdl_write(ctypes.c_void_p(x_new.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                                  x.numel() * 2, 20000, ctypes.c_void_p(s.cuda_stream))
            assert rc == 0
            pool.dispatch(x, stream=s)
            s.synchronize()
            v = pool.view(0)
            R = w.T * w.k
            np.testing.assert_array_equal(v["codes"][:R].cpu().numpy(), codes, err_msg=f"round {rnd}: codes")
            np.testing.assert_array_equal(f32_bits(v["scales"][:R, :w.G].cpu().numpy()), f32_bits(scales),
                                          err_msg=f"round {rnd}: scales")
    assert pool.check() == 0


@pytest.mark.parametrize("name,T", [("t96_h7168_e256_k8", 96), ("t4096_h7168_e256p288_k8", 300),
                                    ("t4096_h7168_e256p288_k8", 600)])
def test_foreign_kernels_writing_inputs_before_plan_dispatch(writer, name, T):
    """moe_plan_dispatch reads logits and x only after its wait: two foreign
    kernels enqueued right before it overwrite the logits and x with another
    batch (each letting its dependents start before it writes), and its plan,
    codes and scales are the oracle's for the new batch (the dispatch loads x
    early, but only once the plan's own wait for those kernels has returned):
    cluster plans at 96 and 300 tokens, three launches at 600."""
    w = wl.small_variant(wl.WORKLOADS[name], T)
    inp_old = wl.make_inputs(w, seed=0, with_expert_out=False)
    inp_new = wl.make_inputs(w, seed=1, with_expert_out=False)
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=1)
    # the replica map of the new batch's seed for both (it follows the seed)
    ro = None if inp_new["rep_off"] is None else dev(inp_new["rep_off"])
    ri = None if inp_new["rep_ids"] is None else dev(inp_new["rep_ids"])
    logits, x = dev(inp_old["logits"]), dev_bf16(inp_old["x"])
    logits_new, x_new = dev(inp_new["logits"]), dev_bf16(inp_new["x"])
    ref = oracle.plan(inp_new["logits"], w.k, inp_new["rep_off"], inp_new["rep_ids"], w.P)
    codes, scales = oracle.dispatch(inp_new["x"], ref["slot"])
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for rnd in range(5):
            logits.copy_(dev(inp_old["logits"]))
            x.copy_(dev_bf16(inp_old["x"]))
            for src, dst in ((logits_new, logits), (x_new, x)):
                rc = writer.pdl_write(ctypes.c_void_p(src.data_ptr()), ctypes.c_void_p(dst.data_ptr()),
                                      dst.numel() * dst.element_size(), 20000, ctypes.c_void_p(s.cuda_stream))
                assert rc == 0
            pool.plan_dispatch(logits, x, ro, ri, stream=s)
            s.synchronize()
            v = pool.view(0)
            R = w.T * w.k
            np.testing.assert_array_equal(v["slot"][: w.T].cpu().numpy(), ref["slot"], err_msg=f"round {rnd}: slot")
            np.testing.assert_array_equal(v["codes"][:R].cpu().numpy(), codes, err_msg=f"round {rnd}: codes")
            np.testing.assert_array_equal(f32_bits(v["scales"][:R, :w.G].cpu().numpy()), f32_bits(scales),
                                          err_msg=f"round {rnd}: scales")
    assert pool.check() == 0

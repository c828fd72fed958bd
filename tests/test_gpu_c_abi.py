"""The C ABI on its own: tests/c_abi_step.c drives a whole step (workspace and
buffers from cudaMalloc, moe_pool_init, moe_plan, moe_dispatch, the identity
experts, moe_combine, moe_pool_check) with nothing but include/moe.h and the
CUDA runtime; its slots and y must equal the oracle's.  tests/c_abi_ep_step.c
does the same for the fully fused expert-parallel split through
include/moe_ep.h."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import assert_y_close, ensure_built

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    ensure_built()
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    cuda_lib = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.exists(os.path.join(d, "libcudart.so")))
    out = str(tmp_path_factory.mktemp("cabi") / "c_abi_step")
    libdir = os.path.join(ROOT, "combine_moe_plan_gb300", "_lib")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", f"-I{os.path.join(ROOT, 'include')}",
                    f"-I{os.path.join(cuda, 'include')}", os.path.join(ROOT, "tests", "c_abi_step.c"), "-o", out,
                    f"-L{libdir}", "-l:libmoe.so", f"-L{cuda_lib}", "-lcudart",
                    f"-Wl,-rpath,{libdir}:{cuda_lib}"], check=True)
    return out


@pytest.mark.parametrize("name,T", [("t4096_h7168_e256p288_k8", 300), ("t96_h7168_e256_k8", 96)])
def test_c_program_step_matches_oracle(exe, tmp_path, name, T):
    w = wl.small_variant(wl.WORKLOADS[name], T)
    inp = wl.make_inputs(w)
    has_rep = inp["rep_off"] is not None
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(fin, "wb") as f:
        f.write(np.array([w.T, w.H, w.E, w.P, w.k, int(has_rep)], np.int32).tobytes())
        f.write(np.ascontiguousarray(inp["logits"], np.float32).tobytes())
        f.write(np.ascontiguousarray(inp["x"], np.uint16).tobytes())
        if has_rep:
            f.write(np.ascontiguousarray(inp["rep_off"], np.int32).tobytes())
            f.write(np.ascontiguousarray(inp["rep_ids"], np.int32).tobytes())
    r = subprocess.run([exe, str(fin), str(fout)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, f"c_abi_step failed at step {r.returncode}: {r.stderr}"
    raw = open(fout, "rb").read()
    n_slot, n_y = w.T * w.k, w.T * w.H
    slot = np.frombuffer(raw, np.int32, n_slot).reshape(w.T, w.k)
    y = np.frombuffer(raw, np.uint16, n_y, offset=4 * n_slot).reshape(w.T, w.H)
    err = int(np.frombuffer(raw, np.int32, 1, offset=4 * n_slot + 2 * n_y)[0])
    ref = oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"], w.P)
    assert err == 0
    np.testing.assert_array_equal(slot, ref["slot"])
    assert_y_close(y, ref["y"], f"{name} from C")


@pytest.fixture(scope="module")
def exe_ep(tmp_path_factory):
    ensure_built()
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    cuda_lib = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                    if os.path.exists(os.path.join(d, "libcudart.so")))
    out = str(tmp_path_factory.mktemp("cabi_ep") / "c_abi_ep_step")
    libdir = os.path.join(ROOT, "combine_moe_plan_gb300", "_lib")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", f"-I{os.path.join(ROOT, 'include')}",
                    f"-I{os.path.join(cuda, 'include')}", os.path.join(ROOT, "tests", "c_abi_ep_step.c"), "-o", out,
                    f"-L{libdir}", "-l:libmoe.so", f"-L{cuda_lib}", "-lcudart",
                    f"-Wl,-rpath,{libdir}:{cuda_lib}"], check=True)
    return out


@pytest.mark.parametrize("name,T,R", [("t96_h7168_e256_k8", 96, 3), ("t4096_h7168_e256p288_k8", 300, 4)])
def test_c_program_fused_split_matches_oracle(exe_ep, tmp_path, name, T, R):
    """tests/c_abi_ep_step.c runs the fully fused split of R ranks from plain
    C (include/moe_ep.h: device window starts, fused dispatch recording each
    copy's row, identity experts on the receive buffers, fused combine from
    the recorded rows); the rows each owner received and every rank's y must
    be the oracle's split."""
    w = wl.small_variant(wl.WORKLOADS[name], T)
    inps = [wl.make_inputs(w, seed=r, with_expert_out=False) for r in range(R)]
    has_rep = inps[0]["rep_off"] is not None
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(fin, "wb") as f:
        f.write(np.array([R, w.T, w.H, w.E, w.P, w.k, int(has_rep)], np.int32).tobytes())
        for i in inps:
            f.write(np.ascontiguousarray(i["logits"], np.float32).tobytes())
            f.write(np.ascontiguousarray(i["x"], np.uint16).tobytes())
        if has_rep:
            f.write(np.ascontiguousarray(inps[0]["rep_off"], np.int32).tobytes())
            f.write(np.ascontiguousarray(inps[0]["rep_ids"], np.int32).tobytes())
    r = subprocess.run([exe_ep, str(fin), str(fout)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, f"c_abi_ep_step failed at step {r.returncode}: {r.stderr}"
    raw = open(fout, "rb").read()
    rows = np.frombuffer(raw, np.int32, R)
    n_y = w.T * w.H
    ys = [np.frombuffer(raw, np.uint16, n_y, offset=4 * R + 2 * n_y * s).reshape(w.T, w.H) for s in range(R)]
    err = int(np.frombuffer(raw, np.int32, 1, offset=4 * R + 2 * n_y * R)[0])
    ref = oracle.ep_forward([i["logits"] for i in inps], [i["x"] for i in inps], w.k, w.P, inps[0]["rep_off"],
                            inps[0]["rep_ids"])
    assert err == 0
    assert rows.tolist() == [c.shape[0] for c in ref["recv_codes"]]
    for s in range(R):
        assert_y_close(ys[s], ref["y"][s], f"{name} rank {s} from C")

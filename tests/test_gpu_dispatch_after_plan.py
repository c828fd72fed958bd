"""moe_dispatch_after_plan right after moe_plan: x loaded and quantized
while the plan still runs, the slots read after the wait for it.

Every form of the one-cluster plan (tiles of 8, 16 and 32 tokens; 1, 8 and
16 CTAs) and every batch boundary up to 512 tokens, one after the other on
one set, against the oracle; then ten plans and dispatches on one set back to
back with no synchronization, where the last call's rows must be its own.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_plan_gb300 import moe
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import compare_plan, dev, dev_bf16, ensure_built, f32_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _check(pool, w, inp, buf=0):
    ref = oracle.plan(inp["logits"], w.k, inp["rep_off"], inp["rep_ids"], w.P)
    v = pool.view(buf)
    T, R = inp["logits"].shape[0], inp["logits"].shape[0] * w.k
    got = {"topk_e": v["topk_e"][:T].cpu().numpy(), "gates": v["gates"][:T].cpu().numpy(),
           "phys": v["phys"][:T].cpu().numpy(), "slot": v["slot"][:T].cpu().numpy(),
           "counts": v["counts"].cpu().numpy(), "offsets": v["offsets"].cpu().numpy(),
           "src_token": v["src_token"][:R].cpu().numpy(), "src_k": v["src_k"][:R].cpu().numpy()}
    compare_plan(got, ref)
    codes, scales = oracle.dispatch(inp["x"], ref["slot"])
    np.testing.assert_array_equal(v["codes"][:R].cpu().numpy(), codes)
    np.testing.assert_array_equal(f32_bits(v["scales"][:R, :w.G].cpu().numpy()), f32_bits(scales))


def test_every_cluster_tile_size_and_boundary():
    """1 to 512 tokens (tiles of 8, 16 and 32 tokens; 1, 8, 16 tiles) on one
    set, each call checked."""
    base = wl.dataclasses.replace(wl.WORKLOADS["t4096_h7168_e256p288_k8"], H=512)
    pool = moe.Pool(512, base.H, base.E, base.P, base.k, n_sets=1)
    for T in (1, 7, 8, 9, 63, 64, 65, 96, 127, 128, 129, 255, 256, 257, 300, 511, 512):
        w = wl.dataclasses.replace(base, T=T)
        inp = wl.make_inputs(w, seed=T, with_expert_out=False)
        pool.plan(dev(inp["logits"]), dev(inp["rep_off"]), dev(inp["rep_ids"]))
        pool.dispatch(dev_bf16(inp["x"]), after_plan=True)
        torch.cuda.synchronize()
        _check(pool, w, inp)
    assert pool.check() == 0


def test_back_to_back_calls_rearm_the_flags():
    """Ten plans and dispatches on one set with no synchronization in
    between, each with its own batch; the last one's rows must be its own."""
    w = wl.WORKLOADS["t96_h7168_e256_k8"]
    pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=1)
    inps = [wl.make_inputs(w, seed=50 + i, with_expert_out=False) for i in range(10)]
    args = [(dev(i["logits"]), dev_bf16(i["x"])) for i in inps]
    torch.cuda.synchronize()
    for logits, x in args:
        pool.plan(logits)
        pool.dispatch(x, after_plan=True)
    torch.cuda.synchronize()
    _check(pool, w, inps[-1])
    assert pool.check() == 0

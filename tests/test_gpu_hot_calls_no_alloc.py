"""The hot calls never allocate device memory: the pool is carved from a
caller-owned workspace at init, and plan, dispatch, the expert stand-in and
combine only use it.  After warm-up calls (the first launch of a kernel loads
its module), 50 more steps leave the device's free memory
unchanged to the byte (the cluster plan at 96 tokens, the three launches
at 1000)."""
import pytest
import torch

from combine_moe_plan_gb300 import moe
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import dev, dev_bf16, ensure_built

pytestmark = pytest.mark.gpu


def test_steps_leave_free_device_memory_unchanged():
    ensure_built()
    base = wl.WORKLOADS["t4096_h7168_e256p288_k8"]
    runs = []
    for T in (96, 1000):  # cluster plan and three launches
        w = wl.small_variant(base, T)
        inp = wl.make_inputs(w, with_expert_out=False)
        pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2)
        runs.append((w, pool, dev(inp["logits"]), dev_bf16(inp["x"]), dev(inp["rep_off"]), dev(inp["rep_ids"]),
                     torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")))
    s = torch.cuda.Stream()

    def steps(n):
        with torch.cuda.stream(s):
            for i in range(n):
                for w, pool, logits, x, ro, ri, y in runs:
                    b = i & 1
                    pool.plan(logits, ro, ri, buf=b, stream=s)
                    pool.dispatch(x, buf=b, stream=s)
                    pool.identity_experts(w.T, buf=b, stream=s)
                    pool.combine(w.T, y=y, buf=b, stream=s)
        torch.cuda.synchronize()

    steps(3)
    free0, _ = torch.cuda.mem_get_info()
    steps(50)
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    for run in runs:
        assert run[1].check() == 0

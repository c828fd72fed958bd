"""The library called from several host threads at once (ctypes releases the
interpreter lock during each call, so the calls really overlap on the host):
each thread drives its own pool on its own stream through plan, dispatch and
combine many times, and one more thread schedules the split's transfers
(moe_ep_schedule_group, whose worker threads a concurrent call finds busy and
then computes on its own thread).  Every result must be the oracle's."""
import threading

import numpy as np
import pytest
import torch

import oracle
from combine_moe_plan_gb300 import ep, moe
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import assert_y_close, dev, dev_bf16, ensure_built, host_u16

pytestmark = pytest.mark.gpu


def test_pools_on_several_host_threads():
    ensure_built()
    cases = [("t96_h7168_e256_k8", 96), ("t4096_h7168_e256p288_k8", 300), ("t16384_h2048_e64_k6", 700),
             ("t64_h256_e8_k2", 64)]
    prepared = []
    for name, T in cases:
        w = wl.small_variant(wl.WORKLOADS[name], T)
        inp = wl.make_inputs(w, seed=3, with_expert_out=False)
        ref = oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"], w.P)
        prepared.append((w, inp, ref))
    errors = []

    def work(i):
        try:
            w, inp, ref = prepared[i]
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            pool = moe.Pool(w.T, w.H, w.E, w.P, w.k, n_sets=2)
            lg, x = dev(inp["logits"]), dev_bf16(inp["x"])
            ro = None if inp["rep_off"] is None else dev(inp["rep_off"])
            ri = None if inp["rep_ids"] is None else dev(inp["rep_ids"])
            ys = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
            with torch.cuda.stream(s):
                for it in range(40):
                    b = it & 1
                    pool.plan_dispatch(lg, x, ro, ri, buf=b, stream=s)
                    pool.identity_experts(w.T, buf=b, stream=s)
                    pool.combine(w.T, y=ys[b], buf=b, stream=s)
            s.synchronize()
            assert pool.check() == 0
            for b in range(2):
                assert_y_close(host_u16(ys[b]), ref["y"], f"thread {i} set {b}")
        except Exception as e:  # reported by the main thread
            errors.append(f"thread {i}: {e!r}")

    def schedules():
        try:
            rng = np.random.default_rng(4)
            R, P = 8, 288
            desc = ep.make_desc(R, P, 16)
            for _ in range(20):
                counts = rng.integers(0, 40, size=(R, P)).astype(np.int32)
                units, core_off, _ = ep.schedule_group(desc, 0, counts, 7168 + 4 * 56)
                want_u, want_off = ep.pack_schedules([ep.schedule(desc, 0, d, counts, 7168 + 4 * 56)
                                                      for d in range(R)])
                np.testing.assert_array_equal(units, want_u)
                np.testing.assert_array_equal(core_off, want_off)
        except Exception as e:
            errors.append(f"schedules: {e!r}")

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(prepared))]
    threads += [threading.Thread(target=schedules) for _ in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, "\n".join(errors)

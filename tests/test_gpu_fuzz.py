"""Randomised parity and write-coverage checks of the CUDA path against the
oracle (fixed seeds): shapes, replica maps, ties, zero groups and outliers
drawn at random, every output compared element by element."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_plan_gb300 import moe
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import (assert_gates_close, assert_y_close, dev, dev_bf16, ensure_built, f32_bits,
                            host_u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _random_case(rng):
    # batch sizes on both sides of every plan form's limit: the cluster plan's
    # tile sizes (8 tokens up to 64, 16 up to 128, 32 up to 512, portable up
    # to 256), the three launches beyond, and 32/33 tiles
    T = int(rng.choice([1, 2, 8, 9, 31, 32, 33, 64, 65, 95, 128, 129, 200, 256, 257, 512, 513, 700, 1024, 1025,
                        1500]))
    H = int(rng.choice([128, 256, 384, 896, 2048]))
    E = int(rng.integers(1, 300))
    k_max = 32 if rng.random() < 0.25 else 12
    k = int(rng.integers(1, min(E, k_max) + 1))
    n_rep = int(rng.integers(0, min(E, 40) + 1)) if rng.random() < 0.6 else 0
    P = E + n_rep
    rep_off = rep_ids = None
    if n_rep:
        hot = set(rng.choice(E, size=n_rep, replace=False).tolist())
        off, ids, nxt = [0], [], E
        for e in range(E):
            mine = [e] + ([nxt] if e in hot else [])
            nxt += e in hot
            ids += mine
            off.append(off[-1] + len(mine))
        perm = rng.permutation(P)  # any relabelling of physical slots is a valid map
        rep_off = np.array(off, np.int32)
        rep_ids = perm[np.array(ids)].astype(np.int32)
    if rng.random() < 0.3:  # heavy ties
        logits = rng.choice(np.float32([-1, 0, 0.5, 2]), size=(T, E)).astype(np.float32)
    else:
        logits = (rng.standard_normal((T, E)) * rng.uniform(0.1, 4)).astype(np.float32)
    x = rng.standard_normal((T, H)).astype(np.float32)
    x[rng.random((T, H)) < 0.001] *= 60.0
    zero_rows = rng.random(T) < 0.05
    x[zero_rows, :128] = 0.0
    return T, H, E, P, k, logits, wl.f32_to_bf16_bits(x), rep_off, rep_ids


@pytest.mark.parametrize("seed", range(600))
def test_random_shapes_match_oracle(seed):
    rng = np.random.default_rng(1000 + seed)
    T, H, E, P, k, logits, x, rep_off, rep_ids = _random_case(rng)
    ex = wl.f32_to_bf16_bits(rng.standard_normal((T * k, H)).astype(np.float32))
    T_max = T + int(rng.integers(0, 64))
    pool = moe.Pool(T_max, H, E, P, k, n_sets=2)
    buf = int(rng.integers(0, 2))
    ro = None if rep_off is None else dev(rep_off)
    ri = None if rep_ids is None else dev(rep_ids)
    pool.plan(dev(logits), ro, ri, buf=buf)
    pool.dispatch(dev_bf16(x), buf=buf)
    y = pool.combine(T, ex_out=dev_bf16(ex), buf=buf)
    assert pool.check() == 0
    ref = oracle.plan(logits, k, rep_off, rep_ids, P)
    v = pool.view(buf)
    R = T * k
    for key in ("topk_e", "phys", "slot"):
        np.testing.assert_array_equal(v[key][:T].cpu().numpy(), ref[key], err_msg=key)
    for key in ("counts", "offsets"):
        np.testing.assert_array_equal(v[key].cpu().numpy(), ref[key], err_msg=key)
    np.testing.assert_array_equal(v["src_token"][:R].cpu().numpy(), ref["src_token"])
    np.testing.assert_array_equal(v["src_k"][:R].cpu().numpy(), ref["src_k"])
    assert_gates_close(v["gates"][:T].cpu().numpy(), ref["gates"], "gates")
    codes, scales = oracle.dispatch(x, ref["slot"])
    np.testing.assert_array_equal(v["codes"][:R].cpu().numpy(), codes)
    np.testing.assert_array_equal(f32_bits(v["scales"][:R, :H // 128].cpu().numpy()), f32_bits(scales))
    assert_y_close(host_u16(y), oracle.combine(ex, ref["slot"], ref["gates"]), "y")


def test_dispatch_writes_exactly_its_rows():
    """Poison both sets (code -128 never occurs; NaN scales), dispatch into
    set 1: its rows [0, T*k) are all written, every other row of set 1 and
    all of set 0 keep the poison."""
    w = wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 300)
    inp = wl.make_inputs(w, with_expert_out=False)
    pool = moe.Pool(512, w.H, w.E, w.P, w.k, n_sets=2)
    for b in range(2):
        v = pool.view(b)
        v["codes"].fill_(-128)
        v["scales"].fill_(float("nan"))
    pool.plan(dev(inp["logits"]), dev(inp["rep_off"]), dev(inp["rep_ids"]), buf=1)
    pool.dispatch(dev_bf16(inp["x"]), buf=1)
    assert pool.check() == 0
    R, G = w.rows, w.G
    v1, v0 = pool.view(1), pool.view(0)
    live = v1["codes"][:R]
    assert int((live == -128).sum()) == 0
    assert torch.isfinite(v1["scales"][:R, :G]).all()
    assert bool((v1["codes"][R:] == -128).all())
    assert bool(torch.isnan(v1["scales"][R:]).all())
    assert bool((v0["codes"] == -128).all())
    assert bool(torch.isnan(v0["scales"]).all())

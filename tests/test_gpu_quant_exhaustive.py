"""Exhaustive check of the dispatch kernel's INT8 codes: every finite bf16
activation against group maxima covering all 128 bf16 significands (and spot
exponents), through moe_plan + moe_dispatch with one expert and k = 1, so
slot = token.  Codes and scales must equal the oracle's (IEEE binary32
division, round-half-even) bit for bit."""
import numpy as np
import pytest

import oracle
from combine_moe_plan_gb300 import moe
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import dev, dev_bf16, ensure_built, f32_bits

pytestmark = pytest.mark.gpu


def _groups():
    allx = wl.bf16_bits_to_f32(np.arange(0x10000, dtype=np.uint16))
    allx = allx[np.isfinite(allx)]
    amaxes = [np.float32(m * 2.0 ** e) for e in (-100, -20, -3, 1, 7, 40, 100)
              for m in (1.0, 1.0078125, 1.5, 1.9921875, 1.3359375, 1.75)]
    amaxes += [np.float32((1.0 + m / 128.0) * 2.0 ** e) for e in (0, 60, -60) for m in range(128)]
    amaxes.append(np.float32(254.0))
    # bf16 subnormal maxima: 1/amax is not a normal binary32 there, so the
    # kernel takes its IEEE-division branch
    amaxes += [wl.bf16_bits_to_f32(np.array([b], np.uint16))[0] for b in (0x0001, 0x0003, 0x0040, 0x007F)]
    rows = []
    for a in amaxes:
        xs = allx[np.abs(allx) <= a]
        xs = xs[np.abs(xs) < 2.0 ** 120]
        xs = np.concatenate([xs, np.zeros((-len(xs)) % 127, np.float32)]).reshape(-1, 127)
        rows.append(np.concatenate([np.full((xs.shape[0], 1), a, np.float32), xs], axis=1))
    return np.concatenate(rows)


def test_dispatch_codes_exhaustive():
    ensure_built()
    g = _groups()
    H = 7168
    per_row = H // 128
    pad = (-g.shape[0]) % per_row
    g = np.concatenate([g, np.zeros((pad, 128), np.float32)])
    x = wl.f32_to_bf16_bits(g.reshape(-1, H))
    T = x.shape[0]
    assert T * H > 12_000_000
    pool = moe.Pool(T, H, 1, 1, 1, n_sets=1)
    pool.plan(dev(np.zeros((T, 1), np.float32)))
    pool.dispatch(dev_bf16(x))
    assert pool.check() == 0
    v = pool.view(0)
    np.testing.assert_array_equal(v["slot"].cpu().numpy()[:, 0], np.arange(T))
    codes, scales = oracle.quantize(x)
    got = v["codes"][:T].cpu().numpy()
    bad = np.nonzero(got != codes)
    assert bad[0].size == 0, f"{bad[0].size} codes differ, first at {bad[0][:3]}, {bad[1][:3]}"
    np.testing.assert_array_equal(f32_bits(v["scales"][:T, :per_row].cpu().numpy()), f32_bits(scales))

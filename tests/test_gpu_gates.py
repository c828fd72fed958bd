"""Gates of the CUDA plan against the oracle's.

The route kernel forms each gate from pairs of floats and keeps the pair's
fp32 rounding only where Ziv's test proves it is the correctly rounded
quotient; the rest of a token goes through fp64.  These cases drive both
paths: every token size class k (including odd k, whose lane segments have
idle lanes, and k = 32, a whole warp per token), logit scales from almost
flat to very peaked, tokens whose selected logits sit 60-120 below the top
(the fp64 path; subnormal and zero gates), exact ties, and a million gates
counted for any difference at all."""
import numpy as np
import pytest

import oracle
from combine_moe_plan_gb300 import moe
from tests.gpu_util import assert_gates_close, dev, ensure_built, f32_bits, ulp_dist_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _gates(logits, k, P=None):
    T, E = logits.shape
    P = E if P is None else P
    pool = moe.Pool(T, 128, E, P, k, n_sets=1)
    pool.plan(dev(logits))
    assert pool.check() == 0
    v = pool.view(0)
    return v["topk_e"][:T].cpu().numpy(), v["gates"][:T].cpu().numpy()


@pytest.mark.parametrize("k", [1, 2, 3, 5, 6, 7, 8, 9, 16, 17, 31, 32])
@pytest.mark.parametrize("scale", [0.01, 1.0, 4.0, 20.0])
def test_gates_every_k_and_scale(k, scale):
    rng = np.random.default_rng(7000 + 37 * k + int(scale * 100))
    T, E = 2048, max(64, k)
    logits = (rng.standard_normal((T, E)) * scale).astype(np.float32)
    topk, g = _gates(logits, k)
    ref = oracle.plan(logits, k)
    np.testing.assert_array_equal(topk, ref["topk_e"])
    assert_gates_close(g, ref["gates"], f"k={k} scale={scale}")


@pytest.mark.parametrize("gaps", [
    [0, 10, 40, 63.9],                     # all within the pair path (d >= -64)
    [0, 10, 63.9, 64.1, 80, 90, 100, 110],  # tokens redone in fp64: gates down to subnormal and zero
])
def test_gates_far_below_the_top(gaps):
    rng = np.random.default_rng(99 + len(gaps))
    T, E, k = 1024, 16, len(gaps)
    gaps = np.float32(gaps)
    logits = np.full((T, E), -1000.0, np.float32)
    base = rng.uniform(-5, 5, T).astype(np.float32)
    jitter = rng.uniform(-0.04, 0.04, (T, k)).astype(np.float32)
    jitter[:, 0] = 0
    for t in range(T):
        cols = rng.permutation(E)[:k]
        logits[t, cols] = base[t] - gaps - jitter[t]
    topk, g = _gates(logits, k)
    ref = oracle.plan(logits, k)
    np.testing.assert_array_equal(topk, ref["topk_e"])
    assert np.all(ulp_dist_f32(g, ref["gates"]) == 0)
    if k == 8:
        assert (ref["gates"][:, 7] == 0).all() and (ref["gates"][:, 6] > 0).all()
        assert (ref["gates"][:, 6] < np.float32(2.0 ** -126)).all()  # subnormal gates


def test_gates_ties_are_exact():
    # Equal logits: 1/k exactly where k is a power of two, and equal gates.
    T, E = 64, 32
    for k in (2, 4, 8, 16, 32, 3, 5):
        logits = np.zeros((T, E), np.float32)
        topk, g = _gates(logits, k)
        ref = oracle.plan(logits, k)
        np.testing.assert_array_equal(topk, ref["topk_e"])
        np.testing.assert_array_equal(f32_bits(g), f32_bits(ref["gates"]))
        assert np.all(g == g[:, :1])
        if k & (k - 1) == 0:
            assert np.all(g == np.float32(1.0 / k))


def test_a_million_gates_identical():
    rng = np.random.default_rng(2024)
    T, E, k = 131072, 256, 8
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits += (-1.2 * np.log1p(rng.permutation(E))).astype(np.float32)  # Zipf-like expert bias
    _, g = _gates(logits, k)
    ref = oracle.route(logits, k)[1]
    d = ulp_dist_f32(g, ref)
    assert d.max() <= 1 and int((d > 0).sum()) <= 2, f"{int((d > 0).sum())} of {d.size} gates differ"

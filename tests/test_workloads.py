"""The seeded input recipe (combine_moe_plan_gb300/workloads.py), the one
module both the oracle and the CUDA path take inputs from.  It holds none of
the method's arithmetic, but what it draws must be what the recipe states:
bf16 by round-to-nearest-even, the replica map's structure, the Zipf bias,
the outlier count, determinism per seed and independent sub-streams.
Host only."""
import numpy as np
import pytest
import torch

from combine_moe_plan_gb300 import workloads as wl


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    scale = np.float32(10.0) ** rng.integers(-30, 30, 100_000).astype(np.float32)
    a = np.concatenate([rng.standard_normal(100_000).astype(np.float32) * scale,
                        np.float32([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1e-40, -1e-40])])
    a = a[np.isfinite(a)]
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(wl.f32_to_bf16_bits(a), ref)
    # and the inverse widens exactly
    widened = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(wl.bf16_bits_to_f32(ref), widened)


def test_replica_map_structure():
    w = wl.WORKLOADS["t4096_h7168_e256p288_k8"]
    off, ids = wl.make_replica_map(w)
    rank = wl.expert_popularity_rank(w)
    assert off[0] == 0 and off[-1] == w.P and np.all(np.diff(off) >= 1)
    assert sorted(ids.tolist()) == list(range(w.P))  # a permutation of the physical slots
    for e in range(w.E):
        mine = ids[off[e]:off[e + 1]].tolist()
        assert mine[0] == e
        if rank[e] <= w.replicas:  # the most popular experts get one extra slot, id E + rank - 1
            assert mine == [e, w.E + int(rank[e]) - 1]
        else:
            assert mine == [e]
    assert wl.make_replica_map(wl.WORKLOADS["t96_h7168_e256_k8"]) == (None, None)


def test_zipf_bias_and_popularity():
    w = wl.WORKLOADS["t4096_h7168_e256p288_k8"]
    rank = wl.expert_popularity_rank(w)
    assert sorted(rank.tolist()) == list(range(1, w.E + 1))
    b = wl.zipf_bias(w)
    np.testing.assert_allclose(b, -1.2 * np.log(rank.astype(np.float64)), rtol=1e-6)
    assert b[np.argmin(rank)] == 0.0
    assert not wl.zipf_bias(wl.WORKLOADS["t96_h7168_e256_k8"]).any()
    # the router sees the skew: the most popular expert is picked far more often
    small = wl.small_variant(w, 2048)
    top1 = np.argmax(wl.make_logits(small), axis=1)
    counts = np.bincount(top1, minlength=w.E)
    assert counts[np.argmin(rank)] > 5 * np.median(counts)


def test_outliers_are_the_stated_fraction():
    w = wl.WORKLOADS["t96_h7168_e256_k8"]
    x = wl.bf16_bits_to_f32(wl.make_x(w))
    n_out = int(round(w.outlier_frac * w.T * w.H))
    assert n_out == 688
    # N(0,1) passes 6 sigma about once in 5e8 draws; 50 z does whenever |z| > 0.12
    big = int((np.abs(x) > 6.0).sum())
    assert 0.8 * n_out <= big <= n_out
    assert np.abs(x).max() <= 50 * 6.5


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_inputs_are_deterministic_and_streams_independent(name):
    w = wl.small_variant(wl.WORKLOADS[name], 64)
    a, b = wl.make_inputs(w, seed=3), wl.make_inputs(w, seed=3)
    for key in a:
        if a[key] is None:
            assert b[key] is None
        else:
            np.testing.assert_array_equal(a[key], b[key])
    c = wl.make_inputs(w, seed=4)
    assert not np.array_equal(a["logits"], c["logits"]) and not np.array_equal(a["x"], c["x"])
    # one tensor's draw does not depend on another's size
    np.testing.assert_array_equal(wl.make_logits(w, seed=3, T=32), a["logits"][:32])
    assert a["logits"].dtype == np.float32 and a["x"].dtype == np.uint16 and np.isfinite(a["logits"]).all()


def test_algorithmic_bytes_of_the_bench_workload():
    b = wl.WORKLOADS["t4096_h7168_e256p288_k8"].algorithmic_bytes()
    assert (b["plan"], b["dispatch"], b["combine"]) == (4_589_832, 301_072_384, 528_744_448)
    assert b["total"] == 834_406_664

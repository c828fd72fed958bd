"""Randomised parity of the expert-parallel split against the oracle's split
(fixed seeds): group size, ragged and empty batches, expert counts with and
without replicas, top-k, hidden size, the transfer schedule's cores, caps
and unit sizes, and the form of the step (both exchanges pulled, the combine
fused, or dispatch and combine fused) drawn at random; every receive buffer,
returned row and y compared."""
import numpy as np
import pytest

import oracle
from combine_moe_plan_gb300 import ep
from combine_moe_plan_gb300 import workloads as wl
from tests.gpu_util import assert_y_close, dev, dev_bf16, ensure_built, f32_bits, host_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _replica_map(rng, E):
    n_rep = int(rng.integers(0, min(E, 24) + 1)) if rng.random() < 0.6 else 0
    if not n_rep:
        return E, None, None
    hot = set(rng.choice(E, size=n_rep, replace=False).tolist())
    off, ids, nxt = [0], [], E
    for e in range(E):
        mine = [e] + ([nxt] if e in hot else [])
        nxt += e in hot
        ids += mine
        off.append(off[-1] + len(mine))
    P = E + n_rep
    perm = rng.permutation(P)
    return P, np.array(off, np.int32), perm[np.array(ids)].astype(np.int32)


@pytest.mark.parametrize("seed", range(500))
def test_random_splits_match_oracle(seed):
    rng = np.random.default_rng(5000 + seed)
    R = int(rng.integers(1, 10))
    Ts = [int(rng.choice([0, 1, 7, 33, 97, 130, 200])) for _ in range(R)]
    H = int(rng.choice([128, 256, 640]))
    E = int(rng.integers(1, 81))
    k = int(rng.integers(1, min(E, 10) + 1))
    P, rep_off, rep_ids = _replica_map(rng, E)
    mode = str(rng.choice(["pull", "fused_combine", "fused"]))
    cores = int(rng.integers(1, 9))
    cap = (int(rng.integers(1, cores + 1)), int(rng.integers(1, cores + 1)))
    S = (int(rng.choice([1, 3, 16, 64])), int(rng.choice([1, 5, 64])))
    logits = []
    for T in Ts:
        if rng.random() < 0.3:
            logits.append(rng.choice(np.float32([-1, 0, 0.5, 2]), size=(T, E)).astype(np.float32))
        else:
            logits.append((rng.standard_normal((T, E)) * rng.uniform(0.1, 4)).astype(np.float32))
    xs = [wl.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)) for T in Ts]
    T_max = max(max(Ts), 1) + int(rng.integers(0, 16))
    g = ep.EmulatedGroup(R, T_max, H, E, P, k, cores=cores, desc_kw=dict(fanout_cap=cap, unit_rows=S))
    ro = None if rep_off is None else dev(rep_off)
    ri = None if rep_ids is None else dev(rep_ids)
    ys, counts, recv_rows = g.step([dev(a) for a in logits], [dev_bf16(a) for a in xs], ro, ri,
                                   fused_combine=mode != "pull", fused_dispatch=mode == "fused")
    ref = oracle.ep_forward(logits, xs, k, P, rep_off, rep_ids)
    np.testing.assert_array_equal(counts, ref["counts"])
    G = H // 128
    for d in range(R):
        n = recv_rows[d]
        assert n == ref["recv_codes"][d].shape[0]
        np.testing.assert_array_equal(g.recv_codes[d][:n].cpu().numpy(), ref["recv_codes"][d], err_msg=f"codes {d}")
        np.testing.assert_array_equal(f32_bits(g.recv_scales[d][:n, :G].cpu().numpy()),
                                      f32_bits(ref["recv_scales"][d]), err_msg=f"scales {d}")
    for s in range(R):
        if mode == "pull":
            rows = int(counts[s].sum())
            np.testing.assert_array_equal(host_u16(g.views[s]["ex_out"][:rows]), ref["ex_out"][s])
        assert_y_close(host_u16(ys[s]), ref["y"][s], f"seed {seed} rank {s} ({mode})")
    assert g.check() == 0
    for p in g.pools:
        assert p.check() == 0

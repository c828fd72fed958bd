"""Pins for the oracle's expert-parallel split (oracle/moe_oracle_ep.c):
closed forms, brute force on tiny inputs, the single-pool plan of the
concatenated batch, exchange invariants, textbook LPT instances, Graham's
bound against an exhaustive optimum, and hand-worked schedules.  Each is
chosen so that a plausible slip (rounding of the ownership, source order
inside a window, an off-by-one piece, LPT order, tie-breaks, the fan-out
cap) fails at least one of them.  Nothing here calls the CUDA library.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from combine_moe_plan_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# -------------------------------------------------------------- ownership --

@pytest.mark.parametrize("R,P", [(1, 8), (2, 8), (3, 8), (8, 288), (7, 256), (32, 288), (5, 5), (4, 64)])
def test_owner_is_the_balanced_block_partition(R, P):
    """Rank d owns exactly the p with d*P/R <= p < (d+1)*P/R, i.e. a block of
    ceil((d+1)P/R) - ceil(dP/R) experts, by exact rational arithmetic."""
    owners = [oracle.ep_owner(p, R, P) for p in range(P)]
    for p, d in enumerate(owners):
        assert Fraction(d * P, R) <= p < Fraction((d + 1) * P, R)
    assert owners == sorted(owners)
    sizes = np.bincount(owners, minlength=R)
    assert sizes.max() - sizes.min() <= 1
    for d in range(R):
        assert sizes[d] == math.ceil(Fraction((d + 1) * P, R)) - math.ceil(Fraction(d * P, R))


# ----------------------------------------------------------------- layout --

def _layout_brute(counts, d):
    """Receiver d's windows: (expert, source) pairs in lexicographic order."""
    R, P = counts.shape
    owners = [int(p * R // P) for p in range(P)]
    mine = [p for p in range(P) if owners[p] == d]
    pairs = sorted((p, s) for p in mine for s in range(R))
    start, row = {}, 0
    for p, s in pairs:
        start[(p, s)] = row
        row += int(counts[s, p])
    expert_off = [start[(p, 0)] for p in mine] + [row]
    chunk = np.array([[start[(p, s)] for p in mine] for s in range(R)], np.int32).reshape(R, len(mine))
    return np.array(expert_off, np.int32), chunk


@pytest.mark.parametrize("R,P,seed", [(1, 8, 0), (2, 8, 1), (3, 10, 2), (4, 17, 3), (8, 288, 4)])
def test_layout_matches_brute_force(R, P, seed):
    counts = np.random.default_rng(seed).integers(0, 50, size=(R, P)).astype(np.int32)
    counts[:, ::5] = 0  # empty windows
    total = 0
    for d in range(R):
        off, chunk = oracle.ep_layout(counts, d)
        bo, bc = _layout_brute(counts, d)
        np.testing.assert_array_equal(off, bo)
        np.testing.assert_array_equal(chunk, bc)
        total += int(off[-1])
    assert total == int(counts.sum())


# ----------------------------------------------------------------- gather --

def _ranks(R, T, H, E, k, seed):
    ws = [wl.Workload(f"ep{r}", T=T, H=H, E=E, P=E, k=k) for r in range(R)]
    return [wl.make_inputs(w, seed=seed + r, with_expert_out=False) for r, w in enumerate(ws)]


@pytest.mark.parametrize("R,T,E,k", [(2, 40, 8, 2), (3, 33, 12, 3), (4, 64, 16, 4), (1, 20, 8, 2)])
def test_gather_equals_plan_of_the_concatenated_batch(R, T, E, k):
    """Receiver d's rows are the rows of d's experts in the single-pool plan of
    all ranks' tokens concatenated in rank order: in that plan each expert's
    window lists tokens by ascending global index, i.e. source rank first,
    then the source's token order.  (Identity replica map: with replicas the
    pick depends on the token index, which concatenation changes.)"""
    H = 256
    inps = _ranks(R, T, H, E, k, seed=10 * R + T)
    fwd = oracle.ep_forward([i["logits"] for i in inps], [i["x"] for i in inps], k)
    cat_logits = np.concatenate([i["logits"] for i in inps])
    cat_x = np.concatenate([i["x"] for i in inps])
    g = oracle.plan(cat_logits, k)
    codes, scales = oracle.dispatch(cat_x, g["slot"])
    for d in range(R):
        mine = [p for p in range(E) if oracle.ep_owner(p, R, E) == d]
        if not mine:
            assert fwd["recv_codes"][d].shape[0] == 0
            continue
        lo, hi = g["offsets"][mine[0]], g["offsets"][mine[-1] + 1]
        np.testing.assert_array_equal(fwd["recv_codes"][d], codes[lo:hi])
        np.testing.assert_array_equal(fwd["recv_scales"][d].view(np.int32), scales[lo:hi].view(np.int32))


def test_gather_brute_force_tiny():
    """Every copy (rank s, token t, j) routed to expert p of rank d, sorted by
    (p, s, t), must appear in that order in d's buffer, holding s's row for
    that copy."""
    R, T, E, k = 3, 7, 6, 2
    inps = _ranks(R, T, 128, E, k, seed=5)
    fwd = oracle.ep_forward([i["logits"] for i in inps], [i["x"] for i in inps], k)
    for d in range(R):
        copies = []
        for s in range(R):
            ph = fwd["plan"][s]["phys"]
            for t in range(T):
                for j in range(k):
                    p = int(ph[t, j])
                    if p * R // E == d:
                        copies.append((p, s, t, int(fwd["plan"][s]["slot"][t, j])))
        copies.sort()
        want = np.stack([fwd["codes"][s][r] for (_, s, _, r) in copies]) if copies else np.zeros((0, 128))
        np.testing.assert_array_equal(fwd["recv_codes"][d], want)


# ----------------------------------------------------------------- return --

@pytest.mark.parametrize("R,P,seed", [(1, 6, 0), (2, 6, 1), (3, 9, 2), (5, 16, 3)])
def test_return_inverts_gather(R, P, seed):
    """Gather then return reproduces every source's rows exactly (random
    bytes as rows, random counts including empty windows)."""
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 9, size=(R, P)).astype(np.int32)
    counts[rng.random((R, P)) < 0.3] = 0
    planes = [rng.integers(0, 256, size=(int(counts[s].sum()), 48), dtype=np.uint8) for s in range(R)]
    recv = [oracle.ep_gather(planes, counts, d) for d in range(R)]
    assert sum(r.shape[0] for r in recv) == counts.sum()
    for s in range(R):
        back = oracle.ep_return(recv, counts, s, planes[s].shape[0])
        np.testing.assert_array_equal(back, planes[s])


def test_one_rank_is_the_identity():
    rng = np.random.default_rng(3)
    counts = rng.integers(0, 9, size=(1, 7)).astype(np.int32)
    plane = rng.integers(0, 256, size=(int(counts.sum()), 32), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.ep_gather([plane], counts, 0), plane)


@pytest.mark.parametrize("R,T", [(2, 48), (4, 33)])
def test_split_forward_equals_local_forward(R, T):
    """With identity experts the split changes only where rows travel: every
    rank's y equals the single-rank forward of its own batch, bit for bit,
    with the 32-replica map of the bench workload's small variant."""
    w = wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], T)
    w = wl.dataclasses.replace(w, H=256)
    inps = [wl.make_inputs(w, seed=r, with_expert_out=False) for r in range(R)]
    off, ids = wl.make_replica_map(w)
    fwd = oracle.ep_forward([i["logits"] for i in inps], [i["x"] for i in inps], w.k, w.P, off, ids)
    for r in range(R):
        loc = oracle.forward(inps[r]["logits"], inps[r]["x"], w.k, off, ids, w.P)
        np.testing.assert_array_equal(fwd["y"][r], loc["y"])
        np.testing.assert_array_equal(fwd["ex_out"][r], loc["ex_out"])


# --------------------------------------------------------------- schedule --

def _sched(counts, C, cap=(64, 64), unit_rows=(1 << 20, 1 << 20), alpha=(0, 0), beta=(1000, 1000), rb=1,
           direction=0, puller=0):
    return oracle.ep_schedule(direction, puller, np.asarray(counts, np.int32), C, list(cap), list(unit_rows),
                              list(alpha), list(beta), rb)


def _loads(r, C):
    return [int(r["cost"][r["core_off"][c]:r["core_off"][c + 1]].sum()) for c in range(C)]


@pytest.mark.parametrize("jobs,C,lpt,opt", [((3, 3, 2, 2, 2), 2, 7, 6), ((5, 5, 4, 4, 3, 3, 3), 3, 11, 9)])
def test_lpt_on_graham_worst_cases(jobs, C, lpt, opt):
    """Graham (1969): on these instances LPT reaches its bound
    (4/3 - 1/(3m)) * OPT exactly.  One rank, one expert per job, one unit per
    expert, cost = rows picoseconds."""
    r = _sched([list(jobs)], C)
    assert r["makespan"] == lpt
    assert Fraction(lpt, opt) == Fraction(4, 3) - Fraction(1, 3 * C)
    assert sorted(r["cost"].tolist()) == sorted(jobs)


def _opt_brute(costs, C):
    best = None
    for assign in itertools.product(range(C), repeat=len(costs)):
        loads = [0] * C
        for c, x in zip(assign, costs):
            loads[c] += x
        m = max(loads)
        best = m if best is None or m < best else best
    return best


@pytest.mark.parametrize("seed", range(12))
def test_lpt_within_graham_bound_of_the_exhaustive_optimum(seed):
    rng = np.random.default_rng(seed)
    C = int(rng.integers(2, 4))
    n = int(rng.integers(C + 1, 9))
    jobs = rng.integers(1, 40, size=n).astype(np.int32)
    r = _sched([jobs.tolist()], C)
    opt = _opt_brute(jobs.tolist(), C)
    assert r["makespan"] >= opt
    assert Fraction(r["makespan"]) <= (Fraction(4, 3) - Fraction(1, 3 * C)) * opt
    assert max(_loads(r, C)) == r["makespan"]


def _check_units(r, counts, direction, puller, unit_rows, cap, C):
    """Coverage, piece sizes and the fan-out cap, from the pages' definitions."""
    R, P = counts.shape
    units = r["units"]
    # destination rows tiled exactly once, source rows where the layout says
    if direction == 0:
        off, chunk = oracle.ep_layout(counts, puller)
        want_dst = int(off[-1])
    else:
        want_dst = int(counts[puller].sum())
    cover = np.zeros(want_dst, np.int32)
    for u in units:
        cover[u["dst_row"]:u["dst_row"] + u["rows"]] += 1
        tier = 0 if u["peer"] == puller else 1
        assert 1 <= u["rows"] <= unit_rows[tier]
    assert (cover == 1).all()
    # fan-out cap per stripe
    stripes = {}
    for c in range(C):
        for i, u in enumerate(units[r["core_off"][c]:r["core_off"][c + 1]]):
            stripes.setdefault((i, int(u["peer"])), set()).add(c)
    for (i, q), cores in stripes.items():
        assert len(cores) <= cap[0 if q == puller else 1]


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("direction", [0, 1])
def test_schedule_covers_every_row_once_and_keeps_the_cap(seed, direction):
    rng = np.random.default_rng(100 + seed)
    R = int(rng.integers(1, 6))
    P = int(rng.integers(R, 3 * R + 4))
    counts = rng.integers(0, 30, size=(R, P)).astype(np.int32)
    counts[rng.random((R, P)) < 0.25] = 0
    C = int(rng.integers(1, 9))
    cap = [int(rng.integers(1, 4)), int(rng.integers(1, 4))]
    unit_rows = [int(rng.integers(1, 9)), int(rng.integers(1, 9))]
    puller = int(rng.integers(0, R))
    r = _sched(counts, C, cap, unit_rows, (int(rng.integers(0, 5)), int(rng.integers(0, 5))),
               (int(rng.integers(50, 3000)), int(rng.integers(50, 3000))), int(rng.integers(1, 5000)),
               direction, puller)
    _check_units(r, counts, direction, puller, unit_rows, cap, C)
    assert r["core_off"][-1] == len(r["units"])
    assert max(_loads(r, C)) == r["makespan"]


def test_schedule_source_rows_follow_the_layout():
    """Dispatch units read each source's own window rows; combine units read
    the owner's receive rows: both from the layout and the sources' scans."""
    rng = np.random.default_rng(9)
    R, P = 3, 8
    counts = rng.integers(0, 12, size=(R, P)).astype(np.int32)
    pool_off = np.concatenate([np.zeros((R, 1), np.int64), np.cumsum(counts, axis=1)], axis=1)
    for d in range(R):
        off, chunk = oracle.ep_layout(counts, d)
        mine = [p for p in range(P) if oracle.ep_owner(p, R, P) == d]
        r = _sched(counts, 4, unit_rows=(5, 3), direction=0, puller=d)
        for u in r["units"]:
            s = int(u["peer"])
            # which of d's windows holds this destination row
            i = int(np.searchsorted(off, u["dst_row"], side="right") - 1)
            p = mine[i]
            delta = u["dst_row"] - chunk[s, i]
            assert 0 <= delta and delta + u["rows"] <= counts[s, p]
            assert u["src_row"] == pool_off[s, p] + delta
    for s in range(R):
        r = _sched(counts, 4, unit_rows=(5, 3), direction=1, puller=s)
        for u in r["units"]:
            d = int(u["peer"])
            p = int(np.searchsorted(pool_off[s], u["dst_row"], side="right") - 1)
            assert oracle.ep_owner(p, R, P) == d
            off, chunk = oracle.ep_layout(counts, d)
            i = [q for q in range(P) if oracle.ep_owner(q, R, P) == d].index(p)
            delta = u["dst_row"] - pool_off[s, p]
            assert u["src_row"] == chunk[s, i] + delta


def test_hand_worked_schedules():
    data = json.load(open(os.path.join(GOLDEN, "ep_schedule.json")))
    for case in data["cases"]:
        r = oracle.ep_schedule(case["direction"], case["puller"], np.array(case["counts"], np.int32), case["C"],
                               case["cap"], case["unit_rows"], case["alpha_ns"], case["beta_gbs"],
                               case["row_bytes"])
        got = [[list(map(int, (u["peer"], u["src_row"], u["dst_row"], u["rows"])))
                for u in r["units"][r["core_off"][c]:r["core_off"][c + 1]]] for c in range(case["C"])]
        assert got == case["core_units"], case["name"]
        assert r["makespan"] == case["makespan"], case["name"]


def _handworked_split():
    g = json.load(open(os.path.join(GOLDEN, "ep_handworked.json")))
    R, H = g["R"], g["H"]
    logits = [np.array(a, np.float32) for a in g["logits"]]
    xs = []
    for s in range(R):
        x = np.zeros((len(g["logits"][s]), H), np.float32)
        x[:, 0] = [1 + 4 * s + t for t in range(x.shape[0])]
        xs.append(wl.f32_to_bf16_bits(x))
    return g, logits, xs


def test_handworked_split():
    """The split worked by hand in tests/golden/ep_handworked.json: every
    rank's plan, every owner's receive layout (window starts and rows), and
    the order of the rows each owner receives (named by their scales)."""
    g, logits, xs = _handworked_split()
    R, P, k = g["R"], g["P"], g["k"]
    for s in range(R):
        pl = oracle.plan(logits[s], k, None, None, P)
        np.testing.assert_array_equal(pl["topk_e"], g["topk_e"][s])
        np.testing.assert_array_equal(pl["counts"], g["counts"][s])
        np.testing.assert_array_equal(pl["offsets"], g["offsets"][s])
        np.testing.assert_array_equal(pl["slot"], g["slot"][s])
    counts = np.array(g["counts"], np.int32)
    for d in range(R):
        expert_off, chunk_row = oracle.ep_layout(counts, d)
        assert int(expert_off[-1]) == g["recv_rows"][d]
        mine = [p for p in range(P) if oracle.ep_owner(p, R, P) == d]
        for i, p in enumerate(mine):
            for s in range(R):
                assert int(chunk_row[s, i]) == g["recv_start"][s][p]
    ref = oracle.ep_forward(logits, xs, k, P)
    for d in range(R):
        want = np.array([np.float32(1 + 4 * s + t) / np.float32(127) for s, t in g["received"][d]], np.float32)
        np.testing.assert_array_equal(ref["recv_scales"][d][:, 0].view(np.int32), want.view(np.int32))

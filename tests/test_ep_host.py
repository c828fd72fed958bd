"""Host-only tests of the expert-parallel split's host calls (no GPU needed):
libmoe's ownership, receive layout and LPT transfer schedules against the
oracle, bit for bit (units, their order on every core, core offsets,
makespan), over random groups and the edge cases; the hand-worked schedules;
and argument checks before anything else runs."""
import ctypes
import json
import os

import numpy as np
import pytest

import oracle
from combine_moe_plan_gb300 import build as moe_build
from combine_moe_plan_gb300 import ep

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    moe_build.build()


def _same_schedule(got, ref, what):
    np.testing.assert_array_equal(got["core_off"], ref["core_off"], err_msg=f"{what}: core_off")
    g = got["units"].view(np.int32).reshape(-1, 4)
    r = ref["units"].view(np.int32).reshape(-1, 4)
    np.testing.assert_array_equal(g, r, err_msg=f"{what}: units")
    assert got["makespan"] == ref["makespan"], what


@pytest.mark.parametrize("R,P", [(1, 8), (2, 8), (3, 8), (8, 288), (7, 256), (64, 288), (5, 3), (64, 64)])
def test_experts_match_the_oracle(R, P):
    for d in range(R):
        first, count = ep.experts(R, P, d)
        mine = [p for p in range(P) if oracle.ep_owner(p, R, P) == d]
        assert count == len(mine)
        if mine:
            assert first == mine[0] and mine == list(range(first, first + count))


@pytest.mark.parametrize("seed", range(8))
def test_layout_matches_the_oracle(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 9))
    P = int(rng.integers(1, 40))
    counts = rng.integers(0, 100, size=(R, P)).astype(np.int32)
    counts[rng.random((R, P)) < 0.2] = 0
    for d in range(R):
        off, chunk = ep.layout(counts, d)
        ro, rc = oracle.ep_layout(counts, d)
        np.testing.assert_array_equal(off, ro)
        np.testing.assert_array_equal(chunk, rc)


def _random_case(rng):
    R = int(rng.integers(1, 9))
    P = int(rng.integers(1, 48))
    counts = rng.integers(0, 200, size=(R, P)).astype(np.int32)
    if rng.random() < 0.3:  # skew: one hot expert
        counts[:, int(rng.integers(0, P))] += int(rng.integers(100, 2000))
    counts[rng.random((R, P)) < 0.2] = 0
    kw = dict(cores=int(rng.integers(1, 40)),
              fanout_cap=(int(rng.integers(1, 5)), int(rng.integers(1, 5))),
              unit_rows=(int(rng.integers(1, 80)), int(rng.integers(1, 80))),
              alpha_ns=(int(rng.integers(0, 4)), int(rng.integers(0, 20))),
              beta_gbs=(int(rng.integers(100, 8000)), int(rng.integers(50, 1000))))
    return R, P, counts, kw


@pytest.mark.parametrize("seed", range(40))
def test_schedule_matches_the_oracle(seed):
    rng = np.random.default_rng(1000 + seed)
    R, P, counts, kw = _random_case(rng)
    desc = ep.make_desc(R, P, kw["cores"], kw["fanout_cap"], kw["unit_rows"], kw["alpha_ns"], kw["beta_gbs"])
    row_bytes = int(rng.choice([7168 + 224, 2 * 7168, 256 + 16, 1]))
    for direction in (0, 1):
        for puller in range(R):
            got = ep.schedule(desc, direction, puller, counts, row_bytes)
            ref = oracle.ep_schedule(direction, puller, counts, kw["cores"], kw["fanout_cap"], kw["unit_rows"],
                                     kw["alpha_ns"], kw["beta_gbs"], row_bytes)
            _same_schedule(got, ref, f"seed {seed} dir {direction} puller {puller}")


@pytest.mark.parametrize("seed", range(6))
def test_group_schedule_packs_every_pullers_schedule(seed):
    rng = np.random.default_rng(2000 + seed)
    R, P, counts, kw = _random_case(rng)
    desc = ep.make_desc(R, P, kw["cores"], kw["fanout_cap"], kw["unit_rows"], kw["alpha_ns"], kw["beta_gbs"])
    for direction, rb in ((0, 7168 + 224), (1, 2 * 7168)):
        units, core_off, ms = ep.schedule_group(desc, direction, counts, rb)
        want_u, want_off = ep.pack_schedules([ep.schedule(desc, direction, r, counts, rb) for r in range(R)])
        np.testing.assert_array_equal(units, want_u)
        np.testing.assert_array_equal(core_off, want_off)
        for r in range(R):
            ref = oracle.ep_schedule(direction, r, counts, kw["cores"], kw["fanout_cap"], kw["unit_rows"],
                                     kw["alpha_ns"], kw["beta_gbs"], rb)
            assert ms[r] == ref["makespan"]


def test_schedule_at_the_bench_shape():
    """Eight ranks of 4096 tokens x top-8 over 288 physical experts with a
    Zipf-skewed histogram (rows as the bench's split run moves them)."""
    rng = np.random.default_rng(7)
    R, P = 8, 288
    pop = 1.0 / (1 + rng.permutation(P)) ** 1.2
    counts = np.stack([rng.multinomial(4096 * 8, pop / pop.sum()) for _ in range(R)]).astype(np.int32)
    desc = ep.make_desc(R, P, 76)
    for direction, rb in ((0, 7168 + 224), (1, 2 * 7168)):
        for puller in (0, 3, 7):
            got = ep.schedule(desc, direction, puller, counts, rb)
            ref = oracle.ep_schedule(direction, puller, counts, 76, list(desc.fanout_cap), list(desc.unit_rows),
                                     list(desc.alpha_ns), list(desc.beta_gbs), rb)
            _same_schedule(got, ref, f"bench shape dir {direction} puller {puller}")


def test_hand_worked_schedules_through_the_library():
    data = json.load(open(os.path.join(GOLDEN, "ep_schedule.json")))
    for case in data["cases"]:
        counts = np.array(case["counts"], np.int32)
        R, P = counts.shape
        desc = ep.make_desc(R, P, case["C"], case["cap"], case["unit_rows"], case["alpha_ns"], case["beta_gbs"])
        r = ep.schedule(desc, case["direction"], case["puller"], counts, case["row_bytes"])
        got = [[list(map(int, (u["peer"], u["src_row"], u["dst_row"], u["rows"])))
                for u in r["units"][r["core_off"][c]:r["core_off"][c + 1]]] for c in range(case["C"])]
        assert got == case["core_units"], case["name"]
        assert r["makespan"] == case["makespan"], case["name"]


def test_empty_and_degenerate_groups():
    desc = ep.make_desc(3, 2, 4)  # P < R: rank 2 owns nothing
    counts = np.array([[0, 5], [3, 0], [0, 0]], np.int32)
    assert ep.experts(3, 2, 0) == (0, 1) and ep.experts(3, 2, 1) == (1, 1) and ep.experts(3, 2, 2) == (2, 0)
    for d in range(3):
        for direction in (0, 1):
            got = ep.schedule(desc, direction, d, counts, 16)
            ref = oracle.ep_schedule(direction, d, counts, 4, list(desc.fanout_cap), list(desc.unit_rows),
                                     list(desc.alpha_ns), list(desc.beta_gbs), 16)
            _same_schedule(got, ref, f"P<R d {d} dir {direction}")
    z = np.zeros((4, 16), np.int32)
    r = ep.schedule(ep.make_desc(4, 16, 8), 0, 2, z, 100)
    assert len(r["units"]) == 0 and (r["core_off"] == 0).all() and r["makespan"] == 0


def test_max_units_bounds_every_schedule():
    rng = np.random.default_rng(3)
    for _ in range(30):
        R, P, counts, kw = _random_case(rng)
        desc = ep.make_desc(R, P, kw["cores"], kw["fanout_cap"], kw["unit_rows"], kw["alpha_ns"], kw["beta_gbs"])
        for direction in (0, 1):
            for puller in range(R):
                moved = counts[:, [p for p in range(P) if p * R // P == puller]].sum() if direction == 0 \
                    else counts[puller].sum()
                bound = ep.max_units(desc, int(moved))
                n = len(ep.schedule(desc, direction, puller, counts, 64, cap_units=bound)["units"])
                assert n <= bound


def test_argument_checks():
    L = ep.lib()
    counts = np.zeros((2, 4), np.int32)
    u = np.zeros(8, ep.UNIT)
    off = np.zeros(9, np.int32)
    n, ms = ctypes.c_int32(), ctypes.c_int64()

    def sched(desc, direction=0, puller=0, rb=64, cap=8, cnt=counts):
        return L.moe_ep_schedule(ctypes.byref(desc), direction, puller, cnt.ctypes.data_as(ctypes.c_void_p), rb,
                                 u.ctypes.data_as(ctypes.c_void_p), cap, ctypes.byref(n),
                                 off.ctypes.data_as(ctypes.c_void_p), ctypes.byref(ms))

    good = ep.make_desc(2, 4, 8)
    assert sched(good) == 0
    assert sched(ep.make_desc(0, 4, 8)) == -2
    assert sched(ep.make_desc(65, 4, 8)) == -2
    assert sched(ep.make_desc(2, 4, 0)) == -2
    assert sched(ep.make_desc(2, 4, 8, fanout_cap=(0, 1))) == -2
    assert sched(ep.make_desc(2, 4, 8, unit_rows=(1, (1 << 20) + 1))) == -2
    assert sched(ep.make_desc(2, 4, 8, beta_gbs=(0, 5))) == -2
    assert sched(good, direction=2) == -2
    assert sched(good, puller=2) == -2
    assert sched(good, rb=0) == -2
    assert sched(good, cnt=np.array([[1, -1, 0, 0], [0, 0, 0, 0]], np.int32)) == -2
    full = np.full((2, 4), 50, np.int32)
    assert sched(ep.make_desc(2, 4, 8, unit_rows=(1, 1)), cnt=full, cap=8) == -2  # more units than room
    assert L.moe_ep_schedule(ctypes.byref(good), 0, 0, None, 64, None, 8, ctypes.byref(n), None, None) == -1
    # pull: host checks before any launch (no GPU here: a launch could only fail with -6)
    p = ep.Plane()
    p.row_bytes = 24  # not a multiple of 16
    dev = ctypes.c_void_p(1 << 41)
    assert L.moe_ep_pull(dev, dev, 1, 2, 8, 0, 2, ctypes.byref(p), 1, dev, None) == -2
    p.row_bytes = 32
    assert L.moe_ep_pull(dev, dev, 1, 2, 8, 1, 2, ctypes.byref(p), 1, dev, None) == -2  # pullers past R
    assert L.moe_ep_pull(dev, dev, 1, 2, 8, 0, 2, ctypes.byref(p), 3, dev, None) == -2  # 3 planes
    p.src[0] = (1 << 41) + 8
    assert L.moe_ep_pull(dev, dev, 1, 2, 8, 0, 2, ctypes.byref(p), 1, dev, None) == -3
    assert L.moe_ep_pull(dev, None, 1, 2, 8, 0, 2, ctypes.byref(p), 1, dev, None) == -1
    assert L.moe_dequant_rows(dev, dev, 4, 200, 4, dev, None) == -2
    assert L.moe_dequant_rows(dev, dev, 4, 256, 2, dev, None) == -2
    assert L.moe_dequant_rows(None, dev, 4, 256, 4, dev, None) == -1
    assert L.moe_dequant_rows(None, None, 0, 256, 4, None, None) == 0


@pytest.mark.filterwarnings("ignore:This process .* is multi-threaded:DeprecationWarning")
def test_group_schedules_from_two_threads_at_once_and_after_fork():
    """The group call's worker threads serve one call at a time; a call that
    finds them busy computes on its own thread, and so does a process forked
    after they started.  Every result equals the per-puller schedules."""
    import concurrent.futures as cf
    import multiprocessing as mp
    rng = np.random.default_rng(77)
    R, P = 8, 288
    counts = rng.integers(0, 400, size=(R, P)).astype(np.int32)
    desc = ep.make_desc(R, P, 40)
    want = {d: ep.pack_schedules([ep.schedule(desc, d, r, counts, 1000) for r in range(R)]) for d in (0, 1)}
    ep.schedule_group(desc, 0, counts, 1000)  # the workers exist from here on

    def one(d):
        units, core_off, _ = ep.schedule_group(desc, d, counts, 1000)
        return d, units, core_off

    with cf.ThreadPoolExecutor(4) as ex:
        for d, units, core_off in ex.map(one, [0, 1, 0, 1, 1, 0, 0, 1] * 3):
            np.testing.assert_array_equal(units, want[d][0])
            np.testing.assert_array_equal(core_off, want[d][1])
    import torch
    if torch.cuda.is_available() and torch.cuda.is_initialized():
        return  # no fork once a CUDA context exists in this process
    ctx = mp.get_context("fork")
    q = ctx.Queue()
    p = ctx.Process(target=_forked_group_call, args=(q, counts))
    p.start()
    units, core_off = q.get(timeout=120)
    p.join(timeout=60)
    assert p.exitcode == 0
    np.testing.assert_array_equal(units, want[0][0])
    np.testing.assert_array_equal(core_off, want[0][1])


def _forked_group_call(q, counts):
    desc = ep.make_desc(8, 288, 40)
    units, core_off, _ = ep.schedule_group(desc, 0, counts, 1000)
    q.put((units, core_off))


@pytest.mark.parametrize("seed", range(6))
def test_recv_start_follows_the_oracle_layout(seed):
    rng = np.random.default_rng(300 + seed)
    R = int(rng.integers(1, 9))
    P = int(rng.integers(1, 40))
    counts = rng.integers(0, 50, size=(R, P)).astype(np.int32)
    counts[rng.random((R, P)) < 0.2] = 0
    for s in range(R):
        st = ep.recv_start(counts, s)
        for d in range(R):
            _, chunk = oracle.ep_layout(counts, d)
            mine = [p for p in range(P) if oracle.ep_owner(p, R, P) == d]
            for i, p in enumerate(mine):
                assert st[p] == chunk[s, i]


def test_fused_combine_checks_before_launch():
    """moe_ep_combine rejects bad arguments on the host (no GPU here: a call
    that got past the checks could only fail with MOE_ERR_CUDA, -6)."""
    import ctypes
    from combine_moe_plan_gb300 import moe
    L = ep.lib()
    d = moe.Desc(64, 256, 8, 8, 2, 128, 1)
    n = ctypes.c_size_t()
    assert L.moe_pool_bytes(ctypes.byref(d), ctypes.byref(n)) == 0
    h = ctypes.c_void_p()
    assert L.moe_pool_init(ctypes.byref(d), ctypes.c_void_p(1 << 40), n.value, ctypes.byref(h)) == 0
    ptrs = (ctypes.c_void_p * 2)(1 << 41, 1 << 41)
    rows = (ctypes.c_int64 * 2)(10, 10)
    good = ctypes.c_void_p(1 << 41)
    assert L.moe_ep_combine(None, 8, 0, 2, ptrs, rows, good, None, good, None) == -1
    assert L.moe_ep_combine(h, 8, 1, 2, ptrs, rows, good, None, good, None) == -4     # no set 1
    assert L.moe_ep_combine(h, 65, 0, 2, ptrs, rows, good, None, good, None) == -2    # T > T_max
    assert L.moe_ep_combine(h, 8, 0, 65, ptrs, rows, good, None, good, None) == -2    # R too large
    assert L.moe_ep_combine(h, 8, 0, 2, ptrs, rows, good, None, good, None) == -9     # no plan on this set
    L.moe_pool_destroy(h)


def test_group_schedules_from_several_host_threads():
    """Four host threads make group schedules at once: one holds the library's
    worker threads, the others find them busy and compute on their own
    thread; every result equals the single-puller schedules."""
    import threading
    errors = []

    def run(seed):
        try:
            rng = np.random.default_rng(3000 + seed)
            for _ in range(6):
                R, P, counts, kw = _random_case(rng)
                desc = ep.make_desc(R, P, kw["cores"], kw["fanout_cap"], kw["unit_rows"], kw["alpha_ns"],
                                    kw["beta_gbs"])
                units, core_off, _ = ep.schedule_group(desc, 1, counts, 2 * 7168)
                want_u, want_off = ep.pack_schedules([ep.schedule(desc, 1, r, counts, 2 * 7168) for r in range(R)])
                np.testing.assert_array_equal(units, want_u)
                np.testing.assert_array_equal(core_off, want_off)
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors

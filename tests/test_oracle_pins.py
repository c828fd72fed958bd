"""Pins for the CPU oracle: brute force, closed forms, hand-worked cases,
exact rational arithmetic and invariants.  Each test is chosen so that a
plausible slip in the oracle (wrong tie order, dropped term, transposed index,
wrong rounding mode, wrong accumulation order) fails at least one of them.

Nothing here calls the CUDA library.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from combine_moe_plan_gb300 import workloads as wl
from tests import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(vals):
    return wl.f32_to_bf16_bits(np.asarray(vals, np.float32))


# ------------------------------------------------------------------ top-k --

def _topk_brute(logits, k):
    T, E = logits.shape
    out = np.empty((T, k), np.int32)
    ids = np.arange(E)
    for t in range(T):
        order = np.lexsort((ids, -logits[t].astype(np.float64)))  # primary: logit desc
        out[t] = order[:k]
    return out


@pytest.mark.parametrize("E,k", [(4, 1), (4, 4), (8, 2), (13, 5), (40, 8), (256, 8), (64, 6)])
def test_topk_matches_full_sort_with_ties(E, k):
    rng = np.random.default_rng(E * 100 + k)
    # Few distinct values so that ties are frequent; includes +0.0 and -0.0.
    vals = np.array([-1.5, -0.0, 0.0, 0.25, 0.25, 2.0, 3.0], np.float32)
    logits = rng.choice(vals, size=(200, E)).astype(np.float32)
    topk_e, gates, phys = oracle.route(logits, k)
    np.testing.assert_array_equal(topk_e, _topk_brute(logits, k))
    np.testing.assert_array_equal(phys, topk_e)


def test_topk_k_equals_E_is_permutation():
    logits = np.random.default_rng(1).standard_normal((50, 16)).astype(np.float32)
    topk_e, _, _ = oracle.route(logits, 16)
    for row in topk_e:
        assert sorted(row.tolist()) == list(range(16))
    # descending logits along j
    lv = np.take_along_axis(logits, topk_e, axis=1)
    assert np.all(np.diff(lv, axis=1) <= 0)


# ------------------------------------------------------------------ gates --

def test_gates_special_values():
    # k = 1: exp(0)/exp(0) = 1 exactly
    _, g, _ = oracle.route(np.array([[0.3, -2.0, 7.0]], np.float32), 1)
    assert g[0, 0] == np.float32(1.0)
    # two equal logits -> 1/2 each; three equal -> RN(1/3)
    _, g, _ = oracle.route(np.array([[5.0, 5.0, -1.0]], np.float32), 2)
    assert g[0].tolist() == [0.5, 0.5]
    _, g, _ = oracle.route(np.array([[1.0, 1.0, 1.0, -9.0]], np.float32), 3)
    assert all(v == np.float32(1.0 / 3.0) for v in g[0])


def test_gates_are_correctly_rounded_softmax():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    rng = np.random.default_rng(7)
    logits = (rng.standard_normal((300, 32)) * 2).astype(np.float32)
    k = 8
    topk_e, gates, _ = oracle.route(logits, k)
    checked = 0
    for t in range(logits.shape[0]):
        sel = [mpmath.mpf(float(logits[t, e])) for e in topk_e[t]]
        exs = [mpmath.exp(v - sel[0]) for v in sel]
        s = mpmath.fsum(exs)
        for j in range(k):
            q = exs[j] / s
            man, e2 = mpmath.frexp(q)
            # exact binary value of the 200-bit approximation
            fr = Fraction(int(mpmath.ldexp(man, 200)), 2 ** (200 - int(e2)))
            ref = exact.to_f32(fr)
            # skip values within 2^-45 (relative) of an fp32 rounding midpoint:
            # there fp64 intermediate rounding may legitimately decide the tie
            ulp = Fraction(2) ** (math.floor(math.log2(float(ref))) - 23)
            mid_dist = abs(fr - exact.round_rne(fr, 24)) - ulp / 2
            if abs(mid_dist) < fr * Fraction(1, 2 ** 45):
                continue
            assert gates[t, j] == ref, (t, j, gates[t, j], ref)
            checked += 1
    assert checked > 2000


def test_gates_sum_and_monotone():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((500, 64)).astype(np.float32)
    _, g, _ = oracle.route(logits, 6)
    assert np.all(np.abs(g.astype(np.float64).sum(1) - 1.0) <= 6 * 2.0 ** -24)
    assert np.all(np.diff(g, axis=1) <= 0)  # logits descend along j


# --------------------------------------------------------------- replicas --

def test_identity_replica_map_equals_no_map():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((100, 12)).astype(np.float32)
    off = np.arange(13, dtype=np.int32)
    ids = np.arange(12, dtype=np.int32)
    a = oracle.route(logits, 3)
    b = oracle.route(logits, 3, off, ids, 12)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_replica_split_is_token_index_mod_count():
    w = wl.small_variant(wl.WORKLOADS["t4096_h7168_e256p288_k8"], 512)
    logits = wl.make_logits(w)
    off, ids = wl.make_replica_map(w)
    topk_e, _, phys = oracle.route(logits, w.k, off, ids, w.P)
    n_rep = np.diff(off)
    assert (n_rep == 2).sum() == 32 and sorted(ids.tolist()) == list(range(w.P))
    for t in range(w.T):
        for j in range(w.k):
            e = topk_e[t, j]
            assert phys[t, j] == ids[off[e] + t % n_rep[e]]
    # every hot expert's copies split between its two replicas by token parity
    for e in np.nonzero(n_rep == 2)[0]:
        toks = np.nonzero((topk_e == e).any(1))[0]
        on_second = np.isin(phys[toks], [ids[off[e] + 1]]).any(1)
        np.testing.assert_array_equal(on_second, toks % 2 == 1)


# -------------------------------------------------------------- placement --

def _place_brute(phys, P):
    T, k = phys.shape
    keys = [(int(phys[t, j]), t, j) for t in range(T) for j in range(k)]
    keys.sort()  # by expert, then token (stable window order)
    slot = np.empty((T, k), np.int32)
    for r, (_, t, j) in enumerate(keys):
        slot[t, j] = r
    counts = np.bincount(phys.ravel(), minlength=P).astype(np.int32)
    return counts, slot


@pytest.mark.parametrize("T,k,P", [(1, 1, 1), (37, 3, 5), (200, 8, 288), (64, 2, 8), (500, 6, 64)])
def test_place_matches_sort(T, k, P):
    rng = np.random.default_rng(T + k + P)
    # distinct experts per token, skewed toward low ids
    phys = np.empty((T, k), np.int32)
    w = 1.0 / np.arange(1, P + 1) ** 1.2
    w /= w.sum()
    for t in range(T):
        phys[t] = rng.choice(P, size=k, replace=False, p=w)
    out = oracle.place(phys, P)
    counts, slot = _place_brute(phys, P)
    np.testing.assert_array_equal(out["counts"], counts)
    np.testing.assert_array_equal(out["slot"], slot)
    off = out["offsets"]
    assert off[0] == 0 and off[-1] == T * k
    np.testing.assert_array_equal(np.diff(off), counts)
    # inverse map and bijection
    assert sorted(out["slot"].ravel().tolist()) == list(range(T * k))
    for t in range(T):
        for j in range(k):
            r = out["slot"][t, j]
            assert out["src_token"][r] == t and out["src_k"][r] == j
    # tokens ascend inside each window
    for p in range(P):
        win = out["src_token"][off[p]:off[p + 1]]
        assert np.all(np.diff(win) > 0)


def test_place_rejects_duplicate_expert_in_token():
    with pytest.raises(oracle.OracleError):
        oracle.place(np.array([[1, 1]], np.int32), 4)


def test_place_everyone_on_one_expert():
    T = 300
    phys = np.zeros((T, 1), np.int32)
    out = oracle.place(phys, 4)
    assert out["counts"].tolist() == [T, 0, 0, 0]
    np.testing.assert_array_equal(out["slot"][:, 0], np.arange(T))


# ----------------------------------------------------------- quantization --

def test_quant_half_even_ties_and_scale():
    x = np.zeros((1, 128), np.float32)
    x[0, :6] = [254, 1, 3, 5, -3, 0.5]
    codes, scales = oracle.quantize(_bf16(x))
    assert scales[0, 0] == np.float32(2.0)
    assert codes[0, :6].tolist() == [127, 0, 2, 2, -2, 0]


def test_quant_zero_group_and_extremes():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((40, 512)).astype(np.float32)
    x[3, 128:256] = 0.0
    x[4, 0:128] = -0.0
    codes, scales = oracle.quantize(_bf16(x))
    assert scales[3, 1] == 0 and not codes[3, 128:256].any()
    assert scales[4, 0] == 0 and not codes[4, 0:128].any()
    g = codes.reshape(40, 4, 128).astype(np.int32)
    nz = scales != 0
    assert np.all(np.abs(g).max(-1)[nz] == 127)  # the amax element maps to +-127
    assert codes.min() >= -127  # -128 never occurs


def test_quant_error_bound():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((64, 1024)) * rng.uniform(0.01, 100, (64, 1))).astype(np.float32)
    xb = _bf16(x)
    xf = wl.bf16_bits_to_f32(xb).astype(np.float64).reshape(64, 8, 128)
    codes, scales = oracle.quantize(xb)
    amax = np.abs(xf).max(-1, keepdims=True)
    s = scales.astype(np.float64)[..., None]
    err = np.abs(xf - codes.astype(np.float64).reshape(64, 8, 128) * s)
    assert np.all(err <= s * (0.5 + 2.0 ** -16) + amax * 2.0 ** -23)


def test_quant_exhaustive_against_double_rounding_identity():
    """Every finite bf16 x against a spread of amax values: the code must be
    rint of the correctly rounded binary32 quotient.  The quotient of two
    binary32 numbers computed in binary64 and then rounded to binary32 is the
    correctly rounded binary32 quotient (Figueroa, 'When is double rounding
    innocuous?', 1995: 53 >= 2*24 + 2), which gives a reference independent
    of the C library's binary32 division."""
    allx = wl.bf16_bits_to_f32(np.arange(0x10000, dtype=np.uint16))
    allx = allx[np.isfinite(allx)]
    amaxes = []
    for e in (-100, -20, -3, 1, 7, 40, 100):
        for m in (1.0, 1.0078125, 1.5, 1.9921875, 1.3359375, 1.75):
            amaxes.append(np.float32(m * 2.0 ** e))
    for e in (0, 60):  # every bf16 significand as amax
        for m in range(128):
            amaxes.append(np.float32((1.0 + m / 128.0) * 2.0 ** e))
    amaxes.append(np.float32(254.0))
    amaxes += [wl.bf16_bits_to_f32(np.array([b], np.uint16))[0] for b in (0x0001, 0x0003, 0x0040, 0x007F)]
    rows = []
    for a in amaxes:
        xs = allx[np.abs(allx) <= a]
        # x * 127 must stay finite and exact; drop values that would overflow
        xs = xs[np.abs(xs) < 2.0 ** 120]
        pad = (-len(xs)) % 127
        xs = np.concatenate([xs, np.zeros(pad, np.float32)]).reshape(-1, 127)
        grp = np.concatenate([np.full((xs.shape[0], 1), a, np.float32), xs], axis=1)
        rows.append(grp)
    groups = np.concatenate(rows)  # each row: amax first, then 127 values
    xb = wl.f32_to_bf16_bits(groups)  # exact: all values are bf16 already
    codes, scales = oracle.quantize(xb)
    gx = groups.astype(np.float64)
    am = gx[:, :1]
    q64 = (gx * 127.0) / am  # x*127 is exact in binary32 and in binary64
    ref = np.rint(q64.astype(np.float32)).astype(np.int32)
    np.testing.assert_array_equal(codes.astype(np.int32), ref)
    np.testing.assert_array_equal(scales[:, 0], (am[:, 0] / 127.0).astype(np.float32))
    assert groups.size > 8_000_000


# ------------------------------------------------------------------ combine --

def test_combine_k1_copies_row():
    rng = np.random.default_rng(13)
    ex = _bf16(rng.standard_normal((10, 256)))
    slot = rng.permutation(10).astype(np.int32)[:, None]
    y = oracle.combine(ex, slot, np.ones((10, 1), np.float32))
    np.testing.assert_array_equal(y, ex[slot[:, 0]])


def test_combine_equal_rows_gates_sum_to_one():
    rng = np.random.default_rng(14)
    row = _bf16(rng.standard_normal((1, 256)))
    ex = np.repeat(row, 2, axis=0)
    y = oracle.combine(ex, np.array([[0, 1]], np.int32), np.array([[0.25, 0.75]], np.float32))
    np.testing.assert_array_equal(y[0], row[0])


def test_combine_is_exact_fma_chain():
    """Each step of the accumulation is one correctly rounded a*b+c in binary32,
    in ascending j, then one bf16 rounding: checked with exact rationals."""
    rng = np.random.default_rng(15)
    T, k, H = 6, 5, 128
    ex = _bf16(rng.standard_normal((T * k, H)) * 3)
    slot = rng.permutation(T * k).astype(np.int32).reshape(T, k)
    gates = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    y = oracle.combine(ex, slot, gates)
    for t in range(T):
        for i in range(0, H, 7):
            acc = Fraction(0)
            for j in range(k):
                g = exact.f32_exact(gates[t, j])
                v = exact.bf16_bits_exact(ex[slot[t, j], i])
                acc = Fraction(float(exact.to_f32(g * v + acc)))
            assert int(y[t, i]) == exact.to_bf16_bits(acc), (t, i)


def test_combine_order_matters_fixture():
    """Accumulation order is observable: with rows 1, 2^-8, 2^-24, 2^-24 and
    unit gates, ascending j lands exactly on the bf16 midpoint 1 + 2^-8 (each
    2^-24 is a binary32 half-ulp tie that rounds to even) and y = 1; the
    reverse order first sums the small terms to 2^-8 + 2^-23, lands above the
    midpoint and rounds up to 1 + 2^-7."""
    ex = _bf16(np.array([[1.0] * 128, [2.0 ** -8] * 128, [2.0 ** -24] * 128, [2.0 ** -24] * 128],
                        np.float32))
    gates = np.ones((1, 4), np.float32)
    y = oracle.combine(ex, np.array([[0, 1, 2, 3]], np.int32), gates)
    assert int(y[0, 0]) == 0x3F80
    y2 = oracle.combine(ex, np.array([[3, 2, 1, 0]], np.int32), gates)
    assert int(y2[0, 0]) == 0x3F81


def test_combine_uses_fused_multiply_add():
    """A case where one rounding per step (fma) and two (multiply, then add)
    differ after the bf16 rounding: rows 1 and 1 + 2^-7, gates 1 and the
    binary32 value with bits 0x3B7E04F7 (about 2^-8 / (1 + 2^-7)).  The exact
    product sits just above 2^-8 + 2^-24, so fma gives 1 + 2^-8 + 2^-23 and y
    rounds up to 1 + 2^-7; rounding the product first lands on the binary32
    tie 1 + 2^-8 + 2^-24, which rounds to even, and y = 1."""
    g1 = np.array([0x3B7E04F7], np.uint32).view(np.float32)[0]
    ex = _bf16(np.array([[1.0] * 128, [1.0 + 2.0 ** -7] * 128], np.float32))
    y = oracle.combine(ex, np.array([[0, 1]], np.int32), np.array([[1.0, g1]], np.float32))
    exp_fma = exact.to_bf16_bits(Fraction(float(exact.to_f32(
        1 + exact.f32_exact(g1) * exact.bf16_bits_exact(0x3F81)))))
    prod = Fraction(float(exact.to_f32(exact.f32_exact(g1) * exact.bf16_bits_exact(0x3F81))))
    exp_two_roundings = exact.to_bf16_bits(Fraction(float(exact.to_f32(1 + prod))))
    assert (exp_fma, exp_two_roundings) == (0x3F81, 0x3F80)
    assert int(y[0, 0]) == 0x3F81


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(16)
    a = rng.standard_normal(100000).astype(np.float32) * 10
    ties = wl.bf16_bits_to_f32(rng.integers(0, 0x7F00, 2000, dtype=np.uint16))
    ties = (ties.view(np.uint32) | np.uint32(0x8000)).view(np.float32)  # exact halfway points
    a = np.concatenate([a, ties, -ties, np.float32([0.0, -0.0, 1e-40, 3.4e38])])
    ours = oracle.f32_to_bf16(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ------------------------------------------------------------ whole path --

def test_handworked_golden_cases():
    with open(os.path.join(GOLDEN, "handworked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        logits = np.array(c["logits"], np.float32)
        pl = oracle.plan(logits, c["k"], np.array(c.get("rep_off"), np.int32) if "rep_off" in c else None,
                         np.array(c.get("rep_ids"), np.int32) if "rep_ids" in c else None, c["P"])
        for key in ("topk_e", "gates", "phys", "counts", "offsets", "slot", "src_token", "src_k"):
            np.testing.assert_array_equal(pl[key], np.array(c[key]), err_msg=f"{c['name']}:{key}")
        if "x_head" not in c:
            continue
        x = np.zeros((c["T"], c["H"]), np.float32)
        for t, head in enumerate(c["x_head"]):
            x[t, :len(head)] = head
        out = oracle.forward(logits, _bf16(x), c["k"], P=c["P"])
        codes = out["codes"]
        for t, head in enumerate(c["codes_head"]):
            for j in range(c["k"]):
                r = c["slot"][t][j]
                np.testing.assert_array_equal(codes[r, :len(head)], head)
                assert not codes[r, len(head):].any()
                assert out["scales"][r].tolist() == c["scales"][t]
        yf = wl.bf16_bits_to_f32(out["y"])
        for t, head in enumerate(c["y_head"]):
            np.testing.assert_array_equal(yf[t, :len(head)], head)
            assert not yf[t, len(head):].any()


@pytest.mark.parametrize("name,T", [("t64_h256_e8_k2", 64), ("t96_h7168_e256_k8", 96),
                                    ("t4096_h7168_e256p288_k8", 64), ("t16384_h2048_e64_k6", 128)])
def test_roundtrip_invariant(name, T):
    """dispatch -> identity experts (dequantize) -> combine recovers x within
    the INT8 rounding bound plus two bf16 roundings."""
    w = wl.small_variant(wl.WORKLOADS[name], T)
    inp = wl.make_inputs(w, with_expert_out=False)
    out = oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"], w.P)
    x = wl.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    y = wl.bf16_bits_to_f32(out["y"]).astype(np.float64)
    q, s = oracle.quantize(inp["x"])
    scale = np.repeat(s.astype(np.float64), 128, axis=1)
    bound = scale * (0.5 + 2.0 ** -12) + 2.0 ** -7 * (np.abs(x) + 0.5 * scale) + 127 * scale * 2.0 ** -20
    assert np.all(np.abs(y - x) <= bound)
    # codes in every slot row equal the token's own quantization
    for t in range(T):
        for j in range(w.k):
            r = out["slot"][t, j]
            np.testing.assert_array_equal(out["codes"][r], q[t])


def test_page_sizes():
    """The bytes model used for the roofline against the sizes the pages print."""
    with open(os.path.join(GOLDEN, "page_sizes.json")) as f:
        pg = json.load(f)
    H = pg["hidden"]
    assert H * 2 == pg["bf16_kb_per_token"] * 1024
    assert pg["local_batch"] * pg["ep_dies"] == pg["global_batch"]
    assert pg["routed_experts"] + pg["shared_experts"] + pg["redundant_experts"] == pg["ep_dies"]
    row_kib = pg["int8_kb_per_token_incl_scale"]
    total = pg["global_batch"] * (row_kib * 1024 + pg["bf16_kb_per_token"] * 1024)
    assert round(total / 2 ** 20) == pg["buffers_mb_per_die"]
    # our dispatch row (codes + one fp32 scale per 128 elements) fits the page's row
    assert H + (H // 128) * 4 <= row_kib * 1024
    w = wl.WORKLOADS["t4096_h7168_e256p288_k8"]
    assert (w.T, w.H, w.k) == (pg["microbench_tokens"], H, pg["microbench_topk"])
    b = w.algorithmic_bytes()
    assert b["dispatch"] == w.T * (H * 2 + w.k * (H + (H // 128) * 4) + w.k * 4)
    assert b["combine"] == w.T * (w.k * H * 2 + w.k * 8 + H * 2)

"""The oracle's per-token loops may run on several host threads (OpenMP).
Each token's arithmetic does not depend on the thread count, so every output
must be byte-identical to the single-thread run, and when several tokens are
outside the method's domain the error reported is the lowest token's, as a
serial loop gives.

Nothing here calls the CUDA library.
"""
import numpy as np
import pytest

import oracle
from combine_moe_plan_gb300 import workloads as wl


@pytest.fixture
def restore_threads():
    n = oracle.threads()
    yield
    oracle.set_threads(n)


def _forward(w, inp):
    return oracle.forward(inp["logits"], inp["x"], w.k, inp["rep_off"], inp["rep_ids"], w.P,
                          ex_out=inp.get("ex_out"))


@pytest.mark.parametrize("name", ["t4096_h7168_e256p288_k8", "t16384_h2048_e64_k6", "t96_h7168_e256_k8"])
def test_outputs_identical_for_any_thread_count(name, restore_threads):
    w = wl.small_variant(wl.WORKLOADS[name], T=203)
    inp = wl.make_inputs(w)
    if "ex_out" in inp:
        inp["ex_out"] = inp["ex_out"][: w.T * w.k]
    oracle.set_threads(1)
    one = _forward(w, inp)
    assert oracle.set_threads(4) in (1, 4)  # 1 where gcc had no OpenMP
    many = _forward(w, inp)
    assert one.keys() == many.keys()
    for key in one:
        assert one[key].tobytes() == many[key].tobytes(), key
    tok = np.array([202, 0, 77, 77, 5], np.int32)
    a = oracle.combine_tokens(one["ex_out"], one["slot"], one["gates"], tok)
    np.testing.assert_array_equal(a, one["y"][tok])


def _bad_batch(nan_token, replica_token):
    """E = 8, k = 2: every token's top expert is 1 except replica_token's,
    which is 0, whose replica list is empty; nan_token holds a NaN logit."""
    T, E = 64, 8
    logits = np.tile(np.linspace(0.0, -1.0, E, dtype=np.float32), (T, 1))
    logits[:, 0] = -5.0
    logits[:, 1] = 2.0
    logits[replica_token, 0] = 3.0
    logits[nan_token, 5] = np.nan
    rep_off = np.array([0, 0, 1, 2, 3, 4, 5, 6, 7], np.int32)  # expert 0 has no replica
    rep_ids = np.arange(1, 8, dtype=np.int32)
    return logits, rep_off, rep_ids


@pytest.mark.parametrize("nan_token,replica_token,expected", [
    (50, 3, "malformed replica map"),
    (3, 50, "non-finite input"),
])
def test_lowest_bad_token_decides_the_error(nan_token, replica_token, expected, restore_threads):
    logits, rep_off, rep_ids = _bad_batch(nan_token, replica_token)
    for n in (1, 4):
        oracle.set_threads(n)
        with pytest.raises(oracle.OracleError, match=expected):
            oracle.route(logits, 2, rep_off, rep_ids, 8)


def test_quantize_finds_a_bad_token_on_any_thread(restore_threads):
    x = np.zeros((40, 128), np.float32)
    x[30, 3] = np.inf
    xb = wl.f32_to_bf16_bits(x)
    for n in (1, 4):
        oracle.set_threads(n)
        with pytest.raises(oracle.OracleError, match="non-finite"):
            oracle.quantize(xb)

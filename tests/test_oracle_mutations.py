"""The oracle's pins must catch plausible mistakes.  Each case below plants one
mistake in a temporary copy of oracle/moe_oracle.c (never in the committed
file), builds that copy, and runs tests/test_oracle_pins.py against it: the
run must fail.  The unchanged copy must pass, so a failure is the mistake's.
Host only (gcc, no GPU)."""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in moe_oracle.c, replacement)
MUTATIONS = [
    ("tie order: higher expert id first",
     "return (a->e < b->e) ? -1 : (a->e > b->e);",
     "return (a->e > b->e) ? -1 : (a->e < b->e);"),
    ("codes rounded half away from zero",
     "q = (int8_t)(int32_t)rintf(quo);",
     "q = (int8_t)(int32_t)roundf(quo);"),
    ("gates exponentials in fp32",
     "ex[j] = exp((double)c[j].v - (double)c[0].v);",
     "ex[j] = (double)expf(c[j].v - c[0].v);"),
    ("gate quotient of values rounded to fp32",
     "gates[j] = (float)(ex[j] / s);",
     "gates[j] = (float)ex[j] / (float)s;"),
    ("replica picked with the wrong token index",
     "p = rep_ids[lo + (t % n)];",
     "p = rep_ids[lo + ((t + 1) % n)];"),
    ("scale by a reciprocal",
     "scales[g] = amax / 127.0f;",
     "scales[g] = amax * (1.0f / 127.0f);"),
    ("quotient perturbed by one part in 10^7",
     "float num = v * 127.0f;",
     "float num = v * 127.0f * 1.0000001f;"),
    ("signed amax",
     "if (a > amax) amax = a;",
     "if (v > amax) amax = v;"),
    ("combine without fma",
     "acc = fmaf(gates[j], orc_bf16_to_f32(ex_out[(size_t)slot[j] * H + i]), acc);",
     "acc = gates[j] * orc_bf16_to_f32(ex_out[(size_t)slot[j] * H + i]) + acc;"),
    ("combine accumulated in descending j",
     "for (int32_t j = 0; j < k; ++j)\n            acc = fmaf(",
     "for (int32_t j = k - 1; j >= 0; --j)\n            acc = fmaf("),
    ("bf16 rounding half up instead of half to even",
     "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;",
     "if (rest >= 0x8000u) keep += 1u;"),
    ("one slot written to the wrong copy",
     "slot[(size_t)t * k + j] = r;",
     "slot[(size_t)t * k + j] = r; if (j == 1 && t == 0) slot[0] = r;"),
    ("amax over the first 127 elements of a group",
     "for (int32_t i = 0; i < 128; ++i) {\n            float v = orc_bf16_to_f32(xs[i]);\n            if (!isfinite(v))",
     "for (int32_t i = 0; i < 127; ++i) {\n            float v = orc_bf16_to_f32(xs[i]);\n            if (!isfinite(v))"),
    ("tokens placed in descending order within a window",
     "    for (int32_t t = 0; t < T; ++t) {\n        for (int32_t j = 0; j < k; ++j) {\n"
     "            int32_t p = phys[(size_t)t * k + j];\n            int32_t r = cursor[p];",
     "    for (int32_t t = T - 1; t >= 0; --t) {\n        for (int32_t j = 0; j < k; ++j) {\n"
     "            int32_t p = phys[(size_t)t * k + j];\n            int32_t r = cursor[p];"),
    ("gate sum accumulated in fp32",
     "    double s = 0.0;\n    for (int32_t j = 0; j < k; ++j) {\n        ex[j] = exp(",
     "    float s = 0.0f;\n    for (int32_t j = 0; j < k; ++j) {\n        ex[j] = exp("),
    ("bf16 rounding by truncation",
     "    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;",
     "    (void)rest;"),
    ("replica picked by expert id instead of token index",
     "p = rep_ids[lo + (t % n)];",
     "p = rep_ids[lo + (e % n)];"),
    ("combine with uniform weights instead of the gates",
     "acc = fmaf(gates[j], orc_bf16_to_f32(",
     "acc = fmaf(1.0f / (float)k, orc_bf16_to_f32("),
    ("identity experts with the next group's scale",
     "scales[(size_t)r * G + i / 128]",
     "scales[(size_t)r * G + (i / 128 + 1) % G]"),
    ("top-k by absolute logit",
     "    if (a->v > b->v) return -1;\n    if (a->v < b->v) return 1;",
     "    if (fabsf(a->v) > fabsf(b->v)) return -1;\n    if (fabsf(a->v) < fabsf(b->v)) return 1;"),
]


def _copy_tree(dst: str) -> None:
    """The oracle, the pin tests and what they import, without build output."""
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ("__init__.py", "moe_oracle.c", "moe_oracle_ep.c"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, "oracle", f))
    os.makedirs(os.path.join(dst, "combine_moe_plan_gb300"))
    for f in ("__init__.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, "combine_moe_plan_gb300", f), os.path.join(dst, "combine_moe_plan_gb300", f))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("__init__.py", "conftest.py", "exact.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


def _pins_pass(dst: str) -> bool:
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=dst, capture_output=True, text=True, timeout=600)
    return r.returncode == 0


def _case(base: str, i: int, old, new) -> tuple:
    dst = os.path.join(base, f"case{i}")
    _copy_tree(dst)
    if old is not None:
        src = os.path.join(dst, "oracle", "moe_oracle.c")
        text = open(src).read()
        assert text.count(old) == 1, f"mutation site not found exactly once: {old!r}"
        open(src, "w").write(text.replace(old, new))
    return i, _pins_pass(dst)


def test_every_planted_mistake_fails_a_pin(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    jobs = [(-1, None, None)] + [(i, old, new) for i, (_, old, new) in enumerate(MUTATIONS)]
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = dict(ex.map(lambda j: _case(str(tmp_path), *j), jobs))
    assert results[-1], "the unchanged oracle copy must pass its pins"
    survivors = [MUTATIONS[i][0] for i in range(len(MUTATIONS)) if results[i]]
    assert not survivors, f"mistakes no pin caught: {survivors}"

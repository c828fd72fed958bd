"""The pins of the oracle's expert-parallel split must catch plausible
mistakes.  Each case plants one mistake in a temporary copy of
oracle/moe_oracle_ep.c (never in the committed file), builds that copy, and
runs tests/test_oracle_ep_pins.py against it: the run must fail.  The
unchanged copy must pass, so a failure is the mistake's.  Host only."""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in moe_oracle_ep.c, replacement)
MUTATIONS = [
    ("ownership rounded up",
     "return (int32_t)(((int64_t)p * R) / P);",
     "return (int32_t)(((int64_t)p * R + P - 1) / P);"),
    ("layout lists sources in descending order",
     "for (int32_t s = 0; s < R; ++s) {\n            chunk_row",
     "for (int32_t s = R - 1; s >= 0; --s) {\n            chunk_row"),
    ("gather appends sources in descending order",
     "for (int32_t s = 0; s < R; ++s) {\n            const int64_t n = counts[(size_t)s * P + p];\n"
     "            const int64_t from",
     "for (int32_t s = R - 1; s >= 0; --s) {\n            const int64_t n = counts[(size_t)s * P + p];\n"
     "            const int64_t from"),
    ("receive row counts the source itself",
     "for (int32_t r = 0; r < s; ++r) row += counts[(size_t)r * P + p];",
     "for (int32_t r = 0; r <= s && r < R; ++r) row += counts[(size_t)r * P + p];"),
    ("window start taken from rank 0's scan",
     "for (int32_t q = 0; q < p; ++q) row += counts[(size_t)s * P + q];",
     "for (int32_t q = 0; q < p; ++q) row += counts[q];"),
    ("return reads the source's own buffer",
     "memcpy(dst + to * row_bytes, recv[d] + from * row_bytes, (size_t)(n * row_bytes));",
     "memcpy(dst + to * row_bytes, recv[s] + from * row_bytes, (size_t)(n * row_bytes));"),
    ("units sorted shortest first",
     "    if (a->cost > b->cost) return -1;\n    if (a->cost < b->cost) return 1;",
     "    if (a->cost < b->cost) return -1;\n    if (a->cost > b->cost) return 1;"),
    ("equal costs in reverse enumeration order",
     "return (a->index < b->index) ? -1 : (a->index > b->index);",
     "return (a->index > b->index) ? -1 : (a->index < b->index);"),
    ("equal loads go to the higher core",
     "if (best < 0 || load[c] < load[best]) best = c;",
     "if (best < 0 || load[c] <= load[best]) best = c;"),
    ("fan-out cap ignored",
     "if (stripe_peer[(size_t)len[c] * R + q] >= cap[t]) continue;",
     "(void)0;"),
    ("fan-out cap off by one",
     "if (stripe_peer[(size_t)len[c] * R + q] >= cap[t]) continue;",
     "if (stripe_peer[(size_t)len[c] * R + q] > cap[t]) continue;"),
    ("pieces one row short",
     "const int64_t rows = (n - done < S) ? (n - done) : S;",
     "const int64_t rows = (n - done < S) ? (n - done) : (S > 1 ? S - 1 : S);"),
    ("tiers swapped for the unit size",
     "unit_rows[s == d ? 0 : 1]);",
     "unit_rows[s == d ? 1 : 0]);"),
    ("cost without the per-unit latency",
     "key[i].cost = alpha_ns[t] * 1000 + (bytes * 1000) / beta_gbs[t];",
     "key[i].cost = (bytes * 1000) / beta_gbs[t];"),
    ("combine units with source and destination swapped",
     "rc = orc_ep_split(u, &nu, max_units, d, orc_ep_recv_row(counts, R, P, s, p),\n"
     "                              orc_ep_pool_row(counts, P, s, p),",
     "rc = orc_ep_split(u, &nu, max_units, d, orc_ep_pool_row(counts, P, s, p),\n"
     "                              orc_ep_recv_row(counts, R, P, s, p),"),
]


def _copy_tree(dst: str) -> None:
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ("__init__.py", "moe_oracle.c", "moe_oracle_ep.c"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, "oracle", f))
    os.makedirs(os.path.join(dst, "combine_moe_plan_gb300"))
    for f in ("__init__.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, "combine_moe_plan_gb300", f), os.path.join(dst, "combine_moe_plan_gb300", f))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("__init__.py", "conftest.py", "test_oracle_ep_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


def _pins_pass(dst: str) -> bool:
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_ep_pins.py", "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=dst, capture_output=True, text=True, timeout=600)
    return r.returncode == 0


def _case(base: str, i: int, old, new) -> tuple:
    dst = os.path.join(base, f"case{i}")
    _copy_tree(dst)
    if old is not None:
        src = os.path.join(dst, "oracle", "moe_oracle_ep.c")
        text = open(src).read()
        assert text.count(old) == 1, f"mutation site not found exactly once: {old!r}"
        open(src, "w").write(text.replace(old, new))
    return i, _pins_pass(dst)


def test_every_planted_mistake_fails_an_ep_pin(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    jobs = [(-1, None, None)] + [(i, old, new) for i, (_, old, new) in enumerate(MUTATIONS)]
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = dict(ex.map(lambda j: _case(str(tmp_path), *j), jobs))
    assert results[-1], "the unchanged oracle copy must pass its pins"
    survivors = [MUTATIONS[i][0] for i in range(len(MUTATIONS)) if results[i]]
    assert not survivors, f"mistakes no pin caught: {survivors}"

"""In-kernel stage probes (trace build): one pass per workload in a child
process (the library build is chosen per process), stamps checked for
consistency."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload,graph", [("t96_h7168_e256_k8", False), ("t4096_h7168_e256p288_k8", False),
                                            ("t96_h7168_e256_k8", True)])
def test_trace_stages(workload, graph):
    r = subprocess.run([sys.executable, "-m", "combine_moe_plan_gb300.trace", "--workload", workload] +
                       (["--graph"] if graph else []), capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    rows = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    names = [x["kernel"] for x in rows]
    if workload.startswith("t96"):
        assert names == ["plan_one_launch", "dispatch", "combine"]
    else:
        assert names == ["route_tile", "column_scan", "assign", "dispatch", "combine"]
    for x in rows:
        assert x["span_ns"] > 0 and x["sms"] >= 1
        for st in x["stages"].values():
            assert st["median_ns"] >= 0 and st["ctas"] >= 1
        # every CTA of the launch was stamped at its first and last stage
        first = next(iter(x["stages"].values()))
        assert first["ctas"] == x["ctas"] or x["kernel"] in ("plan_one_launch",)
        assert 0 <= x["start_at_ns"] < x["end_at_ns"]
    # one pass: each kernel ends after the one before it (PDL lets a kernel
    # start early, but it finishes only after its predecessor's results)
    ends = [x["end_at_ns"] for x in rows]
    assert ends == sorted(ends)

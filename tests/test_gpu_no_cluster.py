"""The plan without thread-block clusters.  A device or partition that refuses
the cluster launch plans batches of up to 128 tokens with the one-launch
ticket kernel instead, and larger ones with the three launches;
MOE_PLAN_NO_CLUSTER=1 forces that.  The cluster plan's parity tests (every
switch point from 1 to 513 tokens, graph capture, chained layers, the small
workloads) are re-run in a child process with the variable set, so the same
oracle comparisons cover the fallback; so is the test file of
moe_plan_dispatch."""
import os
import subprocess
import sys

import pytest

from tests.gpu_util import ensure_built

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cluster_parity_tests_pass_on_the_ticket_plan():
    ensure_built()
    env = dict(os.environ, MOE_PLAN_NO_CLUSTER="1")
    sel = "path_switch_at_cluster_sizes or captures_in_a_cuda_graph or layers_chained or small_parity"
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "-k", sel, "-x", "-q",
                        "-m", "gpu", "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


def test_plan_dispatch_tests_pass_without_clusters():
    """moe_plan_dispatch's whole test file, with the variable set."""
    ensure_built()
    env = dict(os.environ, MOE_PLAN_NO_CLUSTER="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_plan_dispatch.py", "-x", "-q", "-m", "gpu",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


def _plan_ctas(env) -> int:
    """CTAs that ran the 96-token plan, from the trace build's stamps: the
    cluster plan uses 6 (tiles of 16 tokens), the ticket plan 3 (tiles of 32)."""
    import json
    r = subprocess.run([sys.executable, "-m", "combine_moe_plan_gb300.trace", "--workload", "t96_h7168_e256_k8"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    rows = [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]
    return next(x["ctas"] for x in rows if x["kernel"] == "plan_one_launch")


def test_the_switch_selects_the_ticket_plan():
    ensure_built()
    assert _plan_ctas(dict(os.environ)) == 6
    assert _plan_ctas(dict(os.environ, MOE_PLAN_NO_CLUSTER="1")) == 3

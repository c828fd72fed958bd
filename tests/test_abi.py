"""Host-only tests of the C ABI (no GPU needed): the library loads, exports
every function include/moe.h declares, sizes the pool as documented and
rejects bad arguments before launching anything."""
import ctypes

import numpy as np
import pytest

from combine_moe_plan_gb300 import build as moe_build
from combine_moe_plan_gb300 import moe


@pytest.fixture(scope="module")
def L():
    moe_build.build()
    return moe.lib()


def _desc(T=64, H=256, E=8, P=8, k=2, group=128, n_sets=2):
    return moe.Desc(T, H, E, P, k, group, n_sets)


def _api_names():
    from combine_moe_plan_gb300 import ep
    return moe.header_functions() + moe.header_functions(ep.HEADER)


def test_exports_every_header_symbol(L):
    names = _api_names()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n
    # and nothing but the API is exported under the moe_ prefix
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T moe_" in ln}
    assert exported == set(names)


def test_trace_build_exports_probe_api(L):
    """libmoe_trace.so exports moe.h plus moe_trace.h; libmoe.so exports no
    probe entry point."""
    import os
    import subprocess
    from combine_moe_plan_gb300 import build as b
    trace_names = moe.header_functions(os.path.join(os.path.dirname(moe.HEADER), "moe_trace.h"))
    assert trace_names == ["moe_trace_reset", "moe_trace_read"]
    out = subprocess.run(["nm", "-D", "--defined-only", b.TRACE_LIB], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T moe_" in ln}
    assert exported == set(_api_names()) | set(trace_names)


def test_status_strings(L):
    for rc in moe.STATUS:
        assert L.moe_status_str(rc)
    assert L.moe_status_str(0) == b"ok"


def _bytes(L, d):
    n = ctypes.c_size_t()
    rc = L.moe_pool_bytes(ctypes.byref(d), ctypes.byref(n))
    return rc, n.value


def test_pool_bytes_layout(L):
    rc, n = _bytes(L, _desc(T=4096, H=7168, E=256, P=288, k=8))
    assert rc == 0
    R, H = 4096 * 8, 7168
    per_set_payload = R * H + R * 56 * 4 + R * H * 2  # codes + scales + ex_out
    assert n >= 2 * per_set_payload
    assert n < 2 * per_set_payload * 1.25  # metadata + staging are small next to the rows
    rc1, n1 = _bytes(L, _desc(T=4096, H=7168, E=256, P=288, k=8, n_sets=1))
    assert rc1 == 0 and abs(2 * n1 - n) < 4096


@pytest.mark.parametrize("field,val,rc", [
    ("T_max", 0, -2), ("H", 200, -2), ("H", 64, -2), ("E", 0, -2), ("P", 4, -2), ("k", 0, -2),
    ("k", 9, -2), ("group", 64, -2), ("n_sets", 0, -2), ("n_sets", 5, -2), ("E", 2000, -2)])
def test_pool_bytes_rejects(L, field, val, rc):
    d = _desc()
    setattr(d, field, val)
    assert _bytes(L, d)[0] == rc


def _fake_pool(L, **kw):
    d = _desc(**kw)
    rc, n = _bytes(L, d)
    assert rc == 0
    h = ctypes.c_void_p()
    fake_ws = ctypes.c_void_p(1 << 40)  # 256-aligned address that is never dereferenced on the host
    assert L.moe_pool_init(ctypes.byref(d), fake_ws, n, ctypes.byref(h)) == 0
    return h, n


def test_pool_init_checks(L):
    d = _desc()
    rc, n = _bytes(L, d)
    h = ctypes.c_void_p()
    assert L.moe_pool_init(ctypes.byref(d), ctypes.c_void_p(1 << 40), n - 1, ctypes.byref(h)) == -5
    assert L.moe_pool_init(ctypes.byref(d), ctypes.c_void_p((1 << 40) + 16), n, ctypes.byref(h)) == -3
    assert L.moe_pool_init(ctypes.byref(d), None, n, ctypes.byref(h)) == -1
    h, _ = _fake_pool(L)
    v = moe.View()
    assert L.moe_pool_view(h, 0, ctypes.byref(v)) == 0
    assert v.rows == 64 * 2 and v.scale_stride == 4
    addrs = [getattr(v, f) for f, _ in moe.View._fields_[:12]]
    assert all(a % 256 == 0 for a in addrs)
    assert L.moe_pool_view(h, 2, ctypes.byref(v)) == -4
    assert L.moe_pool_destroy(h) == 0


def test_calls_rejected_before_launch(L):
    h, _ = _fake_pool(L)
    good = ctypes.c_void_p(1 << 41)
    odd = ctypes.c_void_p((1 << 41) + 4)
    # T out of range, bad set, NULL and misaligned pointers
    assert L.moe_plan(h, good, -1, None, None, 0, None) == -2
    assert L.moe_plan(h, good, 65, None, None, 0, None) == -2
    assert L.moe_plan(h, good, 8, None, None, 2, None) == -4
    assert L.moe_plan(h, None, 8, None, None, 0, None) == -1
    assert L.moe_plan(h, odd, 8, None, None, 0, None) == -3
    assert L.moe_plan(h, good, 8, good, None, 0, None) == -1  # half a replica map
    assert L.moe_plan(None, good, 8, None, None, 0, None) == -1
    # dispatch / combine before any plan on this set
    assert L.moe_dispatch(h, good, 8, 0, None) == -9
    assert L.moe_identity_experts(h, 8, 0, None) == -9
    assert L.moe_combine(h, None, good, 8, 0, None) == -9
    assert L.moe_combine(h, None, None, 8, 0, None) == -1
    assert L.moe_dispatch(h, odd, 8, 0, None) == -3
    L.moe_pool_destroy(h)


def test_dispatch_after_plan_checks_like_dispatch(L):
    h, _ = _fake_pool(L)
    good = ctypes.c_void_p(1 << 41)
    odd = ctypes.c_void_p((1 << 41) + 4)
    for fn in (L.moe_dispatch, L.moe_dispatch_after_plan):
        assert fn(h, good, 8, 0, None) == -9    # no plan on this set
        assert fn(h, odd, 8, 0, None) == -3
        assert fn(h, None, 8, 0, None) == -1
        assert fn(h, good, 8, 2, None) == -4
        assert fn(h, good, 65, 0, None) == -2
        assert fn(None, good, 8, 0, None) == -1
    L.moe_pool_destroy(h)


def test_plan_dispatch_checks_like_plan_and_dispatch(L):
    """moe_plan_dispatch rejects what moe_plan or moe_dispatch would reject,
    before anything is launched (no GPU here: a call past the checks could
    only fail with MOE_ERR_CUDA)."""
    h, _ = _fake_pool(L)
    good = ctypes.c_void_p(1 << 41)
    odd = ctypes.c_void_p((1 << 41) + 4)
    f = L.moe_plan_dispatch
    assert f(h, good, -1, None, None, good, 0, None) == -2
    assert f(h, good, 65, None, None, good, 0, None) == -2
    assert f(h, good, 8, None, None, good, 2, None) == -4
    assert f(h, None, 8, None, None, good, 0, None) == -1   # no logits
    assert f(h, good, 8, None, None, None, 0, None) == -1   # no x
    assert f(h, odd, 8, None, None, good, 0, None) == -3
    assert f(h, good, 8, None, None, odd, 0, None) == -3
    assert f(h, good, 8, good, None, good, 0, None) == -1   # half a replica map
    assert f(None, good, 8, None, None, good, 0, None) == -1
    L.moe_pool_destroy(h)


@pytest.mark.parametrize("T", [0, 1, 96])
def test_plan_static_checks_do_not_depend_on_T(L, T):
    """Every argument check of moe_plan_static runs before the empty-batch
    branch: with no GPU here, a call that got past the checks could only
    fail with MOE_ERR_CUDA (-6), so these codes come from the checks."""
    p = ctypes.c_void_p(1 << 41)
    odd = ctypes.c_void_p((1 << 41) + 4)
    f = L.moe_plan_static

    def call(logits=p, E=8, P=8, k=2, ro=None, ri=None, counts=p, offsets=p):
        return f(logits, T, E, P, k, ro, ri, p, p, p, counts, offsets, p, p, p, p, None)

    assert call(P=6) == -2                      # P < E
    assert call(E=0) == -2
    assert call(k=9) == -2                      # k > E
    assert call(P=10) == -8                     # P > E needs a replica map
    assert call(ro=p) == -1                     # half a replica map
    assert call(P=10, ro=odd, ri=p) == -3       # misaligned map
    assert call(counts=None) == -1
    assert call(offsets=odd) == -3
    assert f(p, -1, 8, 8, 2, None, None, p, p, p, p, p, p, p, p, p, None) == -2
    if T == 0:
        assert call(logits=None) == -6          # an empty batch needs no logits: it reaches the memset
    else:
        assert call(logits=None) == -1


def test_replica_map_needed_when_P_exceeds_E(L):
    h, _ = _fake_pool(L, E=8, P=10)
    assert L.moe_plan(h, ctypes.c_void_p(1 << 41), 8, None, None, 0, None) == -8
    L.moe_pool_destroy(h)


def test_step_host_rejects_before_enqueueing(L):
    """moe_step_host checks everything moe_plan would reject before its first
    copy: with no GPU here, a check that ran after a copy could only report
    MOE_ERR_CUDA (-6), so these codes show that nothing was enqueued."""
    h, _ = _fake_pool(L, E=8, P=10)
    host = ctypes.c_void_p(1 << 41)
    odd = ctypes.c_void_p((1 << 41) + 4)
    step = L.moe_step_host
    assert step(None, host, host, None, host, 8, None, None, 0, None) == -1
    assert step(h, host, host, None, host, 8, None, None, 2, None) == -4     # bad set
    assert step(h, host, host, None, host, 65, None, None, 0, None) == -2    # T > T_max
    assert step(h, None, host, None, host, 8, None, None, 0, None) == -1     # no logits
    assert step(h, host, host, None, None, 8, None, None, 0, None) == -1     # no y
    assert step(h, host, host, None, host, 8, host, None, 0, None) == -1     # half a replica map
    assert step(h, host, host, None, host, 8, None, None, 0, None) == -8     # P > E needs a map
    assert step(h, host, host, None, host, 8, odd, host, 0, None) == -3      # misaligned map
    L.moe_pool_destroy(h)


def test_replica_check(L):
    def rc(off, ids, E, P):
        return moe.replica_check(np.array(off), np.array(ids), E, P)
    assert rc([0, 2, 3], [0, 2, 1], 2, 3) == 0
    assert rc([0, 1, 2], [1, 0], 2, 2) == 0
    assert rc([0, 2, 3], [0, 0, 1], 2, 3) == -8    # physical id used twice
    assert rc([0, 0, 3], [0, 1, 2], 2, 3) == -8    # expert without a replica
    assert rc([0, 2, 2], [0, 1], 2, 2) == -8
    assert rc([1, 2, 3], [0, 1, 2], 2, 3) == -8
    assert rc([0, 2, 3], [0, 3, 1], 2, 3) == -8    # id out of range
    from combine_moe_plan_gb300 import workloads as wl
    w = wl.WORKLOADS["t4096_h7168_e256p288_k8"]
    off, ids = wl.make_replica_map(w)
    assert rc(off, ids, w.E, w.P) == 0


def test_binding_has_no_oracle_or_cpu_path():
    """The product package never imports, loads or runs the oracle."""
    import pathlib
    import re
    pkg = pathlib.Path(moe.__file__).parent
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle)|moe_oracle|libmoe_oracle", re.M)
    for f in list(pkg.glob("*.py")) + list(pkg.glob("csrc/*")):
        assert not pat.search(f.read_text()), f


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe.h"

int main(void) {
    moe_desc d;
    size_t bytes = 0;
    int32_t off[3] = {0, 2, 3}, ids[3] = {2, 0, 1}, bad_ids[3] = {0, 0, 1};
    d.T_max = 4096; d.H = 7168; d.E = 256; d.P = 288; d.k = 8; d.group = 128; d.n_sets = 2;
    if (moe_pool_bytes(&d, &bytes) != MOE_OK || bytes == 0) return 1;
    if (strcmp(moe_status_str(MOE_OK), "ok") != 0) return 2;
    if (moe_replica_check(off, ids, 2, 3) != MOE_OK) return 3;
    if (moe_replica_check(off, bad_ids, 2, 3) != MOE_ERR_REPLICA) return 4;
    d.k = 0;
    if (moe_pool_bytes(&d, &bytes) != MOE_ERR_SIZE) return 5;
    printf("%zu\n", bytes);
    return 0;
}
"""


def test_header_is_c_and_links_from_c(L, tmp_path):
    """include/moe.h compiles as ISO C11 with every warning an error, and a C
    program links against libmoe.so and calls its host-only entry points:
    the same pool size as the binding reports, status strings, replica-map
    checks, argument rejection."""
    import os
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(moe.LIB_PATH)
    inc = os.path.dirname(moe.HEADER)
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", f"-I{inc}", str(src), "-o", str(exe),
                    f"-L{libdir}", "-l:libmoe.so", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, (out.returncode, out.stderr)
    rc, n = _bytes(L, _desc(T=4096, H=7168, E=256, P=288, k=8))
    assert rc == 0 and int(out.stdout.strip()) == n

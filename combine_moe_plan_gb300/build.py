"""Build libmoe.so (and its trace twin libmoe_trace.so) in-tree with nvcc
for sm_103a.

Each .cu under csrc/ compiles in parallel to an object under _build/<variant>/,
then one nvcc link per variant makes combine_moe_plan_gb300/_lib/libmoe.so
and libmoe_trace.so (the same sources with -DMOE_TRACE: in-kernel stage
probes).  CUDA runtime linked statically; only the extern "C" API exported.
ptxas register/spill reports are kept in _build/ptxas.log.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libmoe.so")
TRACE_LIB = os.path.join(LIBDIR, "libmoe_trace.so")
VARIANTS = {"libmoe.so": [], "libmoe_trace.so": ["-DMOE_TRACE"]}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
          "-Xptxas", "-v", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale() -> bool:
    libs = [os.path.join(LIBDIR, v) for v in VARIANTS]
    if not all(os.path.exists(p) for p in libs):
        return True
    t = min(os.path.getmtime(p) for p in libs)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)

    def compile_one(job):
        variant, src = job
        odir = os.path.join(BUILD, variant.replace(".so", ""))
        os.makedirs(odir, exist_ok=True)
        obj = os.path.join(odir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *CFLAGS, *VARIANTS[variant], "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return variant, obj, r.stderr

    jobs = [(v, src) for v in VARIANTS for src in _sources()]
    with cf.ThreadPoolExecutor(max_workers=min(12, len(jobs))) as ex:
        results = list(ex.map(compile_one, jobs))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for (variant, obj, log) in results:
            if variant == "libmoe.so":
                f.write(f"== {os.path.basename(obj)}\n{log}\n")
    for variant in VARIANTS:
        out = os.path.join(LIBDIR, variant)
        tmp = out + f".tmp{os.getpid()}"
        objs = [o for (v, o, _) in results if v == variant]
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    if verbose:
        print(open(os.path.join(BUILD, "ptxas.log")).read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

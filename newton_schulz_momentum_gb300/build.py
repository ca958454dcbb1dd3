"""Build libdmuon.so in-tree for sm_103a with nvcc (no cmake, no torch extension machinery), and beside it
libdmuon_checked.so: the same sources with the device-side range checks compiled in
(-DDMUON_DEVICE_CHECKS=1), the debugging build.

Each translation unit compiles in its own nvcc process, in parallel; the objects are linked with the
static CUDA runtime, so the libraries need no libcudart at run time and load on machines without a GPU
(the driver is looked up only on first use).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdmuon.so")
CHECKED_LIB = os.path.join(PKG, "libdmuon_checked.so")
SOURCES = ("api.cu", "gemm_tc.cu", "ns_small.cu", "rowwise.cu", "adamw.cu", "noalloc.cu", "partition.cpp")
ARCH = ("-gencode", "arch=compute_103a,code=sm_103a")
# (library, object directory, extra flags)
VARIANTS = ((LIB, BUILD_DIR, ()), (CHECKED_LIB, os.path.join(BUILD_DIR, "checked"), ("-DDMUON_DEVICE_CHECKS=1",)))


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _run(cmd):
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if proc.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + proc.stdout)
    return proc.stdout


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dmuon.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False):
    """Compile every CUDA translation unit for sm_103a and link libdmuon.so and libdmuon_checked.so (each only
    when a source changed since it was linked). Returns the path of libdmuon.so."""
    todo = [v for v in VARIANTS if force or _stale(v[0])]
    if not todo:
        return LIB
    nvcc = _nvcc()
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]

    def compile_one(job):
        src, objdir, extra = job
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        out = _run(common + list(extra) + ["-c", os.path.join(CSRC, src), "-o", obj])
        if verbose and out.strip():
            print(out, file=sys.stderr)
        return obj

    jobs = []
    for _, objdir, extra in todo:
        os.makedirs(objdir, exist_ok=True)
        jobs += [(src, objdir, extra) for src in SOURCES]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for k, (lib, _, _) in enumerate(todo):
        tmp = lib + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs[k * len(SOURCES):(k + 1) * len(SOURCES)], "-Xcompiler", "-fPIC"])
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

"""Builds libdsa.so in-tree with nvcc for sm_103a (no torch extension machinery).

The CUDA translation units compile in parallel; the shared library links
the CUDA runtime statically and exports only the C ABI of include/dsa.h.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdsa.so")
SOURCES = ["dsa_api.cu", "dsa_tc.cu", "dsa_simt.cu", "dsa_noalloc.cu", "dsa_topk.cu", "dsa_selftest.cu",
           "dsa_tp.cu", "dsa_gemm.cu"]
HEADERS = ["dsa_internal.h", "dsa_ptx.cuh", "dsa_merge.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsa.so")


def _stale(extra_flags) -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps += [os.path.join(ROOT, "include", "dsa.h"), __file__]
    if any(os.path.getmtime(d) > t for d in deps):
        return True
    stamp = os.path.join(BUILD, "flags")
    want = " ".join(extra_flags)
    return not os.path.exists(stamp) or open(stamp).read() != want


def build(force: bool = False, extra_flags=(), verbose: bool = False) -> str:
    """Compile libdsa.so; returns its path.  Raises on a compiler error."""
    extra_flags = list(extra_flags)
    if not force and not _stale(extra_flags):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB)
    with open(os.path.join(BUILD, "flags"), "w") as f:
        f.write(" ".join(extra_flags))
    return LIB

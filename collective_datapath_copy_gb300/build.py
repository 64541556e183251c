"""Build libcoll.so in-tree: nvcc for sm_103a (CUDA sources), g++ for the host compiler.

    python -m collective_datapath_copy_gb300.build      # or build() from Python

The translation units compile in parallel; the result is
collective_datapath_copy_gb300/libcoll.so (git-ignored). cudart is linked statically,
so the library needs only the NVIDIA driver at run time.
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcoll.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-ftz=false", "-prec-div=true", "-fmad=false", f"-I{INCLUDE}", f"-I{CSRC}"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", f"-I{INCLUDE}", f"-I{CSRC}"]

CU_SOURCES = ["engine.cu", "bulk.cu", "api.cu", "noalloc.cu"]
CXX_SOURCES = ["plan.cpp"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def _stale(objs, extra=()) -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "coll.h")]
    deps += [os.path.abspath(__file__)] + list(extra)
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libcoll.so if any source is newer; returns its path."""
    if not force and not _stale([]):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append([nvcc, *ARCH, *NVCC_FLAGS, "-Xptxas", "-v", "-c", os.path.join(CSRC, src),
                     "-o", obj])
    for src in CXX_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append([os.environ.get("CXX", "g++"), *CXX_FLAGS, "-c", os.path.join(CSRC, src),
                     "-o", obj])
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(_run, jobs))
    if verbose:
        for o in outs:
            sys.stdout.write(o)
    objs = [os.path.join(BUILD, s + ".o") for s in CU_SOURCES + CXX_SOURCES]
    tmp = LIB + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-Xlinker", "--no-undefined", "-o", tmp,
          *objs])
    os.replace(tmp, LIB)
    if verbose:
        sys.stdout.write("built " + LIB + "\n")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)

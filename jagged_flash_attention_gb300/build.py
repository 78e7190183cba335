"""Builds libjfa.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into a
shared library next to this file.  Static cudart; the driver's tensor-map
encoder is looked up at run time, so the library loads without a GPU.
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
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libjfa.so")
SOURCES = ["aux.cu", "fwd.cu", "fwd_bs.cu", "bwd_kv.cu", "bwd_q.cu", "bwd_qb.cu", "bwd_bs.cu",
           "sparse.cu", "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    hdrs.append(os.path.join(INCLUDE, "jfa.h"))
    return hdrs


def _stale(target, inputs) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(i) > t for i in inputs)


def variant_path(name: str) -> str:
    """Path of a library variant built by build(variant=name)."""
    return os.path.join(PKG, f"libjfa_{name}.so")


def build(verbose: bool = False, force: bool = False, variant: str | None = None,
          defines: tuple = ()) -> str:
    """Builds libjfa.so, or with `variant` a copy of the library compiled with
    the extra preprocessor `defines` (e.g. a short wait limit for the timeout
    test) into libjfa_<variant>.so, with its own object directory."""
    build_dir = BUILD_DIR if variant is None else os.path.join(BUILD_DIR, variant)
    lib_path = LIB_PATH if variant is None else variant_path(variant)
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    hdrs = _deps()
    objs = []
    jobs = []
    extra = [f"-D{d}" for d in defines]
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append([nvcc, *ARCH, *FLAGS, *extra, "-c", s, "-o", o])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib_path, objs):
        run([nvcc, *ARCH, "-shared", "-o", lib_path, *objs])
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv))

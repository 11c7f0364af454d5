"""Compile the clipping library (libgclip.so) in-tree for sm_103a.

Two translation units (the CUDA kernels with the C ABI, and the host planner)
are compiled in parallel and linked into one shared library with the CUDA
runtime linked statically.  The library lands in ``_build/`` beside this
file; ``ptxas.log`` there records registers, spills and shared memory.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libgclip.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "-Xptxas", "-v", f"-I{INCLUDE}"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgclip")


def _sources():
    return [os.path.join(CSRC, f) for f in ("gclip.cu", "plan.cpp")]


def _inputs():
    deps = _sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                         if f.endswith((".hpp", ".cuh", ".h"))]
    deps.append(os.path.join(INCLUDE, "gclip.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Build libgclip.so if any input is newer; return its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    tag = f"{os.getpid()}"

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.basename(src) + f".{tag}.o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=2) as ex:
        results = list(ex.map(compile_one, _sources()))
    objs = [o for o, _ in results]
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        for _, log in results:
            f.write(log)
    tmp = LIB + f".{tag}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(open(os.path.join(OUT_DIR, "ptxas.log")).read())
    return LIB


if __name__ == "__main__":  # pragma: no cover
    print(build(force=True, verbose=True))

"""Build libgpipe.so in-tree for sm_103a (nvcc, one -gencode, parallel TUs)."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgpipe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

CUDA_SOURCES = ["gemm_tc.cu", "gemm_persistent.cu", "gemm_simt.cu", "attention.cu", "elementwise.cu", "launch.cu"]
CXX_SOURCES = ["planner.cpp", "gpipe.cpp", "checkpoint.cpp"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgpipe")


def _sources():
    return [os.path.join(CSRC, s) for s in CUDA_SOURCES + CXX_SOURCES]


def _headers():
    inc = os.path.join(os.path.dirname(PKG), "include")
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    return hs


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _sources() + _headers())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA/C++ translation unit and link libgpipe.so; returns its path."""
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    common = ["-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-lineinfo"]
    jobs = []
    for s in CUDA_SOURCES:
        obj = os.path.join(OUT_DIR, s + ".o")
        jobs.append([nvcc, *common, *ARCH, "-c", os.path.join(CSRC, s), "-o", obj])
    for s in CXX_SOURCES:
        obj = os.path.join(OUT_DIR, s + ".o")
        jobs.append([nvcc, *common, "-x", "c++", "-c", os.path.join(CSRC, s), "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("compile failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)

    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        list(ex.map(run, jobs))
    objs = [os.path.join(OUT_DIR, s + ".o") for s in CUDA_SOURCES + CXX_SOURCES]
    tmp = LIB + ".tmp"
    run([nvcc, "-shared", *ARCH, "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

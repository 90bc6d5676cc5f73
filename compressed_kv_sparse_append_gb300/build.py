"""Builds libckv.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each CUDA translation unit is compiled in parallel with nvcc, then linked
into ``compressed_kv_sparse_append_gb300/libckv.so`` (CUDA runtime linked
statically).  Object files go to ``_build/`` at the repository root.
"""

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libckv.so")
SOURCES = ["append.cu", "indexer.cu", "indexer_umma.cu", "attention.cu", "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I", os.path.join(ROOT, "include")]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src, nvcc):
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = r.stdout + r.stderr
    with open(os.path.join(BUILD, os.path.splitext(src)[0] + ".log"), "w") as f:
        f.write(log)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s" % (src, log[-4000:]))
    return obj


def build(verbose: bool = False) -> str:
    """Compiles and links libckv.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, nvcc), SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s" % (r.stdout + r.stderr)[-4000:])
    os.replace(tmp, LIB)
    if verbose:
        for s in SOURCES:
            with open(os.path.join(BUILD, os.path.splitext(s)[0] + ".log")) as f:
                sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

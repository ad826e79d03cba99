"""Build ``libvqenc.so`` (the CUDA encoder and its C ABI) for sm_103a, in tree.

Usage: ``python -m product_vq_kv_gb300.build`` (or ``build()`` from Python).
The library lands in ``product_vq_kv_gb300/_lib/`` together with the
``ptxas -v`` report of its kernels (registers, spills, shared memory).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libvqenc.so")
PTXAS_LOG = os.path.join(LIB_DIR, "ptxas.txt")
SOURCES = [os.path.join(CSRC, "vq_encode.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "vq_kernels.cuh"), os.path.join(CSRC, "vq_filter.cuh"), os.path.join(CSRC, "vq_tc.cuh"), os.path.join(CSRC, "vq_decode.cuh"),
                     os.path.join(ROOT, "include", "vq_encode.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# --fmad=false: no plain multiply-add in these sources may be contracted into an
# FMA (the encode formula rounds the square and the sum separately); the hot
# loops use explicit round-to-nearest intrinsics as well.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xptxas", "-v",
              "-Xcompiler", "-fPIC", "-shared"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libvqenc.so")


def is_fresh() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    built = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= built for p in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library unless it is newer than all of its sources."""
    if not force and is_fresh():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=LIB_DIR)
    os.close(fd)
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-o", tmp, *SOURCES]
    try:
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
        with open(PTXAS_LOG, "w") as f:
            f.write(" ".join(cmd) + "\n" + res.stderr)
        if verbose:
            sys.stderr.write(res.stderr)
        os.replace(tmp, LIB_PATH)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

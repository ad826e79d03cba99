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
# The bounds-checked build (-DVQ_CHECKED, csrc/vq_check.cuh): the same entry
# points, every kernel index checked, launches waited for; for tests only.
CHECKED_LIB_PATH = os.path.join(LIB_DIR, "libvqenc_checked.so")
PTXAS_LOG = os.path.join(LIB_DIR, "ptxas.txt")
SOURCES = [os.path.join(CSRC, name) for name in ("vq_encode.cu", "vq_attn.cu", "vq_scalar.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, name) for name in (
    "vq_kernels.cuh", "vq_filter.cuh", "vq_tc.cuh", "vq_decode.cuh", "vq_attn.cuh", "vq_host.h", "vq_scalar.cuh", "vq_status.cuh", "vq_check.cuh", "vq_umma.cuh")] + [
    os.path.join(ROOT, "include", "vq_encode.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# --fmad=false: no plain multiply-add in these sources may be contracted into an
# FMA (the encode formula rounds the square and the sum separately); the hot
# loops use explicit round-to-nearest intrinsics as well.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xptxas", "-v",
              "-Xcompiler", "-fPIC"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libvqenc.so")


def is_fresh(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    built = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= built for p in DEPENDS)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile the library unless it is newer than all of its sources.

    The translation units compile in parallel, then link into one shared
    library.  ``checked`` builds the bounds-checked variant instead
    (``libvqenc_checked.so``)."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    if not force and is_fresh(lib_path):
        return lib_path
    os.makedirs(LIB_DIR, exist_ok=True)
    with tempfile.TemporaryDirectory(dir=LIB_DIR) as tmpdir:
        jobs = []
        for src in SOURCES:
            obj = os.path.join(tmpdir, os.path.basename(src) + ".o")
            cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *(["-DVQ_CHECKED"] if checked else []), "-I",
                   os.path.join(ROOT, "include"), "-c", "-o", obj, src]
            jobs.append((cmd, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                    stderr=subprocess.PIPE, text=True)))
        log = []
        for cmd, _, proc in jobs:
            out, err = proc.communicate()
            if proc.returncode != 0:
                raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + out + err)
            log.append(" ".join(cmd) + "\n" + err)
        tmp = os.path.join(tmpdir, "lib.so")
        link = [nvcc(), *ARCH, "-shared", "-o", tmp, *(obj for _, obj, _ in jobs)]
        res = subprocess.run(link, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc link failed:\n" + " ".join(link) + "\n" + res.stdout + res.stderr)
        if not checked:
            with open(PTXAS_LOG, "w") as f:
                f.write("\n".join(log))
        if verbose:
            sys.stderr.write("\n".join(log))
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))

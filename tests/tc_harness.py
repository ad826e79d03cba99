"""Build and load the test-only CUDA harness of the tensor-core encode.

``tests/harness/*.cu`` include the library's ``vq_tc.cuh`` and compile, in
their own shared library ``tests/harness/_build/libtc_harness.so`` (never part
of ``libvqenc.so``):

* ``probe_tf32_chain`` -- a chain of ``tcgen05.mma.kind::tf32`` through the
  library's descriptors and tensor-memory loads, for the accumulation-error
  test;
* ``stats_encode`` -- the library's encode kernel, library configuration, with
  per-row screening statistics;
* ``polls_encode`` -- the same kernel with a tiny per-pass poll limit, for the
  wait give-up path;
* ``check_probe`` -- the bounds-check primitives of the checked build,
  evaluated on described spans;
* ``probe_link_read`` -- a plain read of a device or pinned host buffer, for
  the host-link read rate beside the host-buffer encode.

Same compiler flags as the library (``product_vq_kv_gb300.build``); the units
compile in parallel and are rebuilt only when a source or a library header
is newer than the harness.
"""
from __future__ import annotations

import ctypes
import glob
import os
import subprocess
import tempfile
import threading

from product_vq_kv_gb300 import build as lib_build

HERE = os.path.dirname(os.path.abspath(__file__))
SRC_DIR = os.path.join(HERE, "harness")
BUILD_DIR = os.path.join(SRC_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libtc_harness.so")
SOURCES = sorted(glob.glob(os.path.join(SRC_DIR, "*.cu")))

_lock = threading.Lock()
_lib = None


def _fresh() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    built = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= built for p in SOURCES + lib_build.DEPENDS)


def build() -> str:
    if _fresh():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    with tempfile.TemporaryDirectory(dir=BUILD_DIR) as tmp:
        jobs = []
        for src in SOURCES:
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            cmd = [lib_build.nvcc(), *lib_build.ARCH, *lib_build.NVCC_FLAGS, "-I",
                   lib_build.CSRC, "-I", os.path.join(lib_build.ROOT, "include"), "-c", "-o",
                   obj, src]
            jobs.append((cmd, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                    stderr=subprocess.PIPE, text=True)))
        for cmd, _, proc in jobs:
            out, err = proc.communicate()
            if proc.returncode != 0:
                raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + out + err)
        tmp_lib = os.path.join(tmp, "lib.so")
        link = [lib_build.nvcc(), *lib_build.ARCH, "-shared", "-o", tmp_lib,
                *(obj for _, obj, _ in jobs)]
        res = subprocess.run(link, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
        os.replace(tmp_lib, LIB_PATH)
    return LIB_PATH


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            lib.probe_tf32_chain.restype = i32
            lib.probe_tf32_chain.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
            lib.stats_encode.restype = i32
            lib.stats_encode.argtypes = [i32, i32, i32, vp, vp, i64, i64, i32, i32, vp, vp, i32,
                                         vp]
            lib.stats_read.restype = i32
            lib.stats_read.argtypes = [ctypes.POINTER(ctypes.c_ulonglong), i32]
            lib.stats_status.restype = i32
            lib.stats_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
            lib.polls_encode.restype = i32
            lib.polls_encode.argtypes = [i32, i32, i32, vp, vp, i64, i64, i32, i32, vp, vp]
            lib.polls_status.restype = i32
            lib.polls_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
            lib.check_probe.restype = i32
            lib.check_probe.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32, vp]
            lib.check_status.restype = i32
            lib.check_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
            lib.probe_link_read.restype = i32
            lib.probe_link_read.argtypes = [vp, i64, vp, i32, vp]
            _lib = lib
        return _lib


def read_stats(clear: bool = True) -> list:
    """Rows per screening outcome since the last clear: [1 group, 1 group
    tight, 2 groups, 2 groups tight, queued]."""
    buf = (ctypes.c_ulonglong * 8)()
    assert load().stats_read(buf, 1 if clear else 0) == 0
    return [int(v) for v in buf[:5]]


def status(unit: str, clear: bool = True) -> int:
    bits = ctypes.c_uint32(0)
    fn = {"stats": load().stats_status, "polls": load().polls_status,
          "check": load().check_status}[unit]
    assert fn(ctypes.byref(bits), 1 if clear else 0) == 0
    return int(bits.value)

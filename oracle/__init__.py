"""CPU oracle for the product-VQ encode step (``quantize_vq``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library under ``product_vq_kv_gb300/`` and never imports it.

The arithmetic lives in ``vq_oracle.c`` (plain C, fp32, no FMA contraction);
this module compiles it with the host ``gcc`` on first use and wraps it with
``ctypes``.  See that file's header for what is computed and which passage of
"I Wrote a Metal Kernel to Stop My Mac From OOMing" each step follows.

Parity pins: every exported function is pinned in ``tests/test_oracle.py``
against float64 brute force, closed forms, invariants and golden fixtures.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libvqoracle.so")

# Flags: no FMA contraction and no fast-math, so every fp32 multiply and add
# rounds separately, as the encode formula requires.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
          "-fno-fast-math", "-fno-unsafe-math-optimizations"]

DTYPE_F16, DTYPE_BF16, DTYPE_F32 = 0, 1, 2

_lock = threading.Lock()
_default = None


def compile_source(src_path: str, out_path: str) -> str:
    """Compile one C source of the oracle into a shared library."""
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out_path))
    os.close(fd)
    try:
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, src_path, "-lm"], check=True,
                       capture_output=True, text=True)
        os.replace(tmp, out_path)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``vq_oracle.c`` into ``oracle/_build/libvqoracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
    if fresh and not force:
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _dtype_code(arr: np.ndarray, bf16: bool) -> int:
    if arr.dtype == np.float16:
        return DTYPE_F16
    if arr.dtype == np.float32:
        return DTYPE_F32
    if arr.dtype == np.uint16 and bf16:
        return DTYPE_BF16
    raise TypeError(f"unsupported dtype {arr.dtype} (bf16={bf16})")


class OracleLib:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.vqo_f16_to_f32.restype = ctypes.c_float
        lib.vqo_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.vqo_bf16_to_f32.restype = ctypes.c_float
        lib.vqo_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.vqo_distance.restype = ctypes.c_float
        lib.vqo_distance.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int32, ctypes.c_int32]
        lib.vqo_encode_grouped.restype = ctypes.c_int32
        lib.vqo_encode_grouped.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
            ctypes.c_int32]
        lib.vqo_encode_grouped_smooth.restype = ctypes.c_int32
        lib.vqo_encode_grouped_smooth.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
            ctypes.c_int32]
        lib.vqo_scalar_quantize.restype = ctypes.c_int32
        lib.vqo_scalar_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                            ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
        lib.vqo_hadamard_rotate.restype = ctypes.c_int32
        lib.vqo_hadamard_rotate.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                            ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                            ctypes.c_void_p]
        lib.vqo_hadamard_quantize.restype = ctypes.c_int32
        lib.vqo_hadamard_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                              ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                              ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
        self.path = path
        self._lib = lib

    def f16_to_f32(self, bits: int) -> float:
        return float(self._lib.vqo_f16_to_f32(bits))

    def bf16_to_f32(self, bits: int) -> float:
        return float(self._lib.vqo_bf16_to_f32(bits))

    def distance(self, x: np.ndarray, c: np.ndarray, bf16: bool = False) -> np.float32:
        """fp32 squared distance of one sub-vector to one centroid."""
        x = np.ascontiguousarray(x)
        c = np.ascontiguousarray(c)
        if x.shape != c.shape or x.ndim != 1 or x.dtype != c.dtype:
            raise ValueError("x and c must be 1-D arrays of the same shape and dtype")
        code = _dtype_code(x, bf16)
        return np.float32(self._lib.vqo_distance(x.ctypes.data, c.ctypes.data,
                                                 x.shape[0], code))

    def encode(self, x: np.ndarray, codebook: np.ndarray, *, bf16: bool = False,
               n_threads: int = 1) -> np.ndarray:
        """Nearest-centroid indices (uint32), by the fp32 encode formula.

        ``x`` is ``[N, sub_dim]`` with ``codebook`` ``[n_centroids, sub_dim]``,
        or grouped: ``x`` ``[G, M, sub_dim]`` with ``codebook`` ``[G,
        n_centroids, sub_dim]``.  fp16 and fp32 arrays are taken as they are;
        bf16 data is passed as its raw ``uint16`` bits with ``bf16=True``.
        Returns ``[N]`` or ``[G, M]`` uint32.
        """
        x = np.ascontiguousarray(x)
        codebook = np.ascontiguousarray(codebook)
        if x.dtype != codebook.dtype:
            raise TypeError("x and codebook must share a dtype")
        code = _dtype_code(x, bf16)
        if x.ndim == 2 and codebook.ndim == 2:
            groups, per_group, sub_dim = 1, x.shape[0], x.shape[1]
            out_shape = (x.shape[0],)
        elif x.ndim == 3 and codebook.ndim == 3 and x.shape[0] == codebook.shape[0]:
            groups, per_group, sub_dim = x.shape
            out_shape = (groups, per_group)
        else:
            raise ValueError(f"bad shapes x{x.shape} codebook{codebook.shape}")
        if codebook.shape[-1] != sub_dim:
            raise ValueError("sub_dim mismatch between x and codebook")
        n_centroids = codebook.shape[-2]
        out = np.zeros(out_shape, dtype=np.uint32)
        rc = self._lib.vqo_encode_grouped(x.ctypes.data, codebook.ctypes.data, groups,
                                          per_group, n_centroids, sub_dim, code,
                                          out.ctypes.data, int(n_threads))
        if rc != 0:
            raise RuntimeError(f"oracle encode failed with status {rc}")
        return out

    def scalar_quantize(self, x: np.ndarray, centroids: np.ndarray, *,
                        bf16: bool = False) -> np.ndarray:
        """Scalar (sub_dim = 1) quantize: index of the nearest fp32 centroid of
        every element of ``x`` (any shape), as uint32 of the same shape."""
        x = np.ascontiguousarray(x)
        c = np.ascontiguousarray(centroids, dtype=np.float32).reshape(-1)
        out = np.zeros(x.shape, dtype=np.uint32)
        rc = self._lib.vqo_scalar_quantize(x.ctypes.data, _dtype_code(x, bf16), x.size,
                                           c.ctypes.data, c.size, out.ctypes.data)
        if rc != 0:
            raise RuntimeError(f"oracle scalar quantize failed with status {rc}")
        return out

    def hadamard_rotate(self, x: np.ndarray, diag: np.ndarray, *, scale: float | None = None,
                        bf16: bool = False) -> np.ndarray:
        """Randomised Hadamard rotation of the rows of ``x`` ``[..., D]``:
        float32 ``[..., D]``.  ``scale`` defaults to fp32(1/sqrt(D))."""
        x = np.ascontiguousarray(x)
        dim = x.shape[-1]
        d = np.ascontiguousarray(diag, dtype=np.float32).reshape(-1)
        scale = hadamard_scale(dim) if scale is None else np.float32(scale)
        y = np.zeros(x.shape, dtype=np.float32)
        rc = self._lib.vqo_hadamard_rotate(x.ctypes.data, _dtype_code(x, bf16), d.ctypes.data,
                                           x.size // dim, dim, float(scale), y.ctypes.data)
        if rc != 0:
            raise RuntimeError(f"oracle hadamard rotate failed with status {rc}")
        return y

    def hadamard_quantize(self, x: np.ndarray, diag: np.ndarray, centroids: np.ndarray, *,
                          scale: float | None = None, bf16: bool = False) -> np.ndarray:
        """Rotation then scalar quantize of every rotated element: uint32 of
        ``x``'s shape."""
        x = np.ascontiguousarray(x)
        dim = x.shape[-1]
        d = np.ascontiguousarray(diag, dtype=np.float32).reshape(-1)
        c = np.ascontiguousarray(centroids, dtype=np.float32).reshape(-1)
        scale = hadamard_scale(dim) if scale is None else np.float32(scale)
        out = np.zeros(x.shape, dtype=np.uint32)
        rc = self._lib.vqo_hadamard_quantize(x.ctypes.data, _dtype_code(x, bf16), d.ctypes.data,
                                             x.size // dim, dim, float(scale), c.ctypes.data,
                                             c.size, out.ctypes.data)
        if rc != 0:
            raise RuntimeError(f"oracle hadamard quantize failed with status {rc}")
        return out

    def encode_smooth(self, x: np.ndarray, smooth: np.ndarray, codebooks: np.ndarray,
                      head_dim: int, *, bf16: bool = False, n_threads: int = 1) -> np.ndarray:
        """Encode with per-channel smoothing: each element divided (fp32,
        round to nearest) by its channel's factor before the encode formula.

        ``x`` ``[G, M, sub_dim]``, ``smooth`` ``[G, head_dim]`` float32,
        ``codebooks`` ``[G, n_centroids, sub_dim]``; row ``m`` of a group holds
        channels ``(m % (head_dim // sub_dim)) * sub_dim + i``.  Returns
        ``[G, M]`` uint32.
        """
        x = np.ascontiguousarray(x)
        codebooks = np.ascontiguousarray(codebooks)
        smooth = np.ascontiguousarray(smooth, dtype=np.float32)
        if x.dtype != codebooks.dtype or x.ndim != 3 or codebooks.ndim != 3:
            raise ValueError("x [G, M, sub_dim] and codebooks [G, n_c, sub_dim] of one dtype")
        groups, per_group, sub_dim = x.shape
        if smooth.shape != (groups, head_dim) or codebooks.shape[0] != groups:
            raise ValueError(f"bad shapes smooth{smooth.shape} for x{x.shape}")
        out = np.zeros((groups, per_group), dtype=np.uint32)
        rc = self._lib.vqo_encode_grouped_smooth(
            x.ctypes.data, smooth.ctypes.data, codebooks.ctypes.data, groups, per_group,
            codebooks.shape[1], sub_dim, int(head_dim), _dtype_code(x, bf16), out.ctypes.data,
            int(n_threads))
        if rc != 0:
            raise RuntimeError(f"oracle smoothed encode failed with status {rc}")
        return out


def dequantize(idx: np.ndarray, codebooks: np.ndarray) -> np.ndarray:
    """Decode ("dequantize_vq"): each index becomes a copy of its codebook row.

    Source: "I Wrote a Metal Kernel to Stop My Mac From OOMing", section
    "Mistake 1: I Wrote the Dequant Kernel First" -- the operation takes
    codebook indices and reconstructs the vectors, a gather (``mx.take``).
    ``idx`` is ``[G, M]`` (any integer dtype), ``codebooks`` ``[G, n_c, sub]``
    (any dtype, including raw bf16 bits as uint16); returns ``[G, M, sub]`` in
    the codebooks' dtype.  Reading where the page is silent: an index outside
    ``[0, n_c)`` decodes to a row of zeros.
    """
    idx = np.asarray(idx)
    codebooks = np.asarray(codebooks)
    g, m = idx.shape
    n_c, sub = codebooks.shape[1], codebooks.shape[2]
    out = np.zeros((g, m, sub), dtype=codebooks.dtype)
    for k in range(g):
        valid = idx[k].astype(np.int64) < n_c
        out[k, valid] = codebooks[k, idx[k][valid].astype(np.int64)]
    return out


def attention_decode(q, k_codes, k_codebooks, v_codes, v_codebooks, window: int = 0,
                     scale: float = 0.0) -> np.ndarray:
    """Decode attention over product-VQ codes, in float64.

    Source: "I Wrote a Metal Kernel to Stop My Mac From OOMing", section
    "What's Next: Phase 2" -- scores from a per-query table of q against the
    codebook, looked up by the key codes, then softmax and the weighted sum of
    the values.  Written here as what that computes: keys and values rebuilt
    from their codes by :func:`dequantize` (so a code outside ``[0, n_c)`` is
    a zero row), then ``softmax(scale * K^ q) @ V^`` for every (batch, query
    head), query head ``h`` reading KV head ``h // (Hq / Hkv)``, over the last
    ``window`` tokens (0: all).  Readings where the pages are silent: no
    tokens gives zeros; ``scale <= 0`` means ``1 / sqrt(D)``.  ``q`` is
    ``[B, Hq, D]`` (float16 or float32; bf16 decoded by the caller); codes
    ``[B, Hkv, T, D / sub]``; codebooks ``[Hkv, n_c, sub]``.
    """
    q = np.asarray(q, dtype=np.float64)
    k_codes = np.asarray(k_codes)
    v_codes = np.asarray(v_codes)
    b, hq, d = q.shape
    _, hkv, t, ns = k_codes.shape
    qpk = hq // hkv
    scale = scale if scale > 0 else 1.0 / np.sqrt(d)
    first = t - window if 0 < window < t else 0
    n = t - first
    out = np.zeros((b, hq, d))
    if n == 0:
        return out
    for bi in range(b):
        for h in range(hkv):
            keys = dequantize(k_codes[bi, h, first:].reshape(1, n * ns),
                              np.asarray(k_codebooks)[h:h + 1]).astype(np.float64).reshape(n, d)
            vals = dequantize(v_codes[bi, h, first:].reshape(1, n * ns),
                              np.asarray(v_codebooks)[h:h + 1]).astype(np.float64).reshape(n, d)
            for g in range(qpk):
                logits = scale * (keys @ q[bi, h * qpk + g])
                p = np.exp(logits - logits.max())
                out[bi, h * qpk + g] = (p / p.sum()) @ vals
    return out


def default() -> OracleLib:
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def f16_to_f32(bits: int) -> float:
    return default().f16_to_f32(bits)


def bf16_to_f32(bits: int) -> float:
    return default().bf16_to_f32(bits)


def distance(x, c, bf16: bool = False):
    return default().distance(x, c, bf16=bf16)


def hadamard_scale(dim: int) -> np.float32:
    """fp32 value of 1/sqrt(dim), correctly rounded (dim a power of two: the
    double value 2^(-k/2) rounds to fp32 without double-rounding trouble)."""
    return np.float32(1.0 / np.sqrt(np.float64(dim)))


def scalar_quantize(x, centroids, *, bf16: bool = False):
    return default().scalar_quantize(x, centroids, bf16=bf16)


def hadamard_rotate(x, diag, *, scale=None, bf16: bool = False):
    return default().hadamard_rotate(x, diag, scale=scale, bf16=bf16)


def hadamard_quantize(x, diag, centroids, *, scale=None, bf16: bool = False):
    return default().hadamard_quantize(x, diag, centroids, scale=scale, bf16=bf16)


def encode_smooth(x, smooth, codebooks, head_dim, *, bf16: bool = False, n_threads: int = 1):
    return default().encode_smooth(x, smooth, codebooks, head_dim, bf16=bf16,
                                   n_threads=n_threads)


def encode(x, codebook, *, bf16: bool = False, n_threads: int = 1):
    return default().encode(x, codebook, bf16=bf16, n_threads=n_threads)

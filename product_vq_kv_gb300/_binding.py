"""ctypes binding of ``libvqenc.so``: argument marshalling only.

Every function here has the name of the C entry point it calls (declared in
``include/vq_encode.h``) and does nothing but check and convert its arguments,
allocate the output tensor when asked to, and pass the current CUDA stream.
All computation happens in the library's CUDA kernels; there is no other code
path.  If the library has not been built the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

VQ_OK, VQ_ERR_INVALID_ARG, VQ_ERR_UNSUPPORTED, VQ_ERR_CUDA, VQ_ERR_INTERNAL = range(5)
VQ_F16, VQ_BF16, VQ_F32 = 0, 1, 2

_TORCH_DTYPES = {torch.float16: VQ_F16, torch.bfloat16: VQ_BF16, torch.float32: VQ_F32}

_lock = threading.Lock()
_lib = None


class VQError(RuntimeError):
    """A non-OK status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {vq_status_string(status)}")


class VqSlice(ctypes.Structure):
    """``vq_slice``: rows [row, row + n_rows) of groups [group, group + n_groups)."""
    _fields_ = [("group", ctypes.c_int64), ("n_groups", ctypes.c_int64),
                ("row", ctypes.c_int64), ("n_rows", ctypes.c_int64)]


def _configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the argument and result types of every entry point on ``lib``
    (the library, or its bounds-checked build, which has the same ABI)."""
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.vq_encode.restype = i32
    lib.vq_encode.argtypes = [vp, vp, i64, i32, i32, i32, vp, vp]
    lib.vq_encode_grouped.restype = i32
    lib.vq_encode_grouped.argtypes = [vp, vp, i64, i64, i32, i32, i32, vp, vp]
    lib.vq_encode_grouped_host.restype = i32
    lib.vq_encode_grouped_host.argtypes = [vp, vp, i64, i64, i32, i32, i32, vp, vp, vp,
                                           vp, vp]
    lib.vq_encode_grouped_u8.restype = i32
    lib.vq_encode_grouped_u8.argtypes = [vp, vp, i64, i64, i32, i32, i32, vp, vp]
    lib.vq_dequantize_grouped.restype = i32
    lib.vq_dequantize_grouped.argtypes = [vp, i32, vp, i64, i64, i32, i32, i32, vp, vp]
    lib.vq_attention_decode.restype = i32
    lib.vq_attention_decode.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i64, i32, i32, i32,
                                        i64, ctypes.c_float, i32, vp, vp, ctypes.c_size_t, vp]
    lib.vq_attention_decode_static.restype = i32
    lib.vq_attention_decode_static.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i64, i32,
                                               i32, i32, i64, ctypes.c_float, i32, vp, vp]
    lib.vq_encode_grouped_smooth.restype = i32
    lib.vq_encode_grouped_smooth.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, i32, vp,
                                             i32, vp]
    lib.vq_scalar_quantize_workspace_bytes.restype = ctypes.c_size_t
    lib.vq_scalar_quantize_workspace_bytes.argtypes = [i32]
    lib.vq_scalar_quantize.restype = i32
    lib.vq_scalar_quantize.argtypes = [vp, i32, i64, vp, i32, vp, vp, ctypes.c_size_t, vp]
    lib.vq_scalar_dequantize.restype = i32
    lib.vq_scalar_dequantize.argtypes = [vp, i64, vp, i32, i32, vp, vp]
    lib.vq_hadamard_rotate.restype = i32
    lib.vq_hadamard_rotate.argtypes = [vp, i32, vp, i64, i32, vp, vp]
    lib.vq_hadamard_quantize.restype = i32
    lib.vq_hadamard_quantize.argtypes = [vp, i32, vp, i64, i32, vp, i32, vp, vp]
    lib.vq_attention_workspace_bytes.restype = ctypes.c_size_t
    lib.vq_attention_workspace_bytes.argtypes = [i64, i32, i32, i64, i32, i32, i32, i64]
    lib.vq_status_string.restype = ctypes.c_char_p
    lib.vq_status_string.argtypes = [i32]
    lib.vq_describe_launch.restype = i32
    lib.vq_describe_launch.argtypes = [i64, i64, i32, i32, i32, vp, ctypes.c_char_p, i32]
    lib.vq_abi_version.restype = i32
    lib.vq_abi_version.argtypes = []
    lib.vq_kernel_status.restype = i32
    lib.vq_kernel_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
    lib.vq_partition.restype = i32
    lib.vq_partition.argtypes = [i64, i64, i32, i32, ctypes.POINTER(VqSlice),
                                 ctypes.POINTER(ctypes.c_int32)]
    return lib


def load_library() -> ctypes.CDLL:
    """Load ``libvqenc.so`` (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing; build it with `python -m product_vq_kv_gb300.build` "
                "(there is no fallback implementation)")
        _lib = _configure(ctypes.CDLL(LIB_PATH))
        return _lib


def vq_status_string(status: int) -> str:
    return load_library().vq_status_string(int(status)).decode()


def vq_abi_version() -> int:
    return int(load_library().vq_abi_version())


# Bits of the device status word (vq_kernel_status).
VQ_KSTATUS_WAIT_GAVE_UP = 0x1
VQ_KSTATUS_OUT_OF_BOUNDS = 0x2


def vq_kernel_status(clear: bool = True, device=None) -> int:
    """The status bits the library's kernels set on ``device`` (default: the
    current device) since the last clear, after waiting for that device to
    finish; 0 means every kernel finished normally.  Clears them if
    ``clear``."""
    bits = ctypes.c_uint32(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        st = load_library().vq_kernel_status(ctypes.byref(bits), 1 if clear else 0)
    _check(st, "vq_kernel_status")
    return int(bits.value)


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _TORCH_DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}; expected float16, bfloat16 or float32")


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _check(status: int, where: str) -> None:
    if status != VQ_OK:
        raise VQError(status, where)


def _device_tensor(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def vq_encode(x: torch.Tensor, codebook: torch.Tensor, out: torch.Tensor | None = None,
              stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Indices of the nearest centroid for each row of ``x``.

    ``x`` ``[N, sub_dim]`` and ``codebook`` ``[n_centroids, sub_dim]`` are
    contiguous CUDA tensors of one dtype (float16, bfloat16 or float32).
    Returns (or fills ``out``) a ``[N]`` uint32 tensor.  Asynchronous on
    ``stream`` (default: the current stream).
    """
    _device_tensor(x, "x")
    _device_tensor(codebook, "codebook")
    if x.dim() != 2 or codebook.dim() != 2 or x.shape[1] != codebook.shape[1]:
        raise ValueError(f"expected x [N, sub_dim] and codebook [n_centroids, sub_dim], got "
                         f"{tuple(x.shape)} and {tuple(codebook.shape)}")
    if x.dtype != codebook.dtype:
        raise TypeError("x and codebook must share a dtype")
    if out is None:
        out = torch.empty(x.shape[0], dtype=torch.uint32, device=x.device)
    elif out.dtype != torch.uint32 or out.shape != (x.shape[0],) or not out.is_contiguous():
        raise ValueError("out must be a contiguous uint32 tensor of shape [N]")
    st = load_library().vq_encode(x.data_ptr(), codebook.data_ptr(), x.shape[0],
                                  codebook.shape[0], x.shape[1], _dtype_code(x),
                                  out.data_ptr(), _stream_handle(stream, x.device))
    _check(st, "vq_encode")
    return out


def vq_encode_grouped(x: torch.Tensor, codebooks: torch.Tensor,
                      out: torch.Tensor | None = None,
                      stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Grouped encode: ``x`` ``[G, M, sub_dim]`` against ``codebooks``
    ``[G, n_centroids, sub_dim]`` (row block g uses codebook g).  Returns (or
    fills ``out``) a ``[G, M]`` uint32 tensor.  Asynchronous on ``stream``."""
    _device_tensor(x, "x")
    _device_tensor(codebooks, "codebooks")
    if (x.dim() != 3 or codebooks.dim() != 3 or x.shape[0] != codebooks.shape[0]
            or x.shape[2] != codebooks.shape[2]):
        raise ValueError(f"expected x [G, M, sub_dim] and codebooks [G, n_centroids, sub_dim], "
                         f"got {tuple(x.shape)} and {tuple(codebooks.shape)}")
    if x.dtype != codebooks.dtype:
        raise TypeError("x and codebooks must share a dtype")
    g, m, sub = x.shape
    if out is None:
        out = torch.empty((g, m), dtype=torch.uint32, device=x.device)
    elif out.dtype != torch.uint32 or out.shape != (g, m) or not out.is_contiguous():
        raise ValueError("out must be a contiguous uint32 tensor of shape [G, M]")
    st = load_library().vq_encode_grouped(x.data_ptr(), codebooks.data_ptr(), g, m,
                                          codebooks.shape[1], sub, _dtype_code(x),
                                          out.data_ptr(), _stream_handle(stream, x.device))
    _check(st, "vq_encode_grouped")
    return out


def vq_encode_grouped_u8(x: torch.Tensor, codebooks: torch.Tensor,
                         out: torch.Tensor | None = None,
                         stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Grouped encode to 8-bit codes (at most 256 centroids): the indices of
    :func:`vq_encode_grouped` as a ``[G, M]`` uint8 tensor."""
    _device_tensor(x, "x")
    _device_tensor(codebooks, "codebooks")
    if (x.dim() != 3 or codebooks.dim() != 3 or x.shape[0] != codebooks.shape[0]
            or x.shape[2] != codebooks.shape[2]):
        raise ValueError(f"expected x [G, M, sub_dim] and codebooks [G, n_centroids, sub_dim], "
                         f"got {tuple(x.shape)} and {tuple(codebooks.shape)}")
    if x.dtype != codebooks.dtype:
        raise TypeError("x and codebooks must share a dtype")
    g, m, sub = x.shape
    if out is None:
        out = torch.empty((g, m), dtype=torch.uint8, device=x.device)
    elif out.dtype != torch.uint8 or out.shape != (g, m) or not out.is_contiguous():
        raise ValueError("out must be a contiguous uint8 tensor of shape [G, M]")
    st = load_library().vq_encode_grouped_u8(x.data_ptr(), codebooks.data_ptr(), g, m,
                                             codebooks.shape[1], sub, _dtype_code(x),
                                             out.data_ptr(), _stream_handle(stream, x.device))
    _check(st, "vq_encode_grouped_u8")
    return out


def vq_encode_grouped_smooth(x: torch.Tensor, smooth: torch.Tensor, codebooks: torch.Tensor,
                             head_dim: int, index_bytes: int = 1, out: torch.Tensor | None = None,
                             stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Grouped encode of smoothed keys: every element of ``x`` ``[G, M,
    sub_dim]`` divided by its channel's factor in ``smooth`` ``[G, head_dim]``
    (float32; row ``m`` holds channels ``(m % (head_dim // sub_dim)) * sub_dim
    + i``) before the encode.  Returns ``[G, M]`` uint8 codes
    (``index_bytes=1``) or uint32 indices (``index_bytes=4``)."""
    _device_tensor(x, "x")
    _device_tensor(smooth, "smooth")
    _device_tensor(codebooks, "codebooks")
    if (x.dim() != 3 or codebooks.dim() != 3 or x.shape[0] != codebooks.shape[0]
            or x.shape[2] != codebooks.shape[2]):
        raise ValueError(f"expected x [G, M, sub_dim] and codebooks [G, n_centroids, sub_dim], "
                         f"got {tuple(x.shape)} and {tuple(codebooks.shape)}")
    if x.dtype != codebooks.dtype:
        raise TypeError("x and codebooks must share a dtype")
    if smooth.dtype != torch.float32 or tuple(smooth.shape) != (x.shape[0], head_dim):
        raise ValueError("smooth must be float32 of shape [G, head_dim]")
    if index_bytes not in (1, 4):
        raise ValueError("index_bytes must be 1 or 4")
    g, m, sub = x.shape
    odt = torch.uint8 if index_bytes == 1 else torch.uint32
    if out is None:
        out = torch.empty((g, m), dtype=odt, device=x.device)
    elif out.dtype != odt or out.shape != (g, m) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {odt} tensor of shape [G, M]")
    st = load_library().vq_encode_grouped_smooth(
        x.data_ptr(), smooth.data_ptr(), codebooks.data_ptr(), g, m, codebooks.shape[1], sub,
        head_dim, _dtype_code(x), out.data_ptr(), index_bytes, _stream_handle(stream, x.device))
    _check(st, "vq_encode_grouped_smooth")
    return out


def _f32_vector(t: torch.Tensor, name: str) -> None:
    _device_tensor(t, name)
    if t.dtype != torch.float32 or t.dim() != 1:
        raise ValueError(f"{name} must be a 1-D float32 device tensor")


def vq_scalar_quantize(x: torch.Tensor, centroids: torch.Tensor, out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, use_table: bool = True,
                       stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Scalar (sub_dim = 1) quantize of every element of ``x`` against the
    float32 ``centroids``: uint8 indices of ``x``'s shape.  fp16 input with
    2, 4, 8 or 16 centroids takes the bucket table the kernel builds itself
    (the workspace goes unused); other fp16 / bf16 input takes the table pass
    when a 64 KiB ``workspace`` is given (allocated here when omitted and
    ``use_table``)."""
    _device_tensor(x, "x")
    _f32_vector(centroids, "centroids")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    elif out.dtype != torch.uint8 or out.shape != x.shape or not out.is_contiguous():
        raise ValueError("out must be a contiguous uint8 tensor of x's shape")
    code = _dtype_code(x)
    lib = load_library()
    need = int(lib.vq_scalar_quantize_workspace_bytes(code))
    if workspace is None and use_table and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.vq_scalar_quantize(x.data_ptr(), code, x.numel(), centroids.data_ptr(),
                                centroids.numel(), out.data_ptr(), ws_ptr, ws_bytes,
                                _stream_handle(stream, x.device))
    _check(st, "vq_scalar_quantize")
    return out


def vq_scalar_dequantize(idx: torch.Tensor, centroids: torch.Tensor,
                         dtype: torch.dtype = torch.float16, out: torch.Tensor | None = None,
                         stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """``centroids[idx]`` in ``dtype`` (round to nearest); out-of-range
    indices give 0."""
    _device_tensor(idx, "idx")
    _f32_vector(centroids, "centroids")
    if idx.dtype != torch.uint8:
        raise TypeError("idx must be uint8")
    if out is None:
        out = torch.empty(idx.shape, dtype=dtype, device=idx.device)
    st = load_library().vq_scalar_dequantize(idx.data_ptr(), idx.numel(), centroids.data_ptr(),
                                             centroids.numel(), _dtype_code(out), out.data_ptr(),
                                             _stream_handle(stream, idx.device))
    _check(st, "vq_scalar_dequantize")
    return out


def vq_hadamard_rotate(x: torch.Tensor, diag: torch.Tensor, out: torch.Tensor | None = None,
                       stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Randomised Hadamard rotation of the rows of ``x`` ``[..., D]``:
    float32 of the same shape."""
    _device_tensor(x, "x")
    _f32_vector(diag, "diag")
    dim = x.shape[-1]
    if diag.numel() != dim:
        raise ValueError("diag must have one entry per column")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    st = load_library().vq_hadamard_rotate(x.data_ptr(), _dtype_code(x), diag.data_ptr(),
                                           x.numel() // dim, dim, out.data_ptr(),
                                           _stream_handle(stream, x.device))
    _check(st, "vq_hadamard_rotate")
    return out


def vq_hadamard_quantize(x: torch.Tensor, diag: torch.Tensor, centroids: torch.Tensor,
                         out: torch.Tensor | None = None,
                         stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Rotation fused with the scalar quantize: uint8 indices of ``x``'s
    shape."""
    _device_tensor(x, "x")
    _f32_vector(diag, "diag")
    _f32_vector(centroids, "centroids")
    dim = x.shape[-1]
    if diag.numel() != dim:
        raise ValueError("diag must have one entry per column")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    st = load_library().vq_hadamard_quantize(x.data_ptr(), _dtype_code(x), diag.data_ptr(),
                                             x.numel() // dim, dim, centroids.data_ptr(),
                                             centroids.numel(), out.data_ptr(),
                                             _stream_handle(stream, x.device))
    _check(st, "vq_hadamard_quantize")
    return out


def vq_dequantize_grouped(idx: torch.Tensor, codebooks: torch.Tensor,
                          out: torch.Tensor | None = None,
                          stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Decode ``idx`` ``[G, M]`` (uint32 or uint8) against ``codebooks``
    ``[G, n_centroids, sub_dim]``: returns (or fills ``out``) the ``[G, M,
    sub_dim]`` tensor of codebook rows, in the codebooks' dtype; out-of-range
    indices give zero rows.  Asynchronous on ``stream``."""
    _device_tensor(idx, "idx")
    _device_tensor(codebooks, "codebooks")
    if idx.dtype not in (torch.uint32, torch.uint8):
        raise TypeError("idx must be uint32 or uint8")
    if idx.dim() != 2 or codebooks.dim() != 3 or idx.shape[0] != codebooks.shape[0]:
        raise ValueError(f"expected idx [G, M] and codebooks [G, n_centroids, sub_dim], got "
                         f"{tuple(idx.shape)} and {tuple(codebooks.shape)}")
    g, m = idx.shape
    n_c, sub = codebooks.shape[1], codebooks.shape[2]
    if out is None:
        out = torch.empty((g, m, sub), dtype=codebooks.dtype, device=idx.device)
    elif out.dtype != codebooks.dtype or out.shape != (g, m, sub) or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of shape [G, M, sub_dim] in the "
                         "codebooks' dtype")
    st = load_library().vq_dequantize_grouped(
        idx.data_ptr(), 4 if idx.dtype == torch.uint32 else 1, codebooks.data_ptr(), g, m, n_c,
        sub, _dtype_code(codebooks), out.data_ptr(), _stream_handle(stream, idx.device))
    _check(st, "vq_dequantize_grouped")
    return out


def vq_attention_workspace_bytes(batch: int, heads_q: int, heads_kv: int, tokens: int,
                                 head_dim: int, sub_dim: int, n_centroids: int,
                                 window: int = 0) -> int:
    return int(load_library().vq_attention_workspace_bytes(batch, heads_q, heads_kv, tokens,
                                                           head_dim, sub_dim, n_centroids,
                                                           window))


def _check_attention_args(q, k_codes, k_codebooks, v_codes, v_codebooks):
    """Validate the tensors of an attention call before any pointer is taken.

    Shapes and dtypes are checked first (so every mismatch is reported the
    same way whatever the device), then that every tensor is a contiguous CUDA
    tensor on q's device.  Returns ``(B, Hq, Hkv, T, D, sub_dim, n_c)``.
    """
    named = (("q", q), ("k_codes", k_codes), ("k_codebooks", k_codebooks),
             ("v_codes", v_codes), ("v_codebooks", v_codebooks))
    for name, t in named:
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
    if q.dim() != 3 or k_codes.dim() != 4 or k_codebooks.dim() != 3:
        raise ValueError(f"expected q [B, Hq, D], k_codes [B, Hkv, T, D/sub_dim] and "
                         f"k_codebooks [Hkv, n_c, sub_dim], got {tuple(q.shape)}, "
                         f"{tuple(k_codes.shape)} and {tuple(k_codebooks.shape)}")
    _dtype_code(q)
    if k_codes.dtype != torch.uint8 or v_codes.dtype != torch.uint8:
        raise TypeError("codes must be uint8")
    if k_codebooks.dtype != q.dtype or v_codebooks.dtype != q.dtype:
        raise TypeError("codebooks must share q's dtype")
    b, hq, d = q.shape
    _, hkv, tokens, ns = k_codes.shape
    n_c, sub = k_codebooks.shape[1], k_codebooks.shape[2]
    if (tuple(v_codes.shape) != tuple(k_codes.shape) or k_codes.shape[0] != b or ns * sub != d
            or tuple(k_codebooks.shape) != (hkv, n_c, sub)
            or tuple(v_codebooks.shape) != (hkv, n_c, sub)):
        raise ValueError("inconsistent shapes: q [B, Hq, D], codes [B, Hkv, T, D/sub_dim] (keys "
                         "and values alike), codebooks [Hkv, n_c, sub_dim] (keys and values alike)")
    for name, t in named:
        _device_tensor(t, name)
        if t.device != q.device:
            raise ValueError(f"{name} is on {t.device}, q on {q.device}")
    return b, hq, hkv, tokens, d, sub, n_c


def _check_attention_out(out, q):
    if out is None:
        return torch.empty_like(q)
    if (not isinstance(out, torch.Tensor) or out.dtype != q.dtype or out.shape != q.shape
            or out.device != q.device or not out.is_contiguous()):
        raise ValueError("out must be a contiguous tensor of q's shape, dtype and device")
    return out


def vq_attention_decode(q: torch.Tensor, k_codes: torch.Tensor, k_codebooks: torch.Tensor,
                        v_codes: torch.Tensor, v_codebooks: torch.Tensor, window: int = 0,
                        scale: float = 0.0, out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None,
                        stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Decode attention over 8-bit product-VQ codes.

    ``q`` ``[B, Hq, D]``; ``k_codes`` / ``v_codes`` ``[B, Hkv, T, D/sub_dim]``
    uint8; ``k_codebooks`` / ``v_codebooks`` ``[Hkv, n_c, sub_dim]`` in q's
    dtype.  Returns (or fills ``out``) ``[B, Hq, D]``.  ``workspace`` is a
    device byte tensor for the per-slice partials; if omitted one of
    :func:`vq_attention_workspace_bytes` bytes is allocated here (by torch).
    """
    b, hq, hkv, tokens, d, sub, n_c = _check_attention_args(q, k_codes, k_codebooks, v_codes,
                                                            v_codebooks)
    out = _check_attention_out(out, q)
    if workspace is None:
        nbytes = vq_attention_workspace_bytes(b, hq, hkv, tokens, d, sub, n_c, window)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    else:
        _device_tensor(workspace, "workspace")
        if workspace.device != q.device:
            raise ValueError(f"workspace is on {workspace.device}, q on {q.device}")
    with torch.cuda.device(q.device):
        st = load_library().vq_attention_decode(
            q.data_ptr(), k_codes.data_ptr(), k_codebooks.data_ptr(), v_codes.data_ptr(),
            v_codebooks.data_ptr(), b, hq, hkv, tokens, d, sub, n_c, window, scale,
            _dtype_code(q), out.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    _check(st, "vq_attention_decode")
    return out


# Bytes of the library's built-in scratch array (VQ_ATTN_STATIC_SCRATCH_BYTES).
ATTN_STATIC_SCRATCH_BYTES = 8 << 20


def vq_attention_decode_static(q: torch.Tensor, k_codes: torch.Tensor, k_codebooks: torch.Tensor,
                               v_codes: torch.Tensor, v_codebooks: torch.Tensor, window: int = 0,
                               scale: float = 0.0, out: torch.Tensor | None = None,
                               stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """:func:`vq_attention_decode` with its partials in the library's one
    built-in device array instead of a workspace, for callers that cannot
    allocate device memory per call (a decode loop whose HBM is planned up
    front, host code without a caching allocator).  The library allocates
    nothing; pass ``out`` to allocate nothing here either.  Calls that overlap
    on the GPU share that array and race: keep them in one stream order.  The
    call runs with q's device current, whose copy of the array it uses."""
    b, hq, hkv, tokens, d, sub, n_c = _check_attention_args(q, k_codes, k_codebooks, v_codes,
                                                            v_codebooks)
    if b * hq * (d + 2) * 4 > ATTN_STATIC_SCRATCH_BYTES:
        raise VQError(VQ_ERR_INVALID_ARG,
                      f"vq_attention_decode_static (one token slice needs {b * hq * (d + 2) * 4} "
                      f"bytes of scratch; the built-in array holds {ATTN_STATIC_SCRATCH_BYTES})")
    out = _check_attention_out(out, q)
    with torch.cuda.device(q.device):
        st = load_library().vq_attention_decode_static(
            q.data_ptr(), k_codes.data_ptr(), k_codebooks.data_ptr(), v_codes.data_ptr(),
            v_codebooks.data_ptr(), b, hq, hkv, tokens, d, sub, n_c, window, scale,
            _dtype_code(q), out.data_ptr(), _stream_handle(stream, q.device))
    _check(st, "vq_attention_decode_static")
    return out


def vq_encode_grouped_host(x_host: torch.Tensor, codebooks_host: torch.Tensor,
                           out_host: torch.Tensor, x_dev: torch.Tensor,
                           codebooks_dev: torch.Tensor, out_dev: torch.Tensor,
                           stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Grouped encode of HOST tensors through the caller's device buffers.

    ``x_host`` ``[G, M, sub_dim]``, ``codebooks_host`` ``[G, n_c, sub_dim]`` and
    ``out_host`` ``[G, M]`` uint32 live in host memory (pin them for
    asynchronous copies); ``x_dev``, ``codebooks_dev`` and ``out_dev`` are
    device buffers of at least the same sizes.  Returns ``out_host`` once it
    holds the indices.
    """
    for t, name in ((x_host, "x_host"), (codebooks_host, "codebooks_host"),
                    (out_host, "out_host")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
    for t, name in ((x_dev, "x_dev"), (codebooks_dev, "codebooks_dev"), (out_dev, "out_dev")):
        _device_tensor(t, name)
    if x_host.dim() != 3 or codebooks_host.dim() != 3:
        raise ValueError("expected x_host [G, M, sub_dim] and codebooks_host [G, n_c, sub_dim]")
    g, m, sub = x_host.shape
    n_c = codebooks_host.shape[1]
    if (x_dev.dtype != x_host.dtype or codebooks_dev.dtype != x_host.dtype
            or codebooks_host.dtype != x_host.dtype):
        raise TypeError("all x and codebook tensors must share a dtype")
    if out_host.dtype != torch.uint32 or out_dev.dtype != torch.uint32:
        raise TypeError("out_host and out_dev must be uint32")
    if (x_dev.numel() < x_host.numel() or codebooks_dev.numel() < codebooks_host.numel()
            or out_dev.numel() < g * m or out_host.numel() < g * m):
        raise ValueError("device or output buffers are too small")
    st = load_library().vq_encode_grouped_host(
        x_host.data_ptr(), codebooks_host.data_ptr(), g, m, n_c, sub, _dtype_code(x_host),
        out_host.data_ptr(), x_dev.data_ptr(), codebooks_dev.data_ptr(), out_dev.data_ptr(),
        _stream_handle(stream, x_dev.device))
    _check(st, "vq_encode_grouped_host")
    return out_host


def vq_partition(n_groups: int, n_per_group: int, world: int, rank: int) -> list:
    """The rows of a ``[n_groups, n_per_group]`` encode job that ``rank`` of
    ``world`` owns, as ``(group, n_groups, row, n_rows)`` slices in row order
    (see ``vq_partition`` in ``include/vq_encode.h``)."""
    buf = (VqSlice * 3)()
    count = ctypes.c_int32(0)
    st = load_library().vq_partition(n_groups, n_per_group, world, rank, buf, ctypes.byref(count))
    _check(st, "vq_partition")
    return [(s.group, s.n_groups, s.row, s.n_rows) for s in buf[:count.value]]


def vq_encode_partition(x: torch.Tensor, codebooks: torch.Tensor, world: int, rank: int,
                        out: torch.Tensor | None = None,
                        stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Rank ``rank``'s share of the grouped encode of ``x`` ``[G, M, sub_dim]``
    against the replicated ``codebooks`` ``[G, n_c, sub_dim]``: the indices of
    the rows :func:`vq_partition` gives it, as a 1-D uint32 tensor in row
    order (one grouped encode per slice; no collective).  Concatenated over
    the ranks in rank order they are ``vq_encode_grouped(x, codebooks)``
    flattened."""
    _device_tensor(x, "x")
    _device_tensor(codebooks, "codebooks")
    if (x.dim() != 3 or codebooks.dim() != 3 or x.shape[0] != codebooks.shape[0]
            or x.shape[2] != codebooks.shape[2]):
        raise ValueError(f"expected x [G, M, sub_dim] and codebooks [G, n_centroids, sub_dim], "
                         f"got {tuple(x.shape)} and {tuple(codebooks.shape)}")
    if x.dtype != codebooks.dtype:
        raise TypeError("x and codebooks must share a dtype")
    g, m, sub = x.shape
    slices = vq_partition(g, m, world, rank)
    n = sum(ng * nr for _, ng, _, nr in slices)
    if out is None:
        out = torch.empty(n, dtype=torch.uint32, device=x.device)
    elif out.dtype != torch.uint32 or out.shape != (n,) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous uint32 tensor of shape [{n}]")
    lib = load_library()
    handle = _stream_handle(stream, x.device)
    off = 0
    for g0, ng, r0, nr in slices:
        xs = x[g0:g0 + ng, r0:r0 + nr]  # contiguous: one group, or whole groups
        st = lib.vq_encode_grouped(xs.data_ptr(), codebooks[g0:g0 + ng].data_ptr(), ng, nr,
                                   codebooks.shape[1], sub, _dtype_code(x),
                                   out.data_ptr() + off * 4, handle)
        _check(st, "vq_encode_partition")
        off += ng * nr
    return out


def vq_describe_launch(n_groups: int, n_per_group: int, n_centroids: int, sub_dim: int,
                       dtype: torch.dtype, x_ptr: int = 0) -> str:
    """The kernel and launch shape the library would use (no launch)."""
    buf = ctypes.create_string_buffer(512)
    st = load_library().vq_describe_launch(n_groups, n_per_group, n_centroids, sub_dim,
                                           _TORCH_DTYPES[dtype], x_ptr, buf, len(buf))
    _check(st, "vq_describe_launch")
    return buf.value.decode()

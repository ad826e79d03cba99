"""The C-ABI library builds, loads and exports what its header declares, and
rejects bad arguments on the host (no GPU needed; nothing here launches)."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from product_vq_kv_gb300.build import build

    path = build()
    return ctypes.CDLL(path)


def declared_functions():
    names = set()
    for header in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(header).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(vq_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("vq_encode", "vq_encode_grouped", "vq_encode_grouped_host",
                     "vq_encode_grouped_u8", "vq_dequantize_grouped",
                     "vq_status_string", "vq_describe_launch", "vq_abi_version",
                     "vq_attention_decode", "vq_attention_workspace_bytes",
                     "vq_encode_grouped_smooth", "vq_scalar_quantize", "vq_scalar_dequantize",
                     "vq_hadamard_rotate", "vq_hadamard_quantize"):
        assert required in names


@pytest.mark.parametrize("name", declared_functions())
def test_library_exports_every_declared_function(lib, name):
    assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_checked_build_exports_every_declared_function():
    """The bounds-checked build (-DVQ_CHECKED) compiles and has the same ABI."""
    from product_vq_kv_gb300.build import build

    checked = ctypes.CDLL(build(checked=True))
    for name in declared_functions():
        assert hasattr(checked, name), name


def test_abi_version(lib):
    lib.vq_abi_version.restype = ctypes.c_int32
    assert lib.vq_abi_version() == 1


def test_status_strings(lib):
    lib.vq_status_string.restype = ctypes.c_char_p
    lib.vq_status_string.argtypes = [ctypes.c_int32]
    for code, word in enumerate(["VQ_OK", "VQ_ERR_INVALID_ARG", "VQ_ERR_UNSUPPORTED",
                                 "VQ_ERR_CUDA", "VQ_ERR_INTERNAL"]):
        assert lib.vq_status_string(code).decode().startswith(word)
    assert lib.vq_status_string(99).decode() == "unknown vq_status"


def _encode(lib):
    f = lib.vq_encode
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    return f


def _grouped(lib):
    f = lib.vq_encode_grouped
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                  ctypes.c_void_p]
    return f


# Fake, never-dereferenced device addresses: every case below fails (or
# succeeds with no work) during host-side validation, before any CUDA call.
P = 0x10000


@pytest.mark.parametrize("args,status", [
    ((None, P, 10, 256, 4, 0, P, None), 1),     # null x with work to do
    ((P, None, 10, 256, 4, 0, P, None), 1),     # null codebook
    ((P, P, 10, 256, 4, 0, None, None), 1),     # null output
    ((P, P, -1, 256, 4, 0, P, None), 1),        # negative N
    ((P, P, 10, 256, 4, 3, P, None), 1),        # unknown dtype
    ((P, P, 10, 256, 4, -1, P, None), 1),       # unknown dtype
    ((P + 1, P, 10, 256, 4, 0, P, None), 1),    # x not aligned to its element
    ((P, P, 10, 256, 4, 0, P + 2, None), 1),    # output not aligned to 4 bytes
    ((P, P, 10, 256, 0, 0, P, None), 2),        # sub_dim 0
    ((P, P, 10, 256, 33, 0, P, None), 2),       # sub_dim too large
    ((P, P, 10, 0, 4, 0, P, None), 2),          # no centroids
    ((P, P, 10, 4097, 4, 0, P, None), 2),       # too many centroids
    ((None, None, 0, 256, 4, 0, None, None), 0),  # N = 0: nothing to do
])
def test_encode_argument_errors(lib, args, status):
    assert _encode(lib)(*args) == status


@pytest.mark.parametrize("args,status", [
    ((P, P, -1, 10, 256, 8, 0, P, None), 1),    # negative group count
    ((P, P, 4, -10, 256, 8, 0, P, None), 1),    # negative group size
    ((P, P, 1 << 40, 1 << 40, 256, 8, 0, P, None), 1),  # row count overflows
    ((None, None, 4, 0, 256, 8, 0, None, None), 0),     # empty groups
    ((None, None, 0, 100, 256, 8, 0, None, None), 0),   # no groups
])
def test_grouped_argument_errors(lib, args, status):
    assert _grouped(lib)(*args) == status


def _attention(lib):
    f = lib.vq_attention_decode
    f.restype = ctypes.c_int32
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i64, i32, i32, i32, i64, ctypes.c_float, i32,
                  vp, vp, ctypes.c_size_t, vp]
    return f


# (batch, heads_q, heads_kv, tokens, head_dim, sub_dim, n_centroids, window, dtype,
#  pointer offset, workspace bytes) -> status; pointers are fake and never used
@pytest.mark.parametrize("shape,status", [
    ((2, 8, 3, 100, 128, 8, 256, 0, 0, 0, 1 << 20), 1),    # heads_q not a multiple of heads_kv
    ((2, 8, 2, 100, 128, 7, 256, 0, 0, 0, 1 << 20), 1),    # head_dim not a multiple of sub_dim
    ((2, 8, 2, 100, 128, 8, 257, 0, 0, 0, 1 << 20), 2),    # codes wider than 8 bits
    ((2, 8, 2, 100, 1024, 8, 256, 0, 0, 0, 1 << 20), 2),   # head_dim above 512
    ((2, 8, 2, 100, 128, 1, 256, 0, 0, 0, 1 << 20), 2),    # 128 sub-spaces
    ((2, 8, 2, 100, 96, 8, 256, 0, 0, 0, 1 << 20), 2),     # 12 sub-spaces
    ((2, 8, 2, 100, 128, 2, 256, 0, 0, 0, 1 << 20), 2),    # sub_dim not a multiple of 4
    ((2, 8, 2, -1, 128, 8, 256, 0, 0, 0, 1 << 20), 1),     # negative tokens
    ((2, 8, 2, 100, 128, 8, 256, -5, 0, 0, 1 << 20), 1),   # negative window
    ((2, 8, 2, 100, 128, 8, 256, 0, 7, 0, 1 << 20), 1),    # unknown dtype
    ((2, 8, 2, 100, 128, 8, 256, 0, 0, 1, 1 << 20), 1),    # misaligned pointers
    ((2, 8, 2, 100, 128, 8, 256, 0, 0, 0, 64), 1),         # workspace too small for one slice
    ((0, 8, 2, 100, 128, 8, 256, 0, 0, 0, 0), 0),          # no batch: nothing to do
])
def test_attention_argument_errors(lib, shape, status):
    b, hq, hkv, t, d, sub, nc, window, dtype, off, ws = shape
    p = P + off
    assert _attention(lib)(p, P, p, P, p, b, hq, hkv, t, d, sub, nc, window, 0.0, dtype, p, P, ws,
                           None) == status


def _smooth(lib):
    f = lib.vq_encode_grouped_smooth
    f.restype = ctypes.c_int32
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    f.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, i32, vp, i32, vp]
    return f


# (x, smooth, cb, G, M, n_c, sub, head_dim, dtype, out, index_bytes) -> status
@pytest.mark.parametrize("args,status", [
    ((P, P, P, 2, 64, 256, 4, 16, 0, P, 2), 1),      # index width neither 1 nor 4
    ((P, P, P, 2, 66, 256, 4, 16, 0, P, 4), 1),      # partial key vector in a group
    ((P, P, P, 2, 64, 256, 4, 18, 0, P, 4), 1),      # head_dim not a multiple of sub_dim
    ((P, P, P, 2, 64, 256, 4, 2, 0, P, 4), 1),       # head_dim below sub_dim
    ((P, None, P, 2, 64, 256, 4, 16, 0, P, 4), 1),   # no factors
    ((P, P + 2, P, 2, 64, 256, 4, 16, 0, P, 4), 1),  # factors not 4-byte aligned
    ((P, P, P, 2, 64, 300, 4, 16, 0, P, 1), 2),      # 8-bit codes, 300 centroids
    ((P, P, P, 2, 60, 256, 6, 12, 0, P, 4), 2),      # sub_dim 6
    ((P + 2, P, P, 2, 64, 256, 4, 16, 0, P, 4), 2),  # x not aligned to its row
    ((None, None, None, 2, 0, 256, 4, 16, 0, None, 4), 0),  # empty groups
])
def test_smooth_argument_errors(lib, args, status):
    assert _smooth(lib)(*args, None) == status


def test_sibling_argument_errors(lib):
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    sq = lib.vq_scalar_quantize
    sq.restype, sq.argtypes = i32, [vp, i32, i64, vp, i32, vp, vp, ctypes.c_size_t, vp]
    assert sq(P, 0, -1, P, 16, P, None, 0, None) == 1       # negative n
    assert sq(P, 5, 10, P, 16, P, None, 0, None) == 1       # unknown dtype
    assert sq(P, 0, 10, P, 0, P, None, 0, None) == 2        # no centroids
    assert sq(P, 0, 10, P, 257, P, None, 0, None) == 2      # more than 8-bit codes
    assert sq(P + 1, 0, 10, P, 16, P, None, 0, None) == 1   # x not aligned to its element
    assert sq(None, 0, 0, None, 16, None, None, 0, None) == 0  # nothing to do
    hr = lib.vq_hadamard_rotate
    hr.restype, hr.argtypes = i32, [vp, i32, vp, i64, i32, vp, vp]
    assert hr(P, 0, P, 10, 96, P, None) == 1                # not a power of two
    assert hr(P, 0, P, 10, 0, P, None) == 1
    assert hr(P, 0, P, 10, 2048, P, None) == 2              # above 1024
    assert hr(P, 0, P, -1, 128, P, None) == 1
    assert hr(None, 0, None, 0, 128, None, None) == 0
    hq = lib.vq_hadamard_quantize
    hq.restype, hq.argtypes = i32, [vp, i32, vp, i64, i32, vp, i32, vp, vp]
    assert hq(P, 0, P, 10, 128, P, 300, P, None) == 2       # more than 8-bit codes
    assert hq(P, 0, P, 10, 128, P, 16, P + 2, None) == 1    # 4-byte index stores
    ws = lib.vq_scalar_quantize_workspace_bytes
    ws.restype, ws.argtypes = ctypes.c_size_t, [i32]
    assert (ws(0), ws(1), ws(2)) == (65536, 65536, 0)


def test_attention_workspace_bytes(lib):
    f = lib.vq_attention_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int64]
    per_slice = 8 * 32 * (128 + 2) * 4
    n = f(8, 32, 8, 32768, 128, 8, 256, 0)
    assert n > 0 and n % per_slice == 0 and n // per_slice <= 32
    assert f(8, 32, 8, 0, 128, 8, 256, 0) == per_slice      # empty cache: one slice
    assert f(8, 32, 8, 500, 128, 8, 256, 0) == per_slice    # one chunk: one slice
    assert f(8, 32, 7, 32768, 128, 8, 256, 0) == 0          # invalid sizes
    assert f(8, 32, 8, 32768, 128, 8, 256, 100) == per_slice  # a short window


def test_describe_launch_picks_kernels(lib):
    f = lib.vq_describe_launch
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_char_p, ctypes.c_int32]
    buf = ctypes.create_string_buffer(512)
    assert f(1, 1 << 20, 256, 4, 0, P, buf, 512) == 0        # fp16: tensor-core screening
    assert buf.value.decode().startswith("kernel=encode_tc")
    assert f(256, 131072, 256, 8, 1, P, buf, 512) == 0       # bf16
    assert buf.value.decode().startswith("kernel=encode_tc")
    assert f(1, 1 << 20, 256, 4, 2, P, buf, 512) == 0        # fp32: tensor cores, split into tf32 pieces
    assert buf.value.decode().startswith("kernel=encode_tc")
    assert f(1, 1 << 20, 300, 4, 2, P, buf, 512) == 0        # fp32, more than 256: CUDA-core screening
    assert buf.value.decode().startswith("kernel=encode_filter")
    assert f(1, 1 << 20, 1000, 8, 0, P, buf, 512) == 0       # more than 256 centroids
    assert buf.value.decode().startswith("kernel=encode_filter")
    assert f(1, 1000, 32, 8, 0, P, buf, 512) == 0           # small codebook: brute force
    assert buf.value.decode().startswith("kernel=encode_fast")
    assert f(1, 1000, 4096, 4, 0, P, buf, 512) == 0         # filter layout too big: brute force
    assert buf.value.decode().startswith("kernel=encode_fast")
    assert f(1, 1000, 256, 5, 0, P, buf, 512) == 0          # odd sub_dim
    assert buf.value.decode().startswith("kernel=encode_general")
    assert f(1, 1000, 256, 4, 0, P + 2, buf, 512) == 0      # x not 8-byte aligned
    assert buf.value.decode().startswith("kernel=encode_general")
    assert f(1, 1000, 4096, 8, 0, P, buf, 512) == 0         # codebook too big for smem
    assert buf.value.decode().startswith("kernel=encode_general")
    assert f(1, 1000, 256, 0, 0, P, buf, 512) == 2


def test_describe_launch_tiles_per_step(lib):
    """The tensor-core encode screens two 128-row tiles per step only for
    16-bit rows at sub_dim 4; rows split into two tf32 pieces (fp32 keys) and
    sub_dim 8 take one tile per step (128-thread blocks)."""
    f = lib.vq_describe_launch
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_char_p, ctypes.c_int32]
    buf = ctypes.create_string_buffer(512)
    for dtype, sub, tps in ((0, 4, 2), (1, 4, 2), (2, 4, 1), (0, 8, 1), (2, 8, 1)):
        assert f(1, 1 << 20, 256, sub, dtype, P, buf, 512) == 0
        desc = buf.value.decode()
        assert desc.startswith("kernel=encode_tc") and f"tiles_per_step={tps} " in desc, desc


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import product_vq_kv_gb300._binding as b

    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        b.load_library()


def test_bench_launch_matches_the_measured_traffic_key(lib):
    """The Falcon-shape launch the benchmark times (152 SMs, as on GB300 and
    as the host assumes without a device) is the launch whose DRAM traffic was
    measured; a planner change that alters it retires that figure."""
    import bench

    f = lib.vq_describe_launch
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_char_p, ctypes.c_int32]
    buf = ctypes.create_string_buffer(512)
    assert f(1, 1 << 20, 256, 4, 0, 1 << 20, buf, 512) == 0
    assert buf.value.decode() in bench.MEASURED_TRAFFIC, buf.value.decode()


def _attention_inputs(torch, b=2, hq=8, hkv=2, t=16, d=128, sub=8, n_c=256):
    q = torch.zeros((b, hq, d), dtype=torch.float16)
    kc = torch.zeros((b, hkv, t, d // sub), dtype=torch.uint8)
    cb = torch.zeros((hkv, n_c, sub), dtype=torch.float16)
    return [q, kc, cb, kc.clone(), cb.clone()]


def _bad_attention_inputs(torch):
    """(description, inputs, exception type, message) cases the Python wrappers
    must reject before a pointer reaches the library."""
    cases = []

    def case(name, edit, exc, match):
        args = _attention_inputs(torch)
        edit(args)
        cases.append((name, args, exc, match))

    case("int32 key codes", lambda a: a.__setitem__(1, a[1].to(torch.int32)), TypeError, "uint8")
    case("int32 value codes", lambda a: a.__setitem__(3, a[3].to(torch.int32)), TypeError, "uint8")
    case("key codebook dtype", lambda a: a.__setitem__(2, a[2].float()), TypeError, "q's dtype")
    case("value codebook dtype", lambda a: a.__setitem__(4, a[4].bfloat16()), TypeError, "q's dtype")
    case("int q", lambda a: a.__setitem__(0, a[0].to(torch.int16)), TypeError, "dtype")
    case("short value codes", lambda a: a.__setitem__(3, a[3][:, :, :8].contiguous()),
         ValueError, "inconsistent")
    case("value codebook rows", lambda a: a.__setitem__(4, a[4][:, :128].contiguous()),
         ValueError, "inconsistent")
    case("key codebook sub_dim", lambda a: a.__setitem__(2, torch.zeros((2, 256, 4), dtype=torch.float16)),
         ValueError, "inconsistent")
    case("batch mismatch", lambda a: a.__setitem__(0, torch.zeros((3, 8, 128), dtype=torch.float16)),
         ValueError, "inconsistent")
    case("2-D q", lambda a: a.__setitem__(0, a[0][0]), ValueError, "expected q")
    case("host tensors", lambda a: None, ValueError, "CUDA tensor")
    return cases


@pytest.mark.parametrize("entry", ["vq_attention_decode", "vq_attention_decode_static"])
def test_attention_wrappers_reject_bad_inputs_before_launch(monkeypatch, entry):
    """Both attention wrappers share one check: wrong code or codebook dtypes,
    inconsistent key and value shapes, and host or non-contiguous tensors all
    raise before any pointer is handed to the library."""
    import torch

    import product_vq_kv_gb300._binding as b

    def no_library():
        raise AssertionError("the library was reached with bad inputs")

    monkeypatch.setattr(b, "load_library", no_library)
    fn = getattr(b, entry)
    for name, args, exc, match in _bad_attention_inputs(torch):
        with pytest.raises(exc, match=match):
            fn(*args)
    # a non-contiguous tensor with consistent shapes is rejected by the device
    # check (on a machine without a GPU, as a host tensor)
    args = _attention_inputs(torch)
    args[0] = torch.zeros((2, 128, 8), dtype=torch.float16).transpose(1, 2)
    with pytest.raises(ValueError, match="CUDA tensor|contiguous"):
        fn(*args)

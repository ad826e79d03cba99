"""GPU test of vq_attention_decode_static, the attention entry point that
allocates nothing (its partials live in the library's built-in device array).

It is called through the C ABI (ctypes, raw device pointers) twice in a row
and each result is compared with vq_attention_decode's on the same inputs.
Both use float atomics, so the two may differ in the last bits: each must lie
within the derived error bound of test_attention.py of the float64 oracle, and
the two within twice that bound of each other.  This file is collected last;
it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


def _static_call(lib, dev, out, window=0, scale=0.0):
    q, kc, kcb, vc, vcb = dev
    b, hq, d = q.shape
    _, hkv, t, _ = kc.shape
    n_c, sub = kcb.shape[1], kcb.shape[2]
    dtype = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}[q.dtype]
    return lib.vq_attention_decode_static(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(kcb.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        ctypes.c_void_p(vcb.data_ptr()), b, hq, hkv, t, d, sub, n_c, window, scale, dtype,
        ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape", [
    # (b, hq, hkv, tokens, head_dim, sub_dim, n_centroids, dtype, window)
    (2, 8, 2, 5000, 128, 8, 256, "f16", 0),
    (1, 32, 8, 3000, 128, 4, 256, "bf16", 1500),
    (16, 32, 8, 20000, 128, 8, 256, "f32", 0),  # default plan exceeds the array: fewer slices
], ids=lambda s: "-".join(map(str, s)))
def test_static_scratch_matches_workspace_entry_point(vq, oracle_mod, shape):
    import test_attention as ta

    b, hq, hkv, t, d, sub, n_c, dtype, window = shape
    host, dev = ta.make_case(77 + b + t, b, hq, hkv, t, d, sub, n_c, dtype)
    lib = vq.load_library()
    ref = vq.vq_attention_decode(*dev, window=window)
    want = oracle_mod.attention_decode(*host, window=window)
    tol = ta.attention_tolerance(*host, window=window, dtype=dtype)
    rel_out = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8, "f32": 0.0}[dtype]
    bound = tol + rel_out * np.abs(want) + 1e-30
    ref_np = ref.to(torch.float64).cpu().numpy()
    assert np.all(np.abs(ref_np - want) <= bound)
    for _ in range(2):  # two calls in a row share the one array
        out = torch.full_like(ref, float("nan"))
        assert _static_call(lib, dev, out, window=window) == vq.VQ_OK
        torch.cuda.synchronize()
        got = out.to(torch.float64).cpu().numpy()
        assert np.all(np.abs(got - want) <= bound)
        assert np.all(np.abs(got - ref_np) <= 2 * bound)


def test_static_scratch_rejects_shapes_beyond_the_array(vq):
    lib = vq.load_library()
    fake = ctypes.c_void_p(0x10000)
    # one slice of partials: 64 * 256 * (128 + 2) * 4 bytes > 8 MiB; rejected
    # during validation, before any pointer is used or anything launched
    st = lib.vq_attention_decode_static(fake, fake, fake, fake, fake, 64, 256, 8, 1000, 128, 8,
                                        256, 0, 0.0, 0, fake, None)
    assert st == vq.VQ_ERR_INVALID_ARG
    q = torch.zeros((64, 256, 128), dtype=torch.float16, device="cuda")
    kc = torch.zeros((64, 8, 10, 16), dtype=torch.uint8, device="cuda")
    cb = torch.zeros((8, 256, 8), dtype=torch.float16, device="cuda")
    with pytest.raises(vq.VQError, match="built-in array holds"):
        vq.vq_attention_decode_static(q, kc, cb, kc, cb)

"""GPU test of vq_attention_decode_static, the attention entry point that
allocates nothing (its partials live in the library's built-in device array).

Some callers cannot allocate device memory per call: a decode loop whose HBM
is fully planned up front, or C host code with no caching allocator, where a
cudaMalloc / cudaFree per step would synchronise the device.  This entry point
serves them.

It is called through the C ABI (ctypes, raw device pointers) twice in a row
and each result is compared with vq_attention_decode's on the same inputs.
The attention kernels use no atomics, so a result depends only on the inputs
and the number of token slices: the two static calls must agree bit for bit,
and with vq_attention_decode too when the default plan's partials fit in the
array (same slices).  Where they do not fit, the static call uses fewer
slices, and both results must lie within the derived error bound of
test_attention.py of the float64 oracle.  This file is collected last; it
also passes alone in a fresh process.
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
    # (b, hq, hkv, tokens, head_dim, sub_dim, n_centroids, dtype, window, same plan)
    (2, 8, 2, 5000, 128, 8, 256, "f16", 0, True),
    (1, 32, 8, 3000, 128, 4, 256, "bf16", 1500, True),
    (16, 32, 8, 20000, 128, 8, 256, "f32", 0, True),
    # default plan: 4 slices of 2.1 MB partials; the array holds 3
    (16, 64, 8, 4000, 512, 16, 256, "f16", 0, False),
], ids=lambda s: "-".join(map(str, s)))
def test_static_scratch_matches_workspace_entry_point(vq, oracle_mod, shape):
    import test_attention as ta

    b, hq, hkv, t, d, sub, n_c, dtype, window, expect_same_plan = shape
    host, dev = ta.make_case(77 + b + t, b, hq, hkv, t, d, sub, n_c, dtype)
    lib = vq.load_library()
    ref = vq.vq_attention_decode(*dev, window=window)
    want = oracle_mod.attention_decode(*host, window=window)
    tol = ta.attention_tolerance(*host, window=window, dtype=dtype)
    rel_out = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8, "f32": 0.0}[dtype]
    bound = tol + rel_out * np.abs(want) + 1e-30
    ref_np = ref.to(torch.float64).cpu().numpy()
    assert np.all(np.abs(ref_np - want) <= bound)
    same_plan = vq.vq_attention_workspace_bytes(b, hq, hkv, t, d, sub, n_c, window) \
        <= vq.ATTN_STATIC_SCRATCH_BYTES
    assert same_plan == expect_same_plan
    first = None
    for _ in range(2):  # two calls in a row share the one array
        out = torch.full_like(ref, float("nan"))
        assert _static_call(lib, dev, out, window=window) == vq.VQ_OK
        torch.cuda.synchronize()
        got = out.to(torch.float64).cpu().numpy()
        assert np.all(np.abs(got - want) <= bound)
        if same_plan:
            assert torch.equal(out, ref)
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out, first)


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

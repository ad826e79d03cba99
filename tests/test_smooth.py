"""GPU parity of the encode fused with per-channel smoothing: indices
bit-identical to the oracle's (each element divided by its channel's factor
in fp32, then the exact encode formula)."""
import os

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


def dev(a, bf16=False):
    a = np.ascontiguousarray(a)
    if bf16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def case(seed, dtype, g, m, n_c, sub, head_dim, spread=0.5):
    rng = np.random.default_rng(seed)
    xf = rng.standard_normal((g, m, sub)).astype(np.float32)
    cf = rng.standard_normal((g, n_c, sub)).astype(np.float32)
    smooth = np.exp(spread * rng.standard_normal((g, head_dim))).astype(np.float32)
    if dtype == "f16":
        return xf.astype(np.float16), smooth, cf.astype(np.float16)
    if dtype == "bf16":
        to = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        return to(xf), smooth, to(cf)
    return xf, smooth, cf


def run(vq, x, smooth, cb, head_dim, bf16, index_bytes):
    out = vq.vq_encode_grouped_smooth(dev(x, bf16), dev(smooth), dev(cb, bf16), head_dim,
                                      index_bytes=index_bytes)
    torch.cuda.synchronize()
    if index_bytes == 1:
        return out.cpu().numpy().astype(np.uint32)
    return out.view(torch.int32).cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("sub,head_dim", [(4, 16), (4, 256), (8, 128)])
@pytest.mark.parametrize("n_c", [7, 64, 256, 1000])
def test_smooth_matches_oracle(vq, oracle_mod, dtype, sub, head_dim, n_c):
    ns = head_dim // sub
    m = ns * (3001 // ns + 1)  # whole key vectors, several tiles and a ragged tail
    x, smooth, cb = case(n_c * 7 + sub + head_dim, dtype, 3, m, n_c, sub, head_dim)
    bf = dtype == "bf16"
    want = oracle_mod.encode_smooth(x, smooth, cb, head_dim, bf16=bf, n_threads=THREADS)
    got = run(vq, x, smooth, cb, head_dim, bf, 4)
    assert np.array_equal(got, want)
    if n_c <= 256:
        assert np.array_equal(run(vq, x, smooth, cb, head_dim, bf, 1), want)


def test_smooth_ones_equals_plain_encode(vq):
    x, _, cb = case(5, "f16", 2, 4096, 256, 4, 64)
    ones = np.ones((2, 64), dtype=np.float32)
    plain = vq.vq_encode_grouped(dev(x), dev(cb)).view(torch.int32).cpu().numpy()
    got = run(vq, x, ones, cb, 64, False, 4).view(np.int32)
    assert np.array_equal(got, plain)


def test_smooth_extreme_factors_and_special_values(vq, oracle_mod):
    """Tiny, huge, zero and negative factors and inf / NaN keys: rows whose
    divided values overflow, vanish or turn NaN follow the oracle (queued rows
    take the exact scan)."""
    x, smooth, cb = case(6, "f32", 2, 32 * 64, 256, 4, 128)
    smooth[0, :8] = [1e-30, 1e30, 0.0, -2.0, 1e-38, 3e38, -0.0, 1e-45]
    x[1, :5, 0] = [np.inf, -np.inf, np.nan, 1e38, -1e38]
    want = oracle_mod.encode_smooth(x, smooth, cb, 128, n_threads=THREADS)
    assert np.array_equal(run(vq, x, smooth, cb, 128, False, 4), want)


@pytest.mark.parametrize("name", ["tiny", "llama_decode", "falcon_prefill", "long_context"])
def test_smooth_full_workloads(vq, oracle_mod, name):
    x, smooth, cb = workloads.generate_smooth(name)
    w = workloads.WORKLOADS[name]
    head_dim = w.sub_vectors_per_head * w.sub_dim
    want = oracle_mod.encode_smooth(x, smooth, cb, head_dim, n_threads=THREADS)
    assert np.array_equal(run(vq, x, smooth, cb, head_dim, False, 1), want)


def test_smooth_empty_and_errors(vq):
    x = torch.zeros((2, 0, 4), dtype=torch.float16, device="cuda")
    cb = torch.zeros((2, 256, 4), dtype=torch.float16, device="cuda")
    s = torch.ones((2, 16), dtype=torch.float32, device="cuda")
    assert vq.vq_encode_grouped_smooth(x, s, cb, 16).shape == (2, 0)
    x = torch.zeros((2, 10, 4), dtype=torch.float16, device="cuda")  # 10 rows, 4 per key
    with pytest.raises(vq.VQError):
        vq.vq_encode_grouped_smooth(x, s, cb, 16)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("sub,head_dim", [(4, 256), (8, 128)])
def test_smooth_tensor_core_extreme_factors(vq, oracle_mod, dtype, sub, head_dim):
    """The tensor-core path (16-bit keys, 64..256 centroids): factors whose
    quotients are subnormal, huge, infinite or NaN (those rows are queued for
    the exact scan), and factors like 1/3 or 1/pi whose quotients use every
    bit of fp32, so all three tf32 pieces of the split are nonzero."""
    ns = head_dim // sub
    x, smooth, cb = case(11 + sub, dtype, 2, ns * 300, 200, sub, head_dim)
    smooth[0, :12] = [1e-30, 1e30, 0.0, -2.0, 1e-38, 3e38, -0.0, 1e-45, 3.0, 7.0, 1 / 3, 1e38]
    smooth[1] = np.float32(1 / np.pi) * (1 + np.arange(head_dim, dtype=np.float32) / 7)
    bf = dtype == "bf16"
    want = oracle_mod.encode_smooth(x, smooth, cb, head_dim, bf16=bf, n_threads=THREADS)
    assert np.array_equal(run(vq, x, smooth, cb, head_dim, bf, 4), want)
    assert np.array_equal(run(vq, x, smooth, cb, head_dim, bf, 1), want)

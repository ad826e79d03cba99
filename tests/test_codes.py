"""GPU parity of the 8-bit-code encode and of the decode (dequantize) path."""
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


def inputs(rng, dtype, g, m, n_c, sub):
    xf = rng.standard_normal((g, m, sub)).astype(np.float32)
    cf = rng.standard_normal((g, n_c, sub)).astype(np.float32)
    if dtype == "f16":
        return xf.astype(np.float16), cf.astype(np.float16)
    if dtype == "bf16":
        to = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        return to(xf), to(cf)
    return xf, cf


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("sub_dim", [4, 8, 3])
@pytest.mark.parametrize("n_c", [7, 64, 200, 256])
def test_u8_codes_equal_u32_indices(vq, oracle_mod, dtype, sub_dim, n_c):
    rng = np.random.default_rng(n_c * 10 + sub_dim)
    x, cb = inputs(rng, dtype, 3, 3001, n_c, sub_dim)
    bf = dtype == "bf16"
    xd, cbd = dev(x, bf), dev(cb, bf)
    u32 = vq.vq_encode_grouped(xd, cbd).cpu().numpy()
    u8 = vq.vq_encode_grouped_u8(xd, cbd).cpu().numpy()
    assert u8.dtype == np.uint8
    assert np.array_equal(u8.astype(np.uint32), u32)
    assert np.array_equal(u32, oracle_mod.encode(x, cb, bf16=bf, n_threads=THREADS))


def test_u8_rejects_large_codebooks(vq):
    x = torch.zeros((1, 10, 4), dtype=torch.float16, device="cuda")
    cb = torch.zeros((1, 257, 4), dtype=torch.float16, device="cuda")
    with pytest.raises(vq.VQError) as e:
        vq.vq_encode_grouped_u8(x, cb)
    assert e.value.status == vq.VQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["llama_decode", "grouped_adversarial"])
def test_u8_full_size_workload(vq, name):
    x, cb = workloads.generate(name)
    xd, cbd = dev(x), dev(cb)
    u32 = vq.vq_encode_grouped(xd, cbd)
    u8 = vq.vq_encode_grouped_u8(xd, cbd)
    assert torch.equal(u8.to(torch.int32), u32.view(torch.int32))


@pytest.mark.parametrize("index", ["u32", "u8"])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("sub_dim", [4, 8, 1, 3, 16])
def test_dequantize_matches_oracle(vq, oracle_mod, index, dtype, sub_dim):
    rng = np.random.default_rng(sub_dim * 3 + len(dtype))
    g, m, n_c = 3, 5003, 256
    _, cb = inputs(rng, dtype, g, 1, n_c, sub_dim)
    hi = n_c + 20  # some out-of-range indices
    idx = rng.integers(0, hi if index == "u32" else 256, (g, m)).astype(
        np.uint32 if index == "u32" else np.uint8)
    got = vq.vq_dequantize_grouped(torch.from_numpy(idx).cuda(), dev(cb, dtype == "bf16"))
    got = got.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else got.numpy()
    want = oracle_mod.dequantize(idx, cb)
    assert np.array_equal(got.view(np.uint8), want.view(np.uint8))  # bit for bit


def test_dequantize_misaligned_output_takes_element_path(vq, oracle_mod):
    rng = np.random.default_rng(3)
    cb = rng.standard_normal((1, 256, 8)).astype(np.float16)
    idx = rng.integers(0, 256, (1, 999)).astype(np.uint32)
    buf = torch.zeros(999 * 8 + 1, dtype=torch.float16, device="cuda")
    out = buf[1:].view(1, 999, 8)
    vq.vq_dequantize_grouped(torch.from_numpy(idx).cuda(), dev(cb), out=out)
    assert np.array_equal(out.cpu().numpy(), oracle_mod.dequantize(idx, cb))


def test_encode_decode_round_trip_on_workload(vq, oracle_mod):
    x, cb = workloads.generate("grouped_adversarial", tokens=64)
    xd, cbd = dev(x), dev(cb)
    codes = vq.vq_encode_grouped_u8(xd, cbd)
    rec = vq.vq_dequantize_grouped(codes, cbd).cpu().numpy()
    want = oracle_mod.dequantize(oracle_mod.encode(x, cb, n_threads=THREADS), cb)
    assert np.array_equal(rec, want)
    copies = (x[:, :, None, :] == cb[:, None, :, :]).all(-1).any(-1)
    assert copies.sum() > 0 and np.array_equal(rec[copies], x[copies])


def test_dequantize_full_size(vq, oracle_mod):
    x, cb = workloads.generate("grouped_adversarial")
    cbd = dev(cb)
    codes = vq.vq_encode_grouped_u8(dev(x), cbd)
    rec = vq.vq_dequantize_grouped(codes, cbd)
    rows = np.random.default_rng(0).integers(0, x.shape[1], 2000)
    c = codes.cpu().numpy()[:, rows]
    assert np.array_equal(rec.cpu().numpy()[:, rows], oracle_mod.dequantize(c, cb))


def test_dequantize_argument_errors(vq):
    lib = vq.load_library()
    assert lib.vq_dequantize_grouped(None, 4, None, 1, 0, 256, 4, 0, None, None) == 0
    assert lib.vq_dequantize_grouped(None, 2, None, 1, 5, 256, 4, 0, None, None) == 1
    assert lib.vq_dequantize_grouped(16, 4, 16, 1, 5, 256, 0, 0, 16, None) == 2

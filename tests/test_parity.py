"""GPU parity: the CUDA encoder against the CPU oracle, index for index.

The bar is bit-exact: both sides evaluate the same fp32 formula (separate
round-to-nearest subtract, square and add in ascending i; strict "<" argmin),
so every index must agree.  Cases span several tiles with ragged tails, every
dtype, both fast sub_dims and the general kernel, the configured workloads
(small enough for the oracle in full, and at full size on sampled rows in the
launch configuration the benchmark times), and the method's degenerate cases.
"""
import os

import numpy as np
import pytest
import torch

import workloads
from conftest import parse_pow2_sum  # noqa: F401  (shared helpers)

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


def to_dev(a: np.ndarray, bf16: bool = False) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if bf16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def gpu_encode(vq, x, cb, bf16=False):
    xd, cbd = to_dev(x, bf16), to_dev(cb, bf16)
    if x.ndim == 2:
        out = vq.vq_encode(xd, cbd)
    else:
        out = vq.vq_encode_grouped(xd, cbd)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def random_inputs(rng, dtype, g, m, n_c, sub):
    xf = rng.standard_normal((g, m, sub)).astype(np.float32)
    cf = rng.standard_normal((g, n_c, sub)).astype(np.float32)
    if dtype == "f16":
        return xf.astype(np.float16), cf.astype(np.float16)
    if dtype == "bf16":
        xb = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        cb = torch.from_numpy(cf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        return xb, cb
    return xf, cf


def assert_same(got, want):
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got.ravel() != want.ravel())
        raise AssertionError(f"{bad.size} of {want.size} indices differ; first rows {bad[:8]}, "
                             f"gpu {got.ravel()[bad[:8]]}, oracle {want.ravel()[bad[:8]]}")


# ---------------------------------------------------------------- workloads


@pytest.mark.parametrize("name,tokens", [
    ("tiny", None),
    ("llama_decode", None),
    ("falcon_prefill", None),
    ("long_context", 2048),
    ("grouped_adversarial", 64),
])
def test_workload_bit_exact(vq, oracle_mod, name, tokens):
    x, cb = workloads.generate(name, tokens=tokens)
    got = gpu_encode(vq, x, cb)
    assert_same(got, oracle_mod.encode(x, cb, n_threads=THREADS))


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_full_size_workload_sampled(vq, oracle_mod, name):
    """Full-size inputs, the benchmark's launch (one grouped call); the oracle
    checks a sample of rows: random ones plus the first and last rows of every
    group (tile and group boundaries)."""
    x, cb = workloads.generate(name)
    got = gpu_encode(vq, x, cb)
    g, m, _ = x.shape
    rng = np.random.default_rng(7)
    for k in range(g):
        rows = np.unique(np.concatenate([
            np.arange(min(m, 40)), np.arange(max(0, m - 40), m),
            rng.integers(0, m, max(1, 40000 // g))]))
        want = oracle_mod.encode(x[k, rows], cb[k], n_threads=THREADS)
        assert_same(got[k, rows], want)


@pytest.mark.parametrize("name", ["long_context", "grouped_adversarial"])
def test_full_size_workload_every_row(vq, oracle_mod, name):
    """Every row of the two largest workloads at full size (4.2 M and 33.5 M
    sub-vectors, the benchmark's single grouped launch) against the oracle,
    and the adversarial invariants on the whole cache: every exact copy of a
    centroid maps to the lowest index holding that row."""
    x, cb = workloads.generate(name)
    got = gpu_encode(vq, x, cb)
    assert_same(got, oracle_mod.encode(x, cb, n_threads=THREADS))
    if name == "grouped_adversarial":
        g, m, sub = x.shape
        for k in range(0, g, 37):  # a spread of groups: exact-copy rows
            rows = x[k].view(np.uint16).reshape(m, sub)
            cbr = cb[k].view(np.uint16).reshape(-1, sub)
            lut = {}
            for c in range(cbr.shape[0] - 1, -1, -1):  # lowest index wins
                lut[cbr[c].tobytes()] = c
            hits = [(r, lut[rows[r].tobytes()]) for r in range(m) if rows[r].tobytes() in lut]
            assert len(hits) >= 1000
            for r, c in hits:
                assert got[k, r] == c, (k, r, c, got[k, r])


# ---------------------------------------------------------------- dtypes and shapes


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("sub_dim", [4, 8])
@pytest.mark.parametrize("n_c", [1, 2, 7, 255, 256, 257, 1000])
def test_fast_path_shapes(vq, oracle_mod, dtype, sub_dim, n_c):
    rng = np.random.default_rng(1000 + sub_dim * 7 + n_c)
    x, cb = random_inputs(rng, dtype, 3, 2500, n_c, sub_dim)
    got = gpu_encode(vq, x, cb, bf16=dtype == "bf16")
    assert_same(got, oracle_mod.encode(x, cb, bf16=dtype == "bf16", n_threads=THREADS))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("sub_dim", [1, 2, 3, 5, 7, 12, 16, 32])
def test_general_path_shapes(vq, oracle_mod, dtype, sub_dim):
    rng = np.random.default_rng(2000 + sub_dim)
    x, cb = random_inputs(rng, dtype, 2, 700, 256, sub_dim)
    got = gpu_encode(vq, x, cb, bf16=dtype == "bf16")
    assert_same(got, oracle_mod.encode(x, cb, bf16=dtype == "bf16", n_threads=THREADS))


@pytest.mark.parametrize("n", [1, 2, 31, 255, 1023, 1024, 1025, 2047, 2049, 5000])
@pytest.mark.parametrize("sub_dim", [4, 8])
def test_ragged_sizes(vq, oracle_mod, n, sub_dim):
    rng = np.random.default_rng(n)
    x, cb = random_inputs(rng, "f16", 1, n, 256, sub_dim)
    assert_same(gpu_encode(vq, x[0], cb[0]), oracle_mod.encode(x[0], cb[0]))


@pytest.mark.parametrize("sub_dim", [4, 8])
def test_max_centroids(vq, oracle_mod, sub_dim):
    rng = np.random.default_rng(4096 + sub_dim)
    x, cb = random_inputs(rng, "f16", 1, 3000, 4096, sub_dim)
    assert_same(gpu_encode(vq, x, cb), oracle_mod.encode(x, cb, n_threads=THREADS))


def test_many_small_groups(vq, oracle_mod):
    rng = np.random.default_rng(31)
    x, cb = random_inputs(rng, "f16", 1000, 37, 256, 8)
    assert_same(gpu_encode(vq, x, cb), oracle_mod.encode(x, cb, n_threads=THREADS))


def test_empty_inputs(vq):
    x = torch.zeros((0, 4), dtype=torch.float16, device="cuda")
    cb = torch.zeros((256, 4), dtype=torch.float16, device="cuda")
    assert vq.vq_encode(x, cb).shape == (0,)
    xg = torch.zeros((5, 0, 8), dtype=torch.float16, device="cuda")
    cbg = torch.zeros((5, 256, 8), dtype=torch.float16, device="cuda")
    assert vq.vq_encode_grouped(xg, cbg).shape == (5, 0)


@pytest.mark.parametrize("sub_dim", [4, 8])
def test_misaligned_x_takes_general_path(vq, oracle_mod, sub_dim):
    rng = np.random.default_rng(77)
    x, cb = random_inputs(rng, "f16", 1, 3001, 256, sub_dim)
    flat = torch.from_numpy(x.reshape(-1)).cuda()
    buf = torch.empty(flat.numel() + 1, dtype=torch.float16, device="cuda")
    buf[1:] = flat
    xd = buf[1:].view(3001, sub_dim)  # 2-byte offset: not 8/16-byte aligned
    desc = vq.vq_describe_launch(1, 3001, 256, sub_dim, torch.float16, xd.data_ptr())
    assert desc.startswith("kernel=encode_general")
    out = vq.vq_encode(xd, torch.from_numpy(cb[0]).cuda())
    torch.cuda.synchronize()
    assert_same(out.cpu().numpy(), oracle_mod.encode(x[0], cb[0]))


# ---------------------------------------------------------------- degenerate cases


def test_exact_copies_and_duplicate_centroids(vq, oracle_mod):
    rng = np.random.default_rng(55)
    cb = rng.standard_normal((256, 8)).astype(np.float16)
    cb[100] = cb[5]
    cb[3] = cb[200]
    cb[9] = -0.0
    cb[10] = 0.0
    src = rng.integers(0, 256, 5000)
    x = cb[src].copy()
    got = gpu_encode(vq, x, cb)
    first_equal = np.array([np.flatnonzero((cb == cb[s]).all(1))[0] for s in src])
    assert_same(got, first_equal)
    assert_same(got, oracle_mod.encode(x, cb))


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
@pytest.mark.parametrize("sub_dim", [4, 8])
def test_special_values(vq, oracle_mod, dtype, sub_dim):
    rng = np.random.default_rng(9)
    cb = rng.standard_normal((256, sub_dim)).astype(dtype)
    cb[0, 0] = np.nan
    cb[17, 1] = np.inf
    cb[18, 2] = -np.inf
    x = rng.standard_normal((2048, sub_dim)).astype(dtype)
    x[0, 0] = np.nan
    x[1, 1] = np.inf
    x[2, :] = -np.inf
    x[3] = cb[0]          # copy of the NaN row: NaN distance to itself, never wins
    x[4] = cb[17]         # +inf component
    x[5, 0] = 60000 if dtype == np.float16 else 3e38
    got = gpu_encode(vq, x, cb)
    assert_same(got, oracle_mod.encode(x, cb))
    assert got[0] == 0 and got[1] == 0 and got[2] == 0


def _pow2(values):
    from conftest import parse_pow2_sum

    return np.array([float(parse_pow2_sum(v)) for v in values], dtype=np.float32)


def _pad(rows, sub_dim):
    out = np.zeros((len(rows), sub_dim), np.float32)
    for k, r in enumerate(rows):
        out[k, :len(r)] = r
    return out


@pytest.mark.parametrize("sub_dim", [4, 8])
def test_rounding_trap_no_fma(vq, oracle_mod, sub_dim):
    """x = (2^-12, 1+2^-12): with separate rounding its distance to the zero
    centroid (index 0) is 1+2^-11, equal to that of an exactly representable
    competitor (index 1), so the tie goes to 0; a fused multiply-add would make
    it 1+2^-11+2^-23 and pick 1."""
    x = _pad([_pow2(["2^-12", "1+2^-12"])], sub_dim)
    comp = _pow2(["2^-12+-1", "1+2^-12+-2^-6", "-2^-6", "0"])
    cb = _pad([np.zeros(4, np.float32), comp], sub_dim)
    assert oracle_mod.encode(x, cb).tolist() == [0]
    assert gpu_encode(vq, x, cb).tolist() == [0]


@pytest.mark.parametrize("sub_dim", [4, 8])
def test_rounding_trap_ascending_order(vq, oracle_mod, sub_dim):
    """Rows whose distance to the zero centroid (index 1) is 1.0 only when the
    squares are added in ascending i; adding in reverse, or pairwise, gives
    1+2^-23, a tie with the exact competitor at index 0."""
    xs = _pad([_pow2(["1", "2^-12", "2^-12", "0"]), _pow2(["1", "0", "2^-12", "2^-12"])],
              sub_dim)
    comps = [_pow2(["1+-2^-12", "0", "2^-12+-1", "0"]),
             _pow2(["1+-2^-12", "-2^-12", "2^-12+-1", "2^-12"])]
    for x, comp in zip(xs, comps):
        cb = _pad([comp, np.zeros(4, np.float32)], sub_dim)
        assert oracle_mod.encode(x[None], cb).tolist() == [1]
        assert gpu_encode(vq, x[None], cb).tolist() == [1]


# ---------------------------------------------------------------- execution model


def test_side_stream_and_repeatability(vq, oracle_mod):
    x, cb = workloads.generate("llama_decode")
    xd, cbd = to_dev(x), to_dev(cb)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        a = vq.vq_encode_grouped(xd, cbd)
        b = vq.vq_encode_grouped(xd, cbd)
    side.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert_same(a.cpu().numpy(), oracle_mod.encode(x, cb, n_threads=THREADS))


def test_no_device_allocation(vq):
    x, cb = workloads.generate("falcon_prefill")
    xd, cbd = to_dev(x), to_dev(cb)
    out = torch.empty(x.shape[:2], dtype=torch.uint32, device="cuda")
    vq.vq_encode_grouped(xd, cbd, out=out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        vq.vq_encode_grouped(xd, cbd, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("g,m,sub", [(1, 9_000_000, 4), (3, 3_000_000, 8), (40, 9000, 8),
                                     (2, 7, 4)])
def test_host_entry_point(vq, oracle_mod, g, m, sub, pinned):
    """Host buffers in, host buffers out.  Pinned buffers are read and written
    by the kernel directly (the device scratch stays untouched); pageable ones
    go through the device buffers, in overlapped chunks when large.  Both must
    give the device entry point's indices, twice in a row."""
    rng = np.random.default_rng(g * 1000 + sub)
    x = rng.standard_normal((g, m, sub)).astype(np.float16)
    cb = rng.standard_normal((g, 256, sub)).astype(np.float16)
    xh, cbh = torch.from_numpy(x), torch.from_numpy(cb)
    outh = torch.full((g, m), 0xFFFF, dtype=torch.int32).view(torch.uint32)
    if pinned:
        xh, cbh, outh = xh.pin_memory(), cbh.pin_memory(), outh.pin_memory()
    xd = torch.full(x.shape, 7.0, dtype=torch.float16, device="cuda")
    cbd = torch.empty(cb.shape, dtype=torch.float16, device="cuda")
    outd = torch.full((g, m), 12345, dtype=torch.int32, device="cuda").view(torch.uint32)
    want = vq.vq_encode_grouped(torch.from_numpy(x).cuda(), torch.from_numpy(cb).cuda())
    want = want.cpu().numpy()
    for _ in range(2):
        vq.vq_encode_grouped_host(xh, cbh, outh, xd, cbd, outd)
        assert_same(outh.numpy(), want)
    if pinned:
        torch.cuda.synchronize()
        assert bool((xd == 7.0).all()) and bool((outd.view(torch.int32) == 12345).all())
    rows = np.unique(rng.integers(0, m, 2000))
    assert_same(want[:, rows], oracle_mod.encode(x[:, rows], cb, n_threads=THREADS))


def test_host_entry_point_pageable_codebooks(vq):
    """Pinned keys and indices with pageable codebooks: the kernel still
    reads the keys in place, and the codebooks are copied to the device
    buffer first."""
    rng = np.random.default_rng(77)
    x = rng.standard_normal((4, 50000, 8)).astype(np.float16)
    cb = rng.standard_normal((4, 256, 8)).astype(np.float16)
    xh = torch.from_numpy(x).pin_memory()
    outh = torch.empty((4, 50000), dtype=torch.int32).pin_memory().view(torch.uint32)
    xd = torch.empty(x.shape, dtype=torch.float16, device="cuda")
    cbd = torch.zeros(cb.shape, dtype=torch.float16, device="cuda")
    outd = torch.empty((4, 50000), dtype=torch.int32, device="cuda").view(torch.uint32)
    want = vq.vq_encode_grouped(torch.from_numpy(x).cuda(), torch.from_numpy(cb).cuda()).cpu().numpy()
    vq.vq_encode_grouped_host(xh, torch.from_numpy(cb), outh, xd, cbd, outd)
    assert_same(outh.numpy(), want)
    torch.cuda.synchronize()
    assert torch.equal(cbd.cpu(), torch.from_numpy(cb))


def test_argument_errors_raise(vq):
    x = torch.zeros((10, 4), dtype=torch.float16, device="cuda")
    cb = torch.zeros((5000, 4), dtype=torch.float16, device="cuda")
    with pytest.raises(vq.VQError) as e:
        vq.vq_encode(x, cb)
    assert e.value.status == vq.VQ_ERR_UNSUPPORTED

"""GPU parity of the screening encoders on inputs built to stress them.

Both screening kernels -- tensor-core scores (fp16 / bf16 inputs with at most
256 centroids) and fused multiply-add scores on the CUDA cores (fp32 inputs,
larger codebooks) -- screen centroids with a bounded-error score and
re-evaluate
the exact formula only inside the centroid groups its error bound cannot rule
out; rows with three or more such groups, or with non-finite or huge values,
go to an exact per-block queue.  These cases put the deciding difference at
the last bit of the fp32 distance, spread tied centroids over several groups,
and push rows into the queue, and every index must still equal the oracle's.
"""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


def run(vq, x, cb):
    xd, cbd = torch.from_numpy(np.ascontiguousarray(x)).cuda(), torch.from_numpy(cb).cuda()
    desc = vq.vq_describe_launch(x.shape[0], x.shape[1], cb.shape[1], x.shape[2],
                                 xd.dtype, xd.data_ptr())
    out = vq.vq_encode_grouped(xd, cbd)
    torch.cuda.synchronize()
    return out.cpu().numpy(), desc


def expected_kernel(dtype, n_c):
    if n_c > 1024:
        return ""  # large codebooks: whichever exact kernel fits in shared memory
    if n_c < 64:
        return "encode_fast"
    if n_c <= 256:
        return "encode_tc"
    return "encode_filter"


def check(vq, oracle_mod, x, cb, kernel=None):
    got, desc = run(vq, x, cb)
    kernel = kernel or expected_kernel(x.dtype.type, cb.shape[1])
    assert desc.startswith("kernel=" + kernel), desc
    want = oracle_mod.encode(x, cb, n_threads=THREADS)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"


@pytest.mark.parametrize("n_c", [256, 320])
@pytest.mark.parametrize("dtype", [np.float16, np.float32])
@pytest.mark.parametrize("sub_dim", [4, 8])
def test_permuted_coordinate_ties(vq, oracle_mod, sub_dim, dtype, n_c):
    """Rows x = (a, a, b, b, ...) are exactly equidistant (in real arithmetic)
    from a centroid and its copy with coordinates swapped pairwise; the fp32
    sums differ only by rounding order, so the winner is decided at the last
    bit.  The swapped copies sit in other centroid groups."""
    rng = np.random.default_rng(11 + sub_dim)
    m = 20000  # 256 centroids: the tensor-core kernel; 320: the filter kernel
    half = n_c // 2
    base = rng.standard_normal((half, sub_dim)).astype(dtype)
    swapped = base.reshape(half, sub_dim // 2, 2)[:, :, ::-1].reshape(half, sub_dim)
    cb = np.empty((n_c, sub_dim), dtype)
    cb[0::2] = base          # centroid 2k
    cb[1::2] = swapped       # centroid 2k+1, same group
    perm = rng.permutation(n_c)
    cb = cb[perm]            # scatter the partners over all groups
    pairs = rng.standard_normal((m, sub_dim // 2)).astype(dtype)
    x = np.repeat(pairs, 2, axis=1)  # (a, a, b, b, ...)
    check(vq, oracle_mod, x[None], cb[None])


@pytest.mark.parametrize("n_c", [256, 320])
@pytest.mark.parametrize("dtype", [np.float16, np.float32])
@pytest.mark.parametrize("copies", [2, 3, 5])
def test_duplicated_centroids_across_groups(vq, oracle_mod, copies, dtype, n_c):
    """Exact duplicate centroids in `copies` different groups: with three or
    more, rows near them take the exact queue."""
    rng = np.random.default_rng(20 + copies)
    sub = 8
    cb = rng.standard_normal((n_c, sub)).astype(dtype)
    for src in range(0, 40, 4):
        for k in range(1, copies):
            cb[(src + 37 * k) % n_c] = cb[src]
    src = rng.integers(0, n_c, 30000)
    x = cb[src].astype(np.float32)
    x += rng.standard_normal(x.shape).astype(np.float32) * 0.05
    check(vq, oracle_mod, x.astype(dtype)[None], cb[None])


@pytest.mark.parametrize("n_c", [256, 320])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_extreme_magnitudes(vq, oracle_mod, dtype, n_c):
    """Huge rows (queued: the bound would be near overflow) and tiny rows
    (gradual underflow; the bound's absolute term) next to ordinary ones."""
    rng = np.random.default_rng(5)
    sub = 4
    cb = rng.standard_normal((n_c, sub)).astype(np.float32)
    x = rng.standard_normal((6000, sub)).astype(np.float32)
    x[:1000] *= 1e25
    x[1000:2000] *= 1e-30
    cb[:8] *= 1e-30
    if dtype == "bf16":
        xt = torch.from_numpy(x).to(torch.bfloat16)
        ct = torch.from_numpy(cb).to(torch.bfloat16)
        got = None
        desc = vq.vq_describe_launch(1, x.shape[0], n_c, sub, torch.bfloat16, xt.cuda().data_ptr())
        assert desc.startswith("kernel=" + expected_kernel("bf16", n_c))
        got = vq.vq_encode(xt.cuda(), ct.cuda()).cpu().numpy()
        want = oracle_mod.encode(xt.view(torch.int16).numpy().view(np.uint16),
                                 ct.view(torch.int16).numpy().view(np.uint16), bf16=True,
                                 n_threads=THREADS)
        assert np.array_equal(got, want)
    else:
        check(vq, oracle_mod, x[None], cb[None])


@pytest.mark.parametrize("n_c", [256, 320])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["all_subnormal", "one_dim_subnormal"])
def test_subnormal_codebooks(vq, oracle_mod, layout, dtype, n_c):
    """Codebooks whose coordinates (all, or those of one dimension) are fp32
    subnormals, against rows at the same scale, rows far below it and rows
    with a huge coordinate: the regime where splits lose bits below 2^-136
    and the tensor core may flush operands, covered by the bound's absolute
    term and its floor on the per-dimension maxima."""
    rng = np.random.default_rng(31)
    sub = 4
    cb = rng.standard_normal((n_c, sub)).astype(np.float32)
    tiny = np.float32(2.0 ** -132)
    if layout == "all_subnormal":
        cb *= tiny
    else:
        cb[:, 0] *= tiny
    src = rng.integers(0, n_c, 8000)
    x = cb[src] + rng.standard_normal((8000, sub)).astype(np.float32) * (cb.std(axis=0) * 0.3)
    x[:1000] *= np.float32(2.0 ** -10)
    x[1000:2000, 0] = rng.standard_normal(1000).astype(np.float32) * np.float32(1e20)
    x[2000:3000, 0] = rng.standard_normal(1000).astype(np.float32) * np.float32(2.0 ** -100)
    x = x.astype(np.float32)
    assert (np.abs(cb[cb != 0]) < 2.0 ** -126).any()
    if dtype == "bf16":
        xt = torch.from_numpy(x).to(torch.bfloat16)
        ct = torch.from_numpy(cb).to(torch.bfloat16)
        xd = xt.cuda()
        desc = vq.vq_describe_launch(1, x.shape[0], n_c, sub, torch.bfloat16, xd.data_ptr())
        assert desc.startswith("kernel=" + expected_kernel("bf16", n_c)), desc
        got = vq.vq_encode(xd, ct.cuda()).cpu().numpy()
        want = oracle_mod.encode(xt.view(torch.int16).numpy().view(np.uint16),
                                 ct.view(torch.int16).numpy().view(np.uint16), bf16=True,
                                 n_threads=THREADS)
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}"
    else:
        check(vq, oracle_mod, x[None], cb[None])


@pytest.mark.parametrize("n_c", [200, 300])
def test_codebook_with_nan_queues_every_row(vq, oracle_mod, n_c):
    rng = np.random.default_rng(6)
    cb = rng.standard_normal((n_c, 4)).astype(np.float16)
    cb[123, 2] = np.nan
    x = rng.standard_normal((5000, 4)).astype(np.float16)
    check(vq, oracle_mod, x[None], cb[None])


@pytest.mark.parametrize("sub_dim", [4, 8])
@pytest.mark.parametrize("n_c", [63, 64, 65, 100, 224, 255, 256, 257, 512, 2000])
def test_codebook_sizes_around_the_groups(vq, oracle_mod, n_c, sub_dim):
    rng = np.random.default_rng(n_c + sub_dim)
    x = rng.standard_normal((2, 3000, sub_dim)).astype(np.float16)
    cb = rng.standard_normal((2, n_c, sub_dim)).astype(np.float16)
    check(vq, oracle_mod, x, cb)


@pytest.mark.parametrize("n_c", [256, 320])
@pytest.mark.parametrize("dtype", [np.float16, np.float32])
@pytest.mark.parametrize("scale", [0.01, 1000.0])
def test_clustered_keys_near_many_centroids(vq, oracle_mod, dtype, scale, n_c):
    """Keys concentrated near the origin, where many centroids are at similar
    distances (more candidate groups per row), at small and large scale."""
    rng = np.random.default_rng(8)
    cb = (rng.standard_normal((n_c, 8)) * scale).astype(dtype)
    x = (rng.standard_normal((20000, 8)) * scale).astype(dtype)
    check(vq, oracle_mod, x[None], cb[None])


@pytest.mark.parametrize("m", [1, 127, 128, 129, 1023, 1024, 1025, 3000])
def test_tensor_core_tile_boundaries(vq, oracle_mod, m):
    """Row counts around the 128-row tensor-core tile and the 1024-row block."""
    rng = np.random.default_rng(m)
    x = rng.standard_normal((3, m, 4)).astype(np.float16)
    cb = rng.standard_normal((3, 256, 4)).astype(np.float16)
    check(vq, oracle_mod, x, cb)

"""Row counts past 2^31, and group offsets past 2^32 elements of x: the sizes at
which any 32-bit row, tile or element offset would wrap.

One group of 2^31 + 4099 fp16 sub-vectors (sub_dim 4, 256 centroids: the
tensor-core kernel, a ragged last tile) is encoded to uint32 indices and to
8-bit codes, and the codes are decoded; three groups of 2^30 + 77 rows are
encoded in one grouped launch.  Checks, at full size on the GPU: every output
was written and is a valid index (the output is pre-filled with a value no
index takes), the 8-bit codes equal the uint32 indices, and the decode is the
codebook gather.  Against the oracle: sampled rows, among them the first and
last rows, the rows around 2^31 and 2^30, and the group boundaries.
The inputs are seeded N(0, 1) draws made on the device.
"""
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1
SUB, NC = 4, 256
M_FLAT = (1 << 31) + 4099
G_GROUPED, M_GROUPED = 3, (1 << 30) + 77
CHUNK = 1 << 27          # rows per full-size comparison step
SENTINEL = -559038737    # 0xDEADBEEF as int32: above any index, not the failure marker


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


@pytest.fixture(scope="module")
def big():
    rows = G_GROUPED * M_GROUPED
    x_bytes = rows * SUB * 2
    # x, the uint32 indices of the larger case, 8-bit codes, the decode of the
    # one-group case, and room for the comparison temporaries
    need = x_bytes + rows * 4 + M_FLAT + M_FLAT * SUB * 2 + (4 << 30)
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB of free device memory, {free / 2**30:.0f} GiB free")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(20251)
    x = torch.empty(rows * SUB, dtype=torch.float16, device="cuda")
    step = CHUNK * SUB
    for a in range(0, x.numel(), step):
        x[a:a + step].normal_(generator=gen)
    cb = torch.randn((G_GROUPED, NC, SUB), generator=gen, device="cuda").to(torch.float16)
    yield x, cb
    del x, cb
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def sample_rows(m: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    parts = [np.arange(0, 2000), np.arange(m - 2000, m), rng.integers(0, m, 12000)]
    for centre in (1 << 31, 1 << 30, 1 << 29):
        if centre < m:
            parts.append(np.arange(max(0, centre - 1000), min(m, centre + 1000)))
    return np.unique(np.concatenate(parts)).astype(np.int64)


def sentinel_out(g: int, m: int) -> tuple[torch.Tensor, torch.Tensor]:
    """A [G, M] int32 buffer filled with the sentinel, and its uint32 view."""
    o = torch.full((g, m), SENTINEL, dtype=torch.int32, device="cuda")
    return o, o.view(torch.uint32)


def assert_all_valid(o: torch.Tensor) -> None:
    """Every entry written and in [0, NC), checked chunk by chunk on the GPU."""
    flat = o.reshape(-1)
    for a in range(0, flat.numel(), CHUNK):
        c = flat[a:a + CHUNK]
        bad = (c < 0) | (c >= NC)
        if bool(bad.any()):
            first = a + int(torch.nonzero(bad)[0, 0])
            raise AssertionError(f"entry {first} is {int(flat[first])} (sentinel {SENTINEL})")


def check_sampled(oracle_mod, x3: torch.Tensor, cb: torch.Tensor, o: torch.Tensor, seed: int):
    """Sampled rows of every group against the oracle."""
    g, m, _ = x3.shape
    for k in range(g):
        rows = sample_rows(m, seed + k)
        ridx = torch.from_numpy(rows).cuda()
        xs = x3[k].index_select(0, ridx).cpu().numpy()
        got = o[k].index_select(0, ridx).cpu().numpy().astype(np.int64)
        want = oracle_mod.encode(xs[None], cb[k:k + 1].cpu().numpy(), n_threads=THREADS)[0]
        bad = np.nonzero(got != want.astype(np.int64))[0]
        assert bad.size == 0, (f"group {k}: {bad.size} of {rows.size} sampled rows differ, first "
                               f"row {rows[bad[0]]}: {got[bad[0]]} vs {want[bad[0]]}")


def test_one_group_past_2_31_rows(vq, oracle_mod, big):
    x, cb = big
    x3 = x[:M_FLAT * SUB].view(1, M_FLAT, SUB)
    cb1 = cb[:1].contiguous()
    desc = vq.vq_describe_launch(1, M_FLAT, NC, SUB, torch.float16, x3.data_ptr())
    assert desc.startswith("kernel=encode_tc"), desc

    o, out = sentinel_out(1, M_FLAT)
    vq.vq_encode_grouped(x3, cb1, out=out)
    torch.cuda.synchronize()
    assert_all_valid(o)
    check_sampled(oracle_mod, x3, cb1, o, seed=71)

    codes = vq.vq_encode_grouped_u8(x3, cb1)
    torch.cuda.synchronize()
    for a in range(0, M_FLAT, CHUNK):
        assert torch.equal(codes[0, a:a + CHUNK].to(torch.int32), o[0, a:a + CHUNK]), a
    del o, out

    dec = vq.vq_dequantize_grouped(codes, cb1)
    torch.cuda.synchronize()
    for a in range(0, M_FLAT, CHUNK):
        assert torch.equal(dec[0, a:a + CHUNK], cb1[0][codes[0, a:a + CHUNK].long()]), a
    rows = torch.from_numpy(sample_rows(M_FLAT, 72)).cuda()
    want = oracle_mod.dequantize(codes[0].index_select(0, rows).cpu().numpy()[None],
                                 cb1.cpu().numpy())[0]
    got = dec[0].index_select(0, rows).cpu().numpy()
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    del codes, dec
    torch.cuda.empty_cache()


def test_grouped_offsets_past_2_32_elements(vq, oracle_mod, big):
    x, cb = big
    x3 = x.view(G_GROUPED, M_GROUPED, SUB)
    o, out = sentinel_out(G_GROUPED, M_GROUPED)
    vq.vq_encode_grouped(x3, cb, out=out)
    torch.cuda.synchronize()
    assert_all_valid(o)
    check_sampled(oracle_mod, x3, cb, o, seed=81)
    del o, out
    torch.cuda.empty_cache()

"""Row counts past 2^31, and group offsets past 2^32 elements of x: the sizes at
which any 32-bit row, tile or element offset would wrap.

One group of 2^31 + 4099 fp16 sub-vectors (sub_dim 4, 256 centroids: the
tensor-core kernel, a ragged last tile) is encoded to uint32 indices and to
8-bit codes, and the codes are decoded; three groups of 2^30 + 77 rows are
encoded in one grouped launch, and 2^31 + 4160 rows with per-channel smoothing.
Checks, at full size on the GPU: every output
was written and is a valid index (the output is pre-filled with a value no
index takes), the 8-bit codes equal the uint32 indices, and the decode is the
codebook gather.  Against the oracle: sampled rows, among them the first and
last rows, the rows around 2^31 and 2^30, and the group boundaries.
The sibling encoders run past 2^31 elements as well: the scalar quantize
(both paths, every element checked through the oracle's answer for each of
the 65,536 fp16 bit patterns) with its dequantize, and the Hadamard rotation
with and without the quantize (sampled rows against the oracle).
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



def test_smoothed_encode_past_2_31_rows(vq, oracle_mod, big):
    """Per-channel smoothing fused into the tensor-core encode over 2^31 + 4160
    rows (keys of head_dim 256: the channel of a row comes from its index
    modulo 64).  Every index written and valid; whole sampled keys, among them
    those around row 2^31, against the oracle."""
    x, cb = big
    head_dim = 256
    spk = head_dim // SUB
    m = (1 << 31) + 65 * spk
    x3 = x[:m * SUB].view(1, m, SUB)
    cb1 = cb[:1].contiguous()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(20252)
    smooth = torch.exp(0.5 * torch.randn((1, head_dim), generator=gen, device="cuda"))
    o, out = sentinel_out(1, m)
    vq.vq_encode_grouped_smooth(x3, smooth, cb1, head_dim, index_bytes=4, out=out)
    torch.cuda.synchronize()
    assert_all_valid(o)
    n_keys = m // spk
    rng = np.random.default_rng(91)
    centre = (1 << 31) // spk
    keys = np.unique(np.concatenate([np.arange(0, 30), np.arange(n_keys - 30, n_keys),
                                     np.arange(centre - 30, centre + 30),
                                     rng.integers(0, n_keys, 200)]))
    rows = (keys[:, None] * spk + np.arange(spk)[None, :]).reshape(-1)
    ridx = torch.from_numpy(rows).cuda()
    xs = x3[0].index_select(0, ridx).cpu().numpy()
    want = oracle_mod.encode_smooth(xs[None], smooth.cpu().numpy(), cb1.cpu().numpy(), head_dim,
                                    n_threads=THREADS)[0]
    got = o[0].index_select(0, ridx).cpu().numpy().astype(np.int64)
    bad = np.nonzero(got != want.astype(np.int64))[0]
    assert bad.size == 0, f"{bad.size} sampled rows differ, first row {rows[bad[0]]}"
    del o, out
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- sibling encoders

N_SCALAR = (1 << 31) + 13        # elements: 16-byte units and a ragged tail
HD_DIM, HD_ROWS = 128, (1 << 24) + 3   # 2^31 + 384 rotated elements


@pytest.fixture(scope="module")
def centroids16():
    # sorted, as a Lloyd-Max codebook for N(0, 1) would be
    return torch.linspace(-2.4, 2.4, 16, dtype=torch.float32, device="cuda")


def fp16_normal(n: int, seed: int) -> torch.Tensor:
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    x = torch.empty(n, dtype=torch.float16, device="cuda")
    for a in range(0, n, CHUNK * SUB):
        x[a:a + CHUNK * SUB].normal_(generator=gen)
    return x


def test_scalar_quantize_past_2_31_elements(vq, oracle_mod, centroids16):
    """The fp16 scalar quantize (16 centroids: the bucket-table kernel, with
    and without a workspace) and the dequantize.  A 16-bit key's index
    depends on its bit pattern alone, so the oracle's answer for all 65,536
    patterns checks every element."""
    x = fp16_normal(N_SCALAR, 901)
    c = centroids16
    pats = np.arange(1 << 16, dtype=np.uint16).view(np.float16)
    table = torch.from_numpy(oracle_mod.scalar_quantize(pats, c.cpu().numpy()).astype(np.uint8)).cuda()
    bits = x.view(torch.int16)
    got_t = vq.vq_scalar_quantize(x, c)
    got_s = vq.vq_scalar_quantize(x, c, use_table=False)
    torch.cuda.synchronize()
    for a in range(0, N_SCALAR, CHUNK):
        want = table[bits[a:a + CHUNK].to(torch.int64) & 0xFFFF]
        assert torch.equal(got_t[a:a + CHUNK], want), a
        assert torch.equal(got_s[a:a + CHUNK], want), a
    del got_s
    dq = vq.vq_scalar_dequantize(got_t, c, dtype=torch.float16)
    torch.cuda.synchronize()
    c16 = c.to(torch.float16)
    for a in range(0, N_SCALAR, CHUNK):
        assert torch.equal(dq[a:a + CHUNK], c16[got_t[a:a + CHUNK].long()]), a
    del x, got_t, dq
    torch.cuda.empty_cache()


def test_hadamard_past_2_31_elements(vq, oracle_mod, centroids16):
    """Rotation and rotation + quantize over 2^24 + 3 rows of 128: sampled
    rows against the oracle (bit for bit), every code valid."""
    x = fp16_normal(HD_ROWS * HD_DIM, 902).view(HD_ROWS, HD_DIM)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(903)
    diag = (torch.randint(0, 2, (HD_DIM,), generator=gen, device="cuda") * 2 - 1).to(torch.float32)
    c = centroids16
    codes = vq.vq_hadamard_quantize(x, diag, c)
    torch.cuda.synchronize()
    flat = codes.view(-1)
    for a in range(0, flat.numel(), CHUNK):
        assert int(flat[a:a + CHUNK].max()) < c.numel(), a
    rows = torch.from_numpy(sample_rows(HD_ROWS, 904)).cuda()
    xs = x.index_select(0, rows).cpu().numpy()
    want = oracle_mod.hadamard_quantize(xs, diag.cpu().numpy(), c.cpu().numpy())
    got = codes.index_select(0, rows).cpu().numpy()
    assert np.array_equal(got.astype(np.uint32), want)
    del codes, flat
    y = vq.vq_hadamard_rotate(x, diag)
    torch.cuda.synchronize()
    want_y = oracle_mod.hadamard_rotate(xs, diag.cpu().numpy())
    got_y = y.index_select(0, rows).cpu().numpy()
    assert np.array_equal(got_y.view(np.uint32), want_y.view(np.uint32))
    del x, y
    torch.cuda.empty_cache()

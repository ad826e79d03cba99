"""GPU parity of the sibling encoders: scalar (sub_dim = 1) quantize and
dequantize, and the randomised Hadamard rotation with its fused quantize.
Indices and rotated values are compared bit for bit with the oracle."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


def to_dev(x, dtype):
    """(host array the oracle takes, its bf16 flag, device tensor)."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16), True, t.cuda()
    a = np.ascontiguousarray(x, dtype=np.float16 if dtype == "f16" else np.float32)
    return a, False, torch.from_numpy(a).cuda()


def codebook(rng, n_c):
    c = rng.standard_normal(n_c).astype(np.float32)
    if n_c > 2:
        c[n_c // 2] = c[1]  # a duplicate: ties go to the lower index
    return c


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("n_c", [2, 16, 256])
def test_scalar_every_16_bit_pattern(vq, oracle_mod, dtype, n_c):
    """All 65,536 bit patterns (NaN, inf, subnormals included), table and
    scan (fp16 with 2 or 16 centroids: the bucket table either way)."""
    rng = np.random.default_rng(n_c)
    c = codebook(rng, n_c)
    bits = np.arange(65536, dtype=np.uint16)
    if dtype == "f16":
        host, bf, dev = bits.view(np.float16), False, torch.from_numpy(bits.view(np.int16)).cuda().view(torch.float16)
    else:
        host, bf, dev = bits, True, torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    want = oracle_mod.scalar_quantize(host, c, bf16=bf)
    cd = torch.from_numpy(c).cuda()
    for use_table in (True, False):
        got = vq.vq_scalar_quantize(dev, cd, use_table=use_table).cpu().numpy()
        assert np.array_equal(got.astype(np.uint32), want), use_table


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("n", [0, 1, 7, 8, 4099, 1 << 20])
def test_scalar_sizes_and_alignment(vq, oracle_mod, dtype, n):
    rng = np.random.default_rng(n + 3)
    c = codebook(rng, 16)
    x = 2.0 * rng.standard_normal(n + 3)
    x[: min(3, n)] = [np.inf, -np.nan, 1e-7][: min(3, n)]
    host, bf, dev = to_dev(x, dtype)
    cd = torch.from_numpy(c).cuda()
    for off in (0, 1, 3):  # unaligned starts take the element-wise path
        want = oracle_mod.scalar_quantize(host[off:off + n], c, bf16=bf)
        got = vq.vq_scalar_quantize(dev[off:off + n], cd).cpu().numpy()
        assert np.array_equal(got.astype(np.uint32), want)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_scalar_dequantize(vq, dtype):
    rng = np.random.default_rng(7)
    c = (3 * rng.standard_normal(16)).astype(np.float32)
    idx = rng.integers(0, 20, 10001).astype(np.uint8)  # 16..19 are out of range
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    got = vq.vq_scalar_dequantize(torch.from_numpy(idx).cuda(), torch.from_numpy(c).cuda(),
                                  dtype=tdt).cpu()
    padded = np.concatenate([c, np.zeros(256 - 16, dtype=np.float32)])
    want = torch.from_numpy(padded[idx]).to(tdt)  # round to nearest
    assert torch.equal(got, want)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("dim", [1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024])
def test_hadamard_rotate_bit_exact(vq, oracle_mod, dtype, dim):
    rng = np.random.default_rng(dim)
    rows = 1001 if dim <= 256 else 97
    host, bf, dev = to_dev(rng.standard_normal((rows, dim)), dtype)
    diag = rng.choice([-1.0, 1.0], dim).astype(np.float32)
    diag[0] = 0.75  # any fp32 factor, not only signs
    want = oracle_mod.hadamard_rotate(host, diag, bf16=bf)
    got = vq.vq_hadamard_rotate(dev, torch.from_numpy(diag).cuda()).cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("dim,n_c", [(4, 2), (32, 16), (128, 16), (128, 256), (256, 4), (1024, 16)])
def test_hadamard_quantize_bit_exact(vq, oracle_mod, dtype, dim, n_c):
    rng = np.random.default_rng(dim * 1000 + n_c)
    rows = 777 if dim <= 256 else 65
    host, bf, dev = to_dev(rng.standard_normal((rows, dim)), dtype)
    diag = rng.choice([-1.0, 1.0], dim).astype(np.float32)
    c = np.sort(codebook(rng, n_c))
    want = oracle_mod.hadamard_quantize(host, diag, c, bf16=bf)
    got = vq.vq_hadamard_quantize(dev, torch.from_numpy(diag).cuda(),
                                  torch.from_numpy(c).cuda()).cpu().numpy()
    assert np.array_equal(got.astype(np.uint32), want)


def test_full_turboquant_keys(vq, oracle_mod):
    """The benchmarked cache (8 heads x 32768 tokens x 128, 4-bit codebook):
    every index of the scalar and of the fused Hadamard quantize."""
    x, c, diag = workloads.generate_scalar("turboquant_keys")
    xd, cd, dd = (torch.from_numpy(a).cuda() for a in (x, c, diag))
    got = vq.vq_scalar_quantize(xd, cd).cpu().numpy()
    assert np.array_equal(got.astype(np.uint32), oracle_mod.scalar_quantize(x, c))
    got = vq.vq_hadamard_quantize(xd, dd, cd).cpu().numpy()
    assert np.array_equal(got.astype(np.uint32), oracle_mod.hadamard_quantize(x, diag, c))


@pytest.mark.parametrize("case", ["unsorted_duplicates", "plateaus", "signed_zeros", "non_finite",
                                  "one_centroid", "all_equal", "wide_256"])
def test_hadamard_quantize_codebook_edge_cases(vq, oracle_mod, case):
    """The sorted-codebook search against the rule: duplicates in any order,
    centroids whose fp32 distances tie for large keys, +-0, an infinite
    centroid (the kernel falls back to the scan), degenerate codebooks."""
    rng = np.random.default_rng(sum(map(ord, case)))
    dim, rows = 128, 300
    x = rng.standard_normal((rows, dim)).astype(np.float32)
    if case == "unsorted_duplicates":
        c = rng.standard_normal(16).astype(np.float32)
        c[[3, 9, 14]] = c[5]
        c[[0, 11]] = c[7]
    elif case == "plateaus":
        base = np.float32(1.0)
        c = (base + np.arange(16, dtype=np.float32) * np.float32(2.0 ** -22)).astype(np.float32)
        rng.shuffle(c)
        x *= np.float32(1e4)  # |y - c| ~ 1e3: the ulp of y swamps the centroid gaps
    elif case == "signed_zeros":
        c = np.array([0.0, -0.0, 1.0, -1.0, -0.0, 0.5, 0.0, -0.5], dtype=np.float32)
        x[:, :16] = 0.0
    elif case == "non_finite":
        c = rng.standard_normal(8).astype(np.float32)
        c[2] = np.inf
    elif case == "one_centroid":
        c = np.array([0.25], dtype=np.float32)
    elif case == "all_equal":
        c = np.full(16, 0.75, dtype=np.float32)
    else:
        c = rng.standard_normal(256).astype(np.float32)
        c[rng.integers(0, 256, 40)] = c[rng.integers(0, 256, 40)]
    diag = rng.choice([-1.0, 1.0], dim).astype(np.float32)
    want = oracle_mod.hadamard_quantize(x, diag, c)
    got = vq.vq_hadamard_quantize(torch.from_numpy(x).cuda(), torch.from_numpy(diag).cuda(),
                                  torch.from_numpy(c).cuda()).cpu().numpy()
    assert np.array_equal(got.astype(np.uint32), want)


@pytest.mark.parametrize("n_c", [1, 2, 3, 8, 16, 100, 256])
@pytest.mark.parametrize("kind", ["random", "duplicates", "non_finite"])
def test_scalar_scan_paths(vq, oracle_mod, n_c, kind):
    """fp32 keys (no table): the register scan (2, 4, 8, 16 entries) and the
    sorted-view search (other sizes, with its fallback) against the rule."""
    rng = np.random.default_rng(n_c * 7 + len(kind))
    x = (3.0 * rng.standard_normal(50001)).astype(np.float32)
    x[:6] = [np.nan, np.inf, -np.inf, 0.0, -0.0, 3e38]
    c = rng.standard_normal(n_c).astype(np.float32)
    if kind == "duplicates" and n_c > 2:
        c[rng.integers(0, n_c, n_c // 2)] = c[0]
    if kind == "non_finite":
        c[n_c // 2] = np.inf
    got = vq.vq_scalar_quantize(torch.from_numpy(x).cuda(), torch.from_numpy(c).cuda()).cpu().numpy()
    assert np.array_equal(got.astype(np.uint32), oracle_mod.scalar_quantize(x, c))


def value_sweep_keys(seed: int) -> np.ndarray:
    """Every fp32 value whose low 16 bits are all 0, all 1 or random: every
    sign, exponent and top-7-bit mantissa prefix at both ends and inside,
    NaN, inf and subnormals included."""
    rng = np.random.default_rng(seed)
    top = np.arange(65536, dtype=np.uint32) << 16
    low = rng.integers(0, 65536, 65536, dtype=np.uint32)
    return np.concatenate([top, top | 0xFFFF, top | low]).view(np.float32)


@pytest.mark.parametrize("case", ["normal_3", "normal_5", "normal_100", "normal_256", "scaled_tiny",
                                  "scaled_huge", "negative_only", "close_pairs", "duplicates",
                                  "subnormal", "powers_of_two"])
def test_scalar_scan_value_sweep(vq, oracle_mod, case):
    """fp32 keys over the whole float range against the rule, for codebooks
    of several sizes, scales and shapes (register scan and sorted-view search
    with its fallback)."""
    rng = np.random.default_rng(sum(map(ord, case)))
    if case.startswith("normal_"):
        c = rng.standard_normal(int(case.split("_")[1])).astype(np.float32)
    elif case == "scaled_tiny":
        c = (rng.standard_normal(12) * 1e-30).astype(np.float32)
    elif case == "scaled_huge":
        c = (rng.standard_normal(12) * 1e30).astype(np.float32)
    elif case == "negative_only":
        c = -np.abs(rng.standard_normal(9)).astype(np.float32) - 1.0
    elif case == "close_pairs":  # centroids closer than 2^-10 relative
        base = rng.standard_normal(6).astype(np.float32)
        c = np.concatenate([base, base * np.float32(1 + 2 ** -12), base * np.float32(1 - 2 ** -10)])
    elif case == "duplicates":
        c = rng.standard_normal(20).astype(np.float32)
        c[[2, 7, 11]] = c[15]
        c[[0, 19]] = c[4]
    elif case == "subnormal":
        c = np.array([1e-45, -3e-45, 2e-40, 0.0, -1e-39, 5e-42], dtype=np.float32)
    else:
        c = np.float32(2.0) ** np.arange(-8, 9, 2, dtype=np.float32)
        c = np.concatenate([c, -c])
    x = value_sweep_keys(len(case))
    got = vq.vq_scalar_quantize(torch.from_numpy(x).cuda(), torch.from_numpy(c).cuda()).cpu().numpy()
    assert np.array_equal(got.astype(np.uint32), oracle_mod.scalar_quantize(x, c))


@pytest.mark.parametrize("n_c", [8, 16, 256])
def test_hadamard_quantize_value_sweep(vq, oracle_mod, n_c):
    """The fused quantize on rotated rows spread over the float range: the
    rotation (diag = 1) maps v * sqrt(D) * e_0 to the constant row v, plus a
    little noise from the other columns."""
    rng = np.random.default_rng(n_c)
    c = np.sort(rng.standard_normal(n_c).astype(np.float32))
    dim = 32
    vals = value_sweep_keys(n_c)
    vals = vals[np.isfinite(vals) & (np.abs(vals) < 1e30)]
    x = np.zeros((vals.size, dim), dtype=np.float32)
    x[:, 0] = vals * np.float32(np.sqrt(dim))  # y = H e_0 * v: every element equal to v (up to rounding)
    x[:, 1:] = rng.standard_normal((vals.size, dim - 1)).astype(np.float32) * np.float32(1e-3)
    diag = np.ones(dim, dtype=np.float32)
    want = oracle_mod.hadamard_quantize(x, diag, c)
    got = vq.vq_hadamard_quantize(torch.from_numpy(x).cuda(), torch.from_numpy(diag).cuda(),
                                  torch.from_numpy(c).cuda()).cpu().numpy()
    assert np.array_equal(got.astype(np.uint32), want)


@pytest.mark.parametrize("n_c", [4, 16, 100])
@pytest.mark.parametrize("dim", [32, 64, 128])
def test_hadamard_both_lane_layouts(vq, oracle_mod, n_c, dim):
    """The same rows through the wide lane layout (x 16-byte aligned) and the
    contract's minimal one (x aligned to dim/32 elements only, here 8 bytes
    off a 16-byte boundary): both bit-identical to the oracle."""
    rng = np.random.default_rng(dim + n_c)
    rows = 999
    x = rng.standard_normal((rows, dim)).astype(np.float16)
    diag = rng.choice([-1.0, 1.0], dim).astype(np.float32)
    c = np.sort(rng.standard_normal(n_c).astype(np.float32))
    want = oracle_mod.hadamard_quantize(x, diag, c)
    want_rot = oracle_mod.hadamard_rotate(x, diag)
    dd, cd = torch.from_numpy(diag).cuda(), torch.from_numpy(c).cuda()
    buf = torch.zeros(rows * dim + 64, dtype=torch.float16, device="cuda")
    for off in (0, 4):  # elements: 16-byte aligned, then 8 bytes past
        xv = buf[off:off + rows * dim].view(rows, dim)
        xv.copy_(torch.from_numpy(x))
        got = vq.vq_hadamard_quantize(xv, dd, cd).cpu().numpy()
        assert np.array_equal(got.astype(np.uint32), want), off
        rot = vq.vq_hadamard_rotate(xv, dd).cpu().numpy()
        assert np.array_equal(rot.view(np.uint32), want_rot.view(np.uint32)), off


def cut_point_codebooks(n_c):
    """Codebooks of 2 to 16 entries for the cut-point path: exact fp32 ties
    at every midpoint (dyadic values) in sorted, reversed and shuffled
    original order (both tie-break directions), random normal ones sorted and
    not, and gap ratios just inside and just outside the set-up's 2^15 limit
    (the latter take the rule's scan)."""
    rng = np.random.default_rng(300 + n_c)
    dyadic = (np.arange(n_c, dtype=np.float32) * np.float32(0.5) - np.float32(1.0)).astype(np.float32)
    out = {"dyadic_sorted": dyadic, "dyadic_reversed": dyadic[::-1].copy()}
    shuffled = dyadic.copy()
    rng.shuffle(shuffled)
    out["dyadic_shuffled"] = shuffled
    normal = rng.standard_normal(n_c).astype(np.float32)
    out["normal_sorted"] = np.sort(normal)
    out["normal_unsorted"] = normal
    if n_c >= 4:
        for name, ratio in (("gap_ratio_inside", 2.0 ** 14), ("gap_ratio_outside", 2.0 ** 17)):
            gaps = np.ones(n_c - 1)
            gaps[n_c // 2] = 1.0 / ratio  # one narrow gap beside wide ones
            out[name] = np.concatenate([[0.0], np.cumsum(gaps)]).astype(np.float32)
    return out


def cut_point_keys(c):
    """Keys within 300 ulps of every exact midpoint of neighbouring centroids
    and of the ends of the range the cut points decide (32768 outer gaps
    beyond the extreme centroids), plus the whole-range value sweep."""
    s = np.unique(c.astype(np.float64))
    marks = list((s[:-1] + s[1:]) / 2)
    if s.size > 1:
        marks += [s[0] - 32768 * (s[1] - s[0]), s[-1] + 32768 * (s[-1] - s[-2])]
    keys = []
    for m in marks:
        m32 = np.float32(m)
        bits = np.int64(m32.view(np.int32))
        around = (bits + np.arange(-300, 301)).astype(np.int64)
        around = around[(around >= -(2 ** 31)) & (around < 2 ** 31)].astype(np.int32)
        keys.append(around.view(np.float32))
    keys.append(value_sweep_keys(len(c)))
    return np.concatenate(keys).astype(np.float32)


@pytest.mark.parametrize("n_c", [2, 4, 8, 16])
def test_cut_points_match_the_rule_where_they_decide(vq, oracle_mod, n_c):
    """The 2- to 16-entry quantize (cut points counted by a binary search,
    the rule's scan where they cannot decide) against the rule, for fp32
    keys (scalar quantize) and for rotated rows (Hadamard quantize, a
    constant row per key: diag 1 maps v * sqrt(D) e_0 to v in every column)."""
    for name, c in cut_point_codebooks(n_c).items():
        x = cut_point_keys(c)
        cd = torch.from_numpy(c).cuda()
        got = vq.vq_scalar_quantize(torch.from_numpy(x).cuda(), cd).cpu().numpy()
        want = oracle_mod.scalar_quantize(x, c)
        bad = np.flatnonzero(got.astype(np.uint32) != want)
        assert bad.size == 0, f"{name}: {bad.size} keys differ, first {x[bad[:4]]}"
        dim = 32
        fin = x[np.isfinite(x) & (np.abs(x) < 1e30)]
        rows = np.zeros((fin.size, dim), dtype=np.float32)
        rows[:, 0] = fin * np.float32(np.sqrt(dim))
        diag = np.ones(dim, dtype=np.float32)
        got = vq.vq_hadamard_quantize(torch.from_numpy(rows).cuda(), torch.from_numpy(diag).cuda(),
                                      cd).cpu().numpy()
        assert np.array_equal(got.astype(np.uint32), oracle_mod.hadamard_quantize(rows, diag, c)), name


def bucket_codebooks(n_c):
    """Codebooks for fp16 keys against 2 to 16 centroids (the bucket table):
    the cut-point codebooks, the benchmark's Lloyd-Max levels, centroids
    closer than a bucket is wide (several code changes in one bucket), a
    decided range that ends inside the fp16 range, tiny centroids (most
    patterns outside it), and codebooks that fail the cut points' conditions
    (a repeated value, an infinity: every bucket flagged)."""
    rng = np.random.default_rng(500 + n_c)
    out = dict(cut_point_codebooks(n_c))
    lm = workloads.lloyd_max_gaussian(int(np.log2(n_c)), 20)
    out["lloyd_max"] = lm
    out["closer_than_a_bucket"] = (np.float32(1.0) + np.arange(n_c, dtype=np.float32) * np.float32(0.0015)).astype(np.float32)
    out["range_inside_fp16"] = (np.arange(n_c, dtype=np.float32) * np.float32(0.01)).astype(np.float32)
    out["tiny"] = (rng.standard_normal(n_c) * 1e-6).astype(np.float32)
    dup = lm.copy()
    dup[-1] = dup[0]
    out["repeated"] = dup
    inf = lm.copy()
    inf[n_c // 2] = np.inf
    out["infinite"] = inf
    return out


@pytest.mark.parametrize("n_c", [2, 4, 8, 16])
def test_fp16_bucket_table_every_pattern(vq, oracle_mod, n_c):
    """fp16 keys against 2 to 16 centroids go through the per-block bucket
    table (one entry per top-10-bit prefix, flagged buckets element by
    element): all 65,536 patterns against the rule, for every codebook of
    bucket_codebooks, 16-byte aligned (8-element units) and one element off
    (element by element)."""
    bits = np.arange(65536, dtype=np.uint16)
    host = bits.view(np.float16)
    buf = torch.zeros(65536 + 16, dtype=torch.int16, device="cuda")
    for name, c in bucket_codebooks(n_c).items():
        want = oracle_mod.scalar_quantize(host, c)
        cd = torch.from_numpy(c).cuda()
        for off in (0, 1):
            xv = buf[off:off + 65536]
            xv.copy_(torch.from_numpy(bits.view(np.int16)))
            got = vq.vq_scalar_quantize(xv.view(torch.float16), cd).cpu().numpy()
            bad = np.flatnonzero(got.astype(np.uint32) != want)
            assert bad.size == 0, f"{name} off {off}: {bad.size} patterns differ, first {bits[bad[:4]]}"

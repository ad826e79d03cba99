"""Pins for the CPU oracle (no GPU needed).

The oracle is checked against things other than itself: library decoders for
the number formats, hand-derived rounding cases, exact integer arithmetic,
float64 brute force within a proven fp32 error bound, the boundary-count rule
that the sub_dim = 1 case reduces to, and invariants of the encoding (exact
copies, duplicate rows, permutations, chunking, grouping, special values).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import parse_pow2_sum, read_golden

U32 = 2.0 ** -24  # unit round-off of fp32


# ---------------------------------------------------------------- formats

def test_f16_decode_matches_numpy_for_every_bit_pattern(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle_mod.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_bf16_decode_matches_torch_for_every_bit_pattern(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([oracle_mod.bf16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


# ---------------------------------------------------------------- distance

@pytest.mark.parametrize("row", read_golden("distance_rounding.txt"), ids=lambda r: r[0])
def test_distance_golden_rounding(oracle_mod, row):
    _, xs, cs, bits, _ = row
    x = np.array([float(parse_pow2_sum(v)) for v in xs.split(",")], dtype=np.float32)
    c = np.array([float(parse_pow2_sum(v)) for v in cs.split(",")], dtype=np.float32)
    got = oracle_mod.distance(x, c)
    assert int(np.array([got], dtype=np.float32).view(np.uint32)[0]) == int(bits, 16)


def test_distance_exact_on_small_integers(oracle_mod):
    rng = np.random.default_rng(100)
    for sub_dim in (1, 3, 4, 8, 16):
        for _ in range(50):
            x = rng.integers(-40, 41, sub_dim)
            c = rng.integers(-40, 41, sub_dim)
            want = int(((x - c) ** 2).sum())
            for dt in (np.float16, np.float32):
                assert oracle_mod.distance(x.astype(dt), c.astype(dt)) == want


def test_distance_within_fp32_error_bound_of_exact(oracle_mod):
    """|D32 - D| <= ((1+u)^(s+2) - 1) D, D computed exactly with rationals."""
    rng = np.random.default_rng(101)
    for sub_dim in (2, 4, 8):
        bound = (1 + U32) ** (sub_dim + 2) - 1
        for _ in range(200):
            x = rng.standard_normal(sub_dim).astype(np.float16)
            c = rng.standard_normal(sub_dim).astype(np.float16)
            exact = sum((Fraction(float(a)) - Fraction(float(b))) ** 2 for a, b in zip(x, c))
            got = Fraction(float(oracle_mod.distance(x, c)))
            assert abs(got - exact) <= Fraction(bound) * exact


# ---------------------------------------------------------------- encode

def _d64(x, cb):
    x = x.astype(np.float64)
    cb = cb.astype(np.float64)
    return ((x[:, None, :] - cb[None, :, :]) ** 2).sum(-1)


def test_encode_exact_integers_with_ties(oracle_mod):
    """Small integers: every fp32 step is exact, so the encoding must equal the
    first minimiser of the exact integer distances (np.argmin keeps the first)."""
    rng = np.random.default_rng(102)
    for sub_dim, n_c in ((4, 64), (8, 256), (1, 9), (3, 17)):
        x = rng.integers(-4, 5, (500, sub_dim))
        cb = rng.integers(-4, 5, (n_c, sub_dim))
        want = np.argmin(((x[:, None, :] - cb[None]) ** 2).sum(-1), axis=1)
        for dt in (np.float16, np.float32):
            got = oracle_mod.encode(x.astype(dt), cb.astype(dt))
            assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("sub_dim", [4, 8])
def test_encode_brute_force_float64(oracle_mod, dtype, sub_dim):
    """Where float64 separates the best centroid from the runner-up by more
    than the fp32 error bound, the oracle must pick it; elsewhere its pick
    must lie within the bound of the float64 minimum."""
    rng = np.random.default_rng(103 + sub_dim)
    n, n_c = 3000, 256
    xf = rng.standard_normal((n, sub_dim)).astype(np.float32)
    cf = rng.standard_normal((n_c, sub_dim)).astype(np.float32)
    if dtype == "f16":
        x, cb, kw = xf.astype(np.float16), cf.astype(np.float16), {}
        xv, cv = x, cb
    elif dtype == "bf16":
        xb = torch.from_numpy(xf).to(torch.bfloat16)
        cbt = torch.from_numpy(cf).to(torch.bfloat16)
        x = xb.view(torch.int16).numpy().view(np.uint16)
        cb = cbt.view(torch.int16).numpy().view(np.uint16)
        xv, cv, kw = xb.float().numpy(), cbt.float().numpy(), {"bf16": True}
    else:
        x, cb, kw = xf, cf, {}
        xv, cv = xf, cf
    got = oracle_mod.encode(x, cb, **kw)
    d = _d64(xv, cv)
    e = (1 + U32) ** (sub_dim + 2) - 1 + (sub_dim + 2) * 2.0 ** -52
    order = np.argsort(d, axis=1, kind="stable")
    best, second = d[np.arange(n), order[:, 0]], d[np.arange(n), order[:, 1]]
    separated = second * (1 - e) > best * (1 + e)
    assert separated.mean() > 0.95
    assert np.array_equal(got[separated], order[separated, 0])
    picked = d[np.arange(n), got]
    assert np.all(picked <= best * (1 + e) / (1 - e))


def test_exact_copies_map_to_first_equal_row(oracle_mod):
    rng = np.random.default_rng(104)
    cb = rng.standard_normal((256, 8)).astype(np.float16)
    cb[200] = cb[3]      # duplicate above its source
    cb[7] = cb[150]      # duplicate below its source
    cb[9] = -0.0         # rows equal by value: +0 and -0
    cb[11] = 0.0
    src = rng.integers(0, 256, 2000)
    x = cb[src].copy()
    got = oracle_mod.encode(x, cb)
    first_equal = np.array([np.flatnonzero((cb == cb[s]).all(1))[0] for s in src])
    assert np.array_equal(got, first_equal)
    assert got[src == 200].size == 0 or np.all(got[src == 200] == 3)
    assert np.all(got[src == 150] == 7)
    assert np.all(got[src == 11] == 9)


def test_duplicated_rows_resolve_to_lower_index(oracle_mod):
    rng = np.random.default_rng(105)
    x = rng.standard_normal((4000, 4)).astype(np.float16)
    cb = rng.standard_normal((64, 4)).astype(np.float16)
    base = oracle_mod.encode(x, cb)
    dup = np.concatenate([cb, cb])  # rows 64..127 repeat rows 0..63
    assert np.array_equal(oracle_mod.encode(x, dup), base)
    dup_front = np.concatenate([cb[::-1], cb])  # the copy of row r sits at 63-r
    assert np.array_equal(oracle_mod.encode(x, dup_front), 63 - base)


def test_single_centroid_encodes_everything_to_zero(oracle_mod):
    rng = np.random.default_rng(106)
    x = rng.standard_normal((777, 4)).astype(np.float16)
    cb = rng.standard_normal((1, 4)).astype(np.float16)
    assert np.array_equal(oracle_mod.encode(x, cb), np.zeros(777, np.uint32))


def test_sub_dim_one_reduces_to_boundary_count(oracle_mod):
    """With sub_dim = 1 and a sorted codebook, the nearest centroid's index is
    the number of midpoints between neighbouring centroids that x exceeds."""
    rng = np.random.default_rng(107)
    cb = np.unique(rng.standard_normal(64).astype(np.float16))
    mids = (cb[:-1].astype(np.float64) + cb[1:].astype(np.float64)) / 2
    x = rng.standard_normal(20000).astype(np.float16)
    gap = np.abs(x.astype(np.float64)[:, None] - mids[None]).min(1)
    x = x[gap > 1e-3 * (1 + np.abs(x.astype(np.float64)))]
    want = (x.astype(np.float64)[:, None] > mids[None]).sum(1)
    got = oracle_mod.encode(x[:, None], cb[:, None])
    assert np.array_equal(got, want)


def test_permuting_codebook_rows_permutes_indices(oracle_mod):
    rng = np.random.default_rng(108)
    x = rng.standard_normal((5000, 4)).astype(np.float16)
    cb = rng.standard_normal((256, 4)).astype(np.float16)
    perm = rng.permutation(256)
    inv = np.argsort(perm)
    assert np.array_equal(oracle_mod.encode(x, cb[perm]), inv[oracle_mod.encode(x, cb)])


def test_chunking_grouping_and_threads_do_not_change_results(oracle_mod):
    rng = np.random.default_rng(109)
    x = rng.standard_normal((4, 1001, 8)).astype(np.float16)
    cb = rng.standard_normal((4, 256, 8)).astype(np.float16)
    grouped = oracle_mod.encode(x, cb)
    for g in range(4):
        assert np.array_equal(grouped[g], oracle_mod.encode(x[g], cb[g]))
        assert np.array_equal(grouped[g, 100:433], oracle_mod.encode(x[g, 100:433], cb[g]))
    assert np.array_equal(grouped, oracle_mod.encode(x, cb, n_threads=7))


def test_special_values(oracle_mod):
    cb = np.array([[np.nan, 0, 0, 0], [1, 1, 1, 1], [2, 2, 2, 2], [np.inf, 0, 0, 0],
                   [1, 1, 1, 1]], dtype=np.float16)
    x = np.array([
        [1, 1, 1, 1],          # exact copy of row 1 (row 4 is its duplicate)
        [np.nan, 1, 1, 1],     # every distance NaN -> 0
        [np.inf, 1, 1, 1],     # inf or NaN everywhere -> 0
        [2.1, 2, 2, 2],        # nearest is row 2; NaN row 0 never wins
        [-np.inf, 0, 0, 0],    # inf distances, NaN against row 3 -> 0
        [60000, 0, 0, 0],      # large but finite: picks row 2 (distance still finite)
    ], dtype=np.float16)
    got = oracle_mod.encode(x, cb)
    assert got.tolist() == [1, 0, 0, 2, 0, 2]
    # fp32 overflow of a single square gives +inf for every centroid -> 0
    x32 = np.array([[3e38, 0, 0, 0]], dtype=np.float32)
    cb32 = np.array([[-3e38, 0, 0, 0], [-1e38, 0, 0, 0]], dtype=np.float32)
    assert oracle_mod.encode(x32, cb32).tolist() == [0]
    # huge but finite distances (~1e32) must still compete: the start value is +inf
    x32 = np.array([[1e16, 0, 0, 0]], dtype=np.float32)
    cb32 = np.array([[0, 0, 0, 0], [1e15, 0, 0, 0], [3e15, 0, 0, 0]], dtype=np.float32)
    assert oracle_mod.encode(x32, cb32).tolist() == [2]


def test_empty_input(oracle_mod):
    x = np.zeros((0, 4), np.float16)
    cb = np.zeros((256, 4), np.float16)
    assert oracle_mod.encode(x, cb).shape == (0,)
    assert oracle_mod.encode(np.zeros((3, 0, 8), np.float16),
                             np.zeros((3, 256, 8), np.float16)).shape == (3, 0)


# ---------------------------------------------------------------- decode

def test_dequantize_identity_permutation_and_range(oracle_mod):
    rng = np.random.default_rng(110)
    cb = rng.standard_normal((3, 256, 8)).astype(np.float16)
    ar = np.tile(np.arange(256, dtype=np.uint32), (3, 1))
    assert np.array_equal(oracle_mod.dequantize(ar, cb), cb)
    perm = rng.permutation(256).astype(np.uint32)
    got = oracle_mod.dequantize(np.tile(perm, (3, 1)), cb)
    assert np.array_equal(got, cb[:, perm])
    bad = np.array([[0, 255, 256, 1000, 0xFFFFFFFF]], dtype=np.uint32)
    got = oracle_mod.dequantize(bad, cb[:1])
    assert np.array_equal(got[0, :2], cb[0, [0, 255]])
    assert not got[0, 2:].any()


def test_encode_then_dequantize_round_trips_exact_copies(oracle_mod):
    """Rows that are exact codebook copies come back unchanged; every other
    row comes back as its nearest centroid (no centroid is strictly closer)."""
    rng = np.random.default_rng(111)
    cb = rng.standard_normal((2, 256, 4)).astype(np.float16)
    x = rng.standard_normal((2, 3000, 4)).astype(np.float16)
    x[:, :500] = cb[:, rng.integers(0, 256, 500)]
    rec = oracle_mod.dequantize(oracle_mod.encode(x, cb), cb)
    assert np.array_equal(rec[:, :500], x[:, :500])
    d_rec = ((rec.astype(np.float64) - x) ** 2).sum(-1)
    d_all = ((x.astype(np.float64)[:, :, None, :] - cb[:, None, :, :]) ** 2).sum(-1)
    assert np.all(d_rec <= d_all.min(-1) * (1 + 1e-6) + 1e-12)


# ---------------------------------------------------------------- smoothing

def _smooth_case(seed, groups=3, per_group=96, sub_dim=4, head_dim=16, n_c=64, dtype=np.float16):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((groups, per_group, sub_dim)).astype(dtype)
    cb = rng.standard_normal((groups, n_c, sub_dim)).astype(dtype)
    smooth = np.exp(0.5 * rng.standard_normal((groups, head_dim))).astype(np.float32)
    return x, cb, smooth


def test_smooth_ones_is_the_plain_encode(oracle_mod):
    x, cb, _ = _smooth_case(120)
    ones = np.ones((3, 16), dtype=np.float32)
    assert np.array_equal(oracle_mod.encode_smooth(x, ones, cb, 16), oracle_mod.encode(x, cb))


def test_smooth_equals_encoding_numpy_divided_rows(oracle_mod):
    """Division by the channel's factor in IEEE fp32 (numpy's own division),
    channel (m % (head_dim / sub_dim)) * sub_dim + i of group g, then the plain
    encode on the fp32 rows: bit-identical indices."""
    for seed, sub_dim, head_dim in ((121, 4, 16), (122, 8, 128), (123, 4, 256)):
        x, cb, smooth = _smooth_case(seed, sub_dim=sub_dim, head_dim=head_dim,
                                     per_group=3 * head_dim // sub_dim)
        g, m, _ = x.shape
        ns = head_dim // sub_dim
        blocks = smooth.reshape(g, ns, sub_dim)[:, np.arange(m) % ns, :]  # [G, M, sub]
        xs = x.astype(np.float32) / blocks
        want = oracle_mod.encode(xs, cb.astype(np.float32))
        assert np.array_equal(oracle_mod.encode_smooth(x, smooth, cb, head_dim), want)


def test_smooth_by_powers_of_two_scales_the_codebook(oracle_mod):
    """A factor 2^k on every channel scales every distance by 4^-k exactly, so
    the indices equal those of the codebook scaled by 2^k."""
    x, cb, _ = _smooth_case(124, dtype=np.float32)
    for k in (-3, 1, 5):
        s = np.full((3, 16), 2.0 ** k, dtype=np.float32)
        assert np.array_equal(oracle_mod.encode_smooth(x, s, cb, 16),
                              oracle_mod.encode(x, (cb * np.float32(2.0 ** k)).astype(np.float32)))


def test_smooth_factors_are_per_group(oracle_mod):
    """Groups use their own factor rows: group 1 with group 0's factors gives
    other indices."""
    x, cb, smooth = _smooth_case(125)
    base = oracle_mod.encode_smooth(x, smooth, cb, 16)
    swapped = smooth.copy()
    swapped[1] = smooth[0]
    other = oracle_mod.encode_smooth(x, swapped, cb, 16)
    assert np.array_equal(base[0], other[0]) and np.array_equal(base[2], other[2])
    assert not np.array_equal(base[1], other[1])


def test_smooth_rejects_partial_key_vectors(oracle_mod):
    x, cb, smooth = _smooth_case(126, per_group=10)  # 10 rows, 4 per key vector
    with pytest.raises(RuntimeError):
        oracle_mod.encode_smooth(x, smooth, cb, 16)


# ---------------------------------------------------------------- fp16 arithmetic vs the rule

def test_fp16_subtract_variant_differs_rarely_at_equal_error(oracle_mod):
    """The pages contrast the fp32 rule (widen, then subtract) with an fp16
    path ("Correctness": about 0.1 % of indices differ, reconstruction MSE the
    same to 3 digits, on their calibrated codebook).  The kind of result, on
    synthetic keys: an fp16 subtract-square-sum variant (numpy float16, written
    here, not the oracle) disagrees with the oracle on a small nonzero fraction
    of indices, and the two reconstructions have the same MSE to within 1 %."""
    rng = np.random.default_rng(130)
    x = rng.standard_normal((1, 16384, 8)).astype(np.float16)
    cb = rng.standard_normal((1, 256, 8)).astype(np.float16)
    exact = oracle_mod.encode(x, cb)[0].astype(np.int64)
    d16 = x[0][:, None, :] - cb[0][None, :, :]          # float16 subtract
    dist16 = (d16 * d16).sum(axis=-1, dtype=np.float16)  # float16 squares and sums
    half = np.argmin(dist16, axis=1)
    frac = float((half != exact).mean())
    assert 0.0 < frac < 0.05, frac
    x64 = x[0].astype(np.float64)
    mse = lambda idx: float(((cb[0][idx].astype(np.float64) - x64) ** 2).mean())
    assert abs(mse(half) - mse(exact)) / mse(exact) < 0.01
    # the exact rule is never worse row by row (in float64)
    d_exact = ((cb[0][exact].astype(np.float64) - x64) ** 2).sum(-1)
    d_half = ((cb[0][half].astype(np.float64) - x64) ** 2).sum(-1)
    assert np.all(d_exact <= d_half * (1 + 1e-6) + 1e-12)

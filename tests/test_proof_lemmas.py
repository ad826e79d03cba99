"""The arithmetic facts the GPU kernels' exactness arguments rest on, checked
on the CPU with IEEE float32 arithmetic (numpy), exhaustively where the
domain is small.  None of these calls the library: they pin the lemmas the
kernels' comments state, so that a wrong lemma fails here and not only as a
rare mismatch on the GPU.

- tf32 pieces: a float's top 11 significant bits (hi), the next 11 of the
  exact remainder (mid) and the rest (lo) add up to it exactly, hi and mid are
  tf32 values, and |lo| <= 2^-20 |x| while the remainder is normal, below
  2^-136 otherwise (the two-piece split of smoothed and fp32 rows and of fp32
  codebooks; three pieces hold |c|^2).
- 16-bit inputs: every fp16 and bf16 value, and twice it, is a tf32 value, so
  the tensor-core products of 16-bit rows and -2c are exact.
- sign-bit tests: for finite a and b (or b = +inf), the sign bit of
  fl(a - b) is clear exactly when b <= a (candidate masks from thr - gmin,
  and the lowest index holding the least distance from least - d_j).
- finite-codebook distances: for finite centroids and a finite key, every
  fl(fl(y - c)^2) is finite or +inf, never NaN (the packed scan's premise).
"""
import numpy as np

F32 = np.float32


def tf32_trunc(x: np.ndarray) -> np.ndarray:
    """Keep the top 10 stored significand bits (11 significant bits)."""
    return (np.asarray(x, dtype=F32).view(np.uint32) & np.uint32(0xFFFFE000)).view(F32)


def sample_floats(n: int, seed: int) -> np.ndarray:
    """Random finite float32 bit patterns over the whole range, plus edge
    values: zeros, the smallest subnormal, powers of two, the largest float."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(F32)
    x = x[np.isfinite(x)]
    edge = np.array([0.0, -0.0, 1e-45, -1e-45, 1.0, -1.0, 2.0 ** -126, 3.4028235e38, -3.4028235e38,
                     1.0000001, 0.99999994, 65504.0, 2.0 ** 100], dtype=F32)
    return np.concatenate([x, edge])


def is_tf32(x: np.ndarray) -> np.ndarray:
    return (np.asarray(x, dtype=F32).view(np.uint32) & np.uint32(0x1FFF)) == 0


def split3(x):
    """hi, mid and the dropped rest, as the kernels form them in fp32."""
    hi = tf32_trunc(x)
    r1 = (x - hi).astype(F32)
    mid = tf32_trunc(r1)
    lo = (r1 - mid).astype(F32)
    return hi, r1, mid, lo


def test_tf32_split_is_exact_and_small_remainder():
    x = sample_floats(400_000, 1)
    x = np.concatenate([x, (x * F32(2.0 ** -120)).astype(F32)])  # many subnormals
    hi, r1, mid, lo = split3(x)
    # both subtractions are exact
    assert np.array_equal(r1.astype(np.float64), x.astype(np.float64) - hi.astype(np.float64))
    assert np.array_equal(lo.astype(np.float64), r1.astype(np.float64) - mid.astype(np.float64))
    total = hi.astype(np.float64) + mid.astype(np.float64) + lo.astype(np.float64)
    assert np.array_equal(total, x.astype(np.float64))
    assert is_tf32(hi).all() and is_tf32(mid).all()
    ax = np.abs(x.astype(np.float64))
    alo = np.abs(lo.astype(np.float64))
    # relative while the remainder is normal; below 2^-136 absolute otherwise
    normal_r1 = np.abs(r1) >= F32(2.0 ** -126)
    assert (alo[normal_r1] <= 2.0 ** -20 * ax[normal_r1]).all()
    assert (alo[~normal_r1] < 2.0 ** -136).all()
    assert ((alo <= 2.0 ** -20 * ax) | (alo < 2.0 ** -136)).all()
    # and the dropped part is a tf32 value (at most 2 significant bits) unless subnormal
    normal_lo = np.abs(lo) >= F32(2.0 ** -126)
    assert is_tf32(lo[normal_lo]).all()
    assert (np.abs(mid.astype(np.float64)) <= 2.0 ** -10 * ax + 2.0 ** -126).all()
    assert (np.abs(hi.astype(np.float64)) <= ax).all()


def test_three_tf32_pieces_hold_a_normal_float():
    """|c|^2 in three tf32 pieces: exact for normal values (24 = 11 + 11 + 2
    significant bits), short by less than 2^-136 below 2^-126."""
    x = np.abs(sample_floats(400_000, 7))
    x = np.concatenate([x, (x * F32(2.0 ** -110)).astype(F32)])
    hi, r1, mid, lo = split3(x)
    lo3 = tf32_trunc(lo)
    total = hi.astype(np.float64) + mid.astype(np.float64) + lo3.astype(np.float64)
    err = np.abs(total - x.astype(np.float64))
    assert (err[np.abs(lo) >= F32(2.0 ** -126)] == 0).all()
    assert (err < 2.0 ** -136).all()


def test_sixteen_bit_values_and_twice_them_are_tf32():
    """All 65,536 fp16 and bf16 bit patterns: each finite value, and -2 times
    it where that is finite, has no bit below the top 11 significant ones."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    f16 = bits.view(np.float16).astype(F32)
    bf16 = (bits.astype(np.uint32) << 16).view(F32)
    for v in (f16, bf16):
        v = v[np.isfinite(v)]
        assert is_tf32(v).all()
        with np.errstate(over="ignore"):
            w = (F32(-2.0) * v).astype(F32)
        fin = np.isfinite(w)
        assert is_tf32(w[fin]).all()
        assert np.array_equal(w[fin].astype(np.float64), -2.0 * v[fin].astype(np.float64))


def test_sign_of_the_rounded_difference():
    rng = np.random.default_rng(2)
    a = sample_floats(200_000, 3)
    b = a.copy()
    rng.shuffle(b)
    # nearby pairs too, where rounding decides: b one or two ulps from a
    with np.errstate(over="ignore"):
        near = np.nextafter(a, np.float32(np.inf)).astype(F32)
    a_all = np.concatenate([a, a, a, np.full(1000, F32(1.5))])
    b_all = np.concatenate([b, near, a, np.full(1000, F32(np.inf))])
    with np.errstate(over="ignore", invalid="ignore"):
        d = (a_all - b_all).astype(F32)
    ok = np.isfinite(a_all) & ~np.isnan(d)
    sign_clear = (d.view(np.uint32) >> np.uint32(31)) == 0
    assert np.array_equal(sign_clear[ok], (b_all <= a_all)[ok])
    # equal operands give +0, whatever their sign
    z = (a - a).astype(F32)
    assert ((z.view(np.uint32)) == 0).all()


def test_finite_codebook_distances_are_never_nan():
    rng = np.random.default_rng(4)
    c = sample_floats(2000, 5)
    y = np.concatenate([sample_floats(2000, 6), rng.standard_normal(2000).astype(F32)])
    with np.errstate(over="ignore"):
        t = (y[:, None] - c[None, :]).astype(F32)
        d = (t * t).astype(F32)
    assert not np.isnan(d).any()
    assert ((d >= 0) | np.isinf(d)).all()

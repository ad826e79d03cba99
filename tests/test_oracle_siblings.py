"""Pins of the oracle's sibling encoders (CPU only): the scalar (sub_dim = 1)
quantize and the randomised Hadamard rotation with its fused quantize.

Independent references: numpy's own fp32 arithmetic and argmin for the
scalar formula, the midpoint-count rule the pages state for sorted
codebooks, scipy's Hadamard matrix on integer data (exact), float64 products
within the fp32 error bound, and the orthogonality of the rotation.  Each pin
takes the oracle object so that planted mistakes can be run through it.
"""
import math

import numpy as np
import pytest
import scipy.linalg

U = 2.0 ** -24


def _to(dtype, a):
    if dtype == "f16":
        return a.astype(np.float16), False
    if dtype == "bf16":
        import torch

        t = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16), True
    return a.astype(np.float32), False


def _widen(x, bf16):
    if bf16:
        return (x.astype(np.uint32) << 16).view(np.float32)
    return x.astype(np.float32)


def _numpy_nearest(vals, centroids):
    """Index of the least fp32 (v - c)^2, first index on ties; NaN never wins."""
    d = vals[..., None] - centroids.astype(np.float32)   # fp32, round to nearest
    dist = d * d
    dist = np.where(np.isnan(dist), np.float32(np.inf), dist)
    return np.argmin(dist, axis=-1).astype(np.uint32)


def test_scalar_matches_numpy(oracle_mod):
    rng = np.random.default_rng(200)
    for dtype in ("f16", "bf16", "f32"):
        for n_c in (2, 4, 8, 16, 100, 256):
            x, bf = _to(dtype, 2.0 * rng.standard_normal(5000))
            c = rng.standard_normal(n_c).astype(np.float32)
            c[n_c // 2] = c[0]  # a duplicate: ties go to the lower index
            assert np.array_equal(oracle_mod.scalar_quantize(x, c, bf16=bf),
                                  _numpy_nearest(_widen(x, bf), c))


def test_scalar_special_values(oracle_mod):
    c = np.array([-1.0, 0.5, 2.0, 0.5], dtype=np.float32)
    x = np.array([np.nan, np.inf, -np.inf, 0.5, -0.25, 1.25, 3e38], dtype=np.float32)
    got = oracle_mod.scalar_quantize(x, c)
    # NaN: no distance wins -> 0; +inf and -inf: every distance is inf -> 0;
    # 0.5 sits on c[1] (and its copy c[3]); -0.25 ties c[0] and c[1] exactly;
    # 1.25 ties c[1] and c[2]; 3e38: (3e38 - c)^2 overflows for all -> 0
    assert got.tolist() == [0, 0, 0, 1, 0, 1, 0]


def test_scalar_midpoint_rule(oracle_mod):
    """For sorted distinct centroids the index is the number of midpoints the
    value exceeds, away from the midpoints themselves."""
    rng = np.random.default_rng(201)
    c = np.sort(rng.standard_normal(16)).astype(np.float32)
    mids = (c[:-1].astype(np.float64) + c[1:]) / 2
    x = rng.standard_normal(20000).astype(np.float32)
    far = np.min(np.abs(x[:, None] - mids[None, :]), axis=1) > 1e-5
    count = (x[:, None] > mids[None, :]).sum(axis=1)
    assert np.array_equal(oracle_mod.scalar_quantize(x, c)[far], count[far])


@pytest.mark.parametrize("dim", [1, 2, 4, 32, 128, 256])
def test_hadamard_exact_on_integers(oracle_mod, dim):
    """Integer rows (sums stay below 2^24): with scale 1 the rotation is
    exactly H_dim @ (diag * x), H the Sylvester Hadamard matrix."""
    rng = np.random.default_rng(202 + dim)
    x = rng.integers(-50, 51, (7, dim)).astype(np.float32)
    diag = rng.choice([-1.0, 1.0], dim).astype(np.float32)
    h = scipy.linalg.hadamard(dim).astype(np.float64)
    want = (diag.astype(np.float64) * x) @ h.T
    assert np.array_equal(oracle_mod.hadamard_rotate(x, diag, scale=1.0), want.astype(np.float32))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("dim", [8, 128, 512])
def test_hadamard_within_fp32_bound(oracle_mod, dtype, dim):
    """Against float64 H @ (diag * x) / sqrt(dim): each output is a pairwise
    sum over log2(dim) levels, then one scaling, so the error is at most
    (log2(dim) + 3) u sum_i |x_i| / sqrt(dim)."""
    rng = np.random.default_rng(203 + dim)
    x, bf = _to(dtype, rng.standard_normal((9, dim)))
    xf = _widen(x, bf).astype(np.float64)
    diag = rng.choice([-1.0, 1.0], dim).astype(np.float32)
    h = scipy.linalg.hadamard(dim).astype(np.float64)
    want = (diag * xf) @ h.T / math.sqrt(dim)
    got = oracle_mod.hadamard_rotate(x, diag, bf16=bf).astype(np.float64)
    bound = (math.log2(dim) + 3) * U * np.abs(xf).sum(axis=1, keepdims=True) / math.sqrt(dim)
    assert np.all(np.abs(got - want) <= bound)


def test_hadamard_twice_is_identity(oracle_mod):
    rng = np.random.default_rng(204)
    x = rng.standard_normal((5, 256)).astype(np.float32)
    ones = np.ones(256, dtype=np.float32)
    back = oracle_mod.hadamard_rotate(oracle_mod.hadamard_rotate(x, ones), ones)
    assert np.allclose(back, x, rtol=0, atol=40 * U * np.abs(x).sum() / 16)


def test_hadamard_scale_is_correctly_rounded(oracle_mod):
    assert oracle_mod.hadamard_scale(2).view(np.uint32) == 0x3F3504F3  # 1/sqrt(2)
    assert oracle_mod.hadamard_scale(128) == np.float32(0.70710677 / 8)
    assert oracle_mod.hadamard_scale(256) == np.float32(1 / 16)


def test_hadamard_quantize_is_rotate_then_scalar(oracle_mod):
    rng = np.random.default_rng(205)
    x = rng.standard_normal((11, 128)).astype(np.float16)
    diag = rng.choice([-1.0, 1.0], 128).astype(np.float32)
    c = np.sort(rng.standard_normal(16)).astype(np.float32)
    y = oracle_mod.hadamard_rotate(x, diag)
    assert np.array_equal(oracle_mod.hadamard_quantize(x, diag, c), _numpy_nearest(y, c))


def test_dim_one_rotation_is_the_sign_flip(oracle_mod):
    x = np.array([[1.5], [-2.0], [0.25]], dtype=np.float32)
    diag = np.array([-1.0], dtype=np.float32)
    assert np.array_equal(oracle_mod.hadamard_rotate(x, diag), -x)


PINS = [test_scalar_matches_numpy, test_scalar_special_values, test_scalar_midpoint_rule,
        lambda o: [test_hadamard_exact_on_integers(o, d) for d in (2, 32, 128)],
        lambda o: [test_hadamard_within_fp32_bound(o, t, d) for t in ("f16", "f32")
                   for d in (8, 128)],
        test_hadamard_twice_is_identity, test_hadamard_quantize_is_rotate_then_scalar,
        test_dim_one_rotation_is_the_sign_flip]

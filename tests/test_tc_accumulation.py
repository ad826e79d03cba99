"""The accumulation-error premise of the tensor-core screening encode,
measured on the GPU.

The bit-exactness of the library's tensor-core encode (``encode_tc``) rests on
one property of ``tcgen05.mma.kind::tf32`` that NVIDIA does not document: the
fp32 result of a chain of MMAs, accumulating K products of tf32 values in
tensor memory, differs from the exact sum of those products by at most
``eps_tc = 2^-16`` times the sum of their magnitudes.  Where products or
partial sums fall below the fp32 normal range the tensor core may flush them;
that costs at most ``2^-125`` per term, ``K * 2^-125`` in all, which the
kernel's absolute slack of ``2^-100`` covers.

This test drives the same instruction, descriptors, commit, wait and
tensor-memory loads as the library (``tests/harness/tc_probe.cu``) on
adversarial sets of scores, chains of 1 to 6 MMAs (K = 8 to 48 products, as
the library's fp32 and smoothed encodes chain up to 6), and checks the bound on
every score.  The worst ratio seen is printed (``pytest -s``).

The exact sums are float64: a product of two tf32 values (11 significant bits
each) is exact in float64, and a float64 sum of at most 48 of them errs by at
most ``48 * 2^-53`` (about ``2^-47.4``) of the sum of magnitudes, far below the
``2^-16`` being tested.
"""
import ctypes
import math
import zlib

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

EPS_TC = 2.0 ** -16
TILES = 16


@pytest.fixture(scope="module")
def harness():
    import tc_harness

    return tc_harness.load()


def tf32(v):
    """Nearest-below-in-magnitude tf32 value of each element (the top 10
    mantissa bits kept), as float32."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFFE000)
    return u.view(np.float32)


def tf32_next(v):
    """The tf32 value one unit in the last place above |v| (same sign)."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32) + np.uint32(0x2000)
    return u.view(np.float32)


def rand_tf32(rng, shape, lo_exp, hi_exp):
    m = 1.0 + rng.integers(0, 1024, shape) / 1024.0
    e = rng.integers(lo_exp, hi_exp + 1, shape)
    s = rng.choice([-1.0, 1.0], shape)
    return (s * np.ldexp(m, e)).astype(np.float32)


# ---------------------------------------------------------------- score sets
# Each returns A [TILES, 128, K] and B [TILES, ncols, K] of tf32 values.

def set_normal(rng, k, ncols):
    return (tf32(rng.standard_normal((TILES, 128, k))),
            tf32(rng.standard_normal((TILES, ncols, k))))


def set_decades(rng, k, ncols):
    # products spanning 2^-40 .. 2^40 within one row
    return rand_tf32(rng, (TILES, 128, k), -20, 20), rand_tf32(rng, (TILES, ncols, k), -20, 20)


def set_cancel_pairs(rng, k, ncols):
    # terms 2j and 2j+1 nearly cancel: a (b) + a (-(b + ulp b)) = -a ulp(b)
    a = rand_tf32(rng, (TILES, 128, k // 2), -6, 6)
    b = rand_tf32(rng, (TILES, ncols, k // 2), -6, 6)
    A = np.repeat(a, 2, axis=2)
    B = np.empty((TILES, ncols, k), np.float32)
    B[..., 0::2] = b
    B[..., 1::2] = -tf32_next(b)
    return A, B


def set_cancel_far(rng, k, ncols):
    # the cancelling partner sits in the other half of K (another MMA of the
    # chain when K > 8), so the cancellation happens across the accumulator
    a = rand_tf32(rng, (TILES, 128, k // 2), -8, 8)
    b = rand_tf32(rng, (TILES, ncols, k // 2), -8, 8)
    A = np.concatenate([a, a], axis=2)
    B = np.concatenate([b, -tf32_next(b)], axis=2)
    return A, B


def set_alternating(rng, k, ncols):
    # equal magnitudes with alternating signs: the exact sum is a small
    # multiple of the magnitudes' spacing
    base = 1.0 + rng.integers(0, 1024, (TILES, 128, 1)) / 1024.0
    A = np.broadcast_to(base * np.ldexp(1.0, rng.integers(-4, 5, (TILES, 128, 1))),
                        (TILES, 128, k)).astype(np.float32)
    signs = np.where(np.arange(k) % 2 == 0, 1.0, -1.0)
    mant = 1.0 + rng.integers(0, 4, (TILES, ncols, k)) / 1024.0
    B = (signs * mant).astype(np.float32)
    return A, B


def set_big_then_small(rng, k, ncols):
    # the first MMA's products are ~2^24 times the later ones
    A = rand_tf32(rng, (TILES, 128, k), -2, 2)
    B = rand_tf32(rng, (TILES, ncols, k), -2, 2)
    B[..., :8] *= np.float32(2.0 ** 24)
    return A, B


def set_small_then_big(rng, k, ncols):
    A = rand_tf32(rng, (TILES, 128, k), -2, 2)
    B = rand_tf32(rng, (TILES, ncols, k), -2, 2)
    B[..., -8:] *= np.float32(2.0 ** 24)
    return A, B


def _screen_operands(x, c):
    """The library's screening operands for 16-bit rows x [R, sub] and
    codebook c [C, sub] (float32 values): A = [x, 1, 1, 1, 0 ...],
    B = [-2c, |c|^2 as three tf32 pieces, 0 ...], K = 8 (sub 4) or 16."""
    sub = x.shape[-1]
    kk = 8 if sub == 4 else 16
    A = np.zeros(x.shape[:-1] + (kk,), np.float32)
    A[..., :sub] = x
    A[..., sub:sub + 3] = 1.0
    nrm = np.zeros(c.shape[:-1], np.float32)
    for i in range(sub):  # the kernel's fp32 |c|^2: square, then fused adds
        nrm = (nrm.astype(np.float64) + c[..., i].astype(np.float64) ** 2).astype(np.float32) \
            if i else (c[..., 0] * c[..., 0]).astype(np.float32)
    hi = tf32(nrm)
    mid = tf32(nrm - hi)
    lo = tf32(nrm - hi - mid)
    B = np.zeros(c.shape[:-1] + (kk,), np.float32)
    B[..., :sub] = -2.0 * c
    B[..., sub], B[..., sub + 1], B[..., sub + 2] = hi, mid, lo
    return A, B


def set_screen_offset(rng, k, ncols):
    # the library's fp16 screening operands for keys and centroids sharing a
    # large common offset: |c|^2 and -2 x.c nearly cancel
    sub = 4 if k == 8 else 8
    off = np.float32(rng.choice([64.0, 256.0, 1024.0]))
    x = (off + rng.standard_normal((TILES, 128, sub))).astype(np.float16).astype(np.float32)
    c = (off + rng.standard_normal((TILES, ncols, sub))).astype(np.float16).astype(np.float32)
    return _screen_operands(x, c)


def set_split_pieces(rng, k, ncols):
    # the library's fp32 screening operands: rows and -2c split into two tf32
    # pieces, three chained products (hi, b_hi), (mid, b_hi), (hi, b_mid)
    kk = k // 3
    sub = 4 if kk == 8 else 8
    scale = np.ldexp(1.0, rng.integers(-6, 7, (TILES, 1, 1)))
    x = (scale * rng.standard_normal((TILES, 128, sub))).astype(np.float32)
    c = (scale * rng.standard_normal((TILES, ncols, sub))).astype(np.float32)
    A0, B0 = _screen_operands(tf32(x), c)
    A0[..., :sub] = tf32(x)
    A1 = np.zeros_like(A0)
    A1[..., :sub] = tf32(x - tf32(x))
    w = (-2.0 * c).astype(np.float32)
    B0[..., :sub] = tf32(w)
    B1 = np.zeros_like(B0)
    B1[..., :sub] = tf32(w - tf32(w))
    return np.concatenate([A0, A1, A0], axis=2), np.concatenate([B0, B0, B1], axis=2)


def set_tiny(rng, k, ncols):
    # products and partial sums around and below the fp32 normal range
    return rand_tf32(rng, (TILES, 128, k), -66, -52), rand_tf32(rng, (TILES, ncols, k), -66, -52)


SETS = {
    "normal": (set_normal, (1, 2, 6)),
    "decades": (set_decades, (1, 2, 6)),
    "cancel_pairs": (set_cancel_pairs, (1, 2, 6)),
    "cancel_far": (set_cancel_far, (2, 4, 6)),
    "alternating": (set_alternating, (1, 2, 6)),
    "big_then_small": (set_big_then_small, (2, 6)),
    "small_then_big": (set_small_then_big, (2, 6)),
    "screen_offset": (set_screen_offset, (1, 2)),
    "split_pieces": (set_split_pieces, (3, 6)),
    "tiny": (set_tiny, (1, 2, 6)),
}


def run_chain(harness, A, B, nk, ncols):
    dev = torch.device("cuda")
    a = torch.from_numpy(np.ascontiguousarray(A)).to(dev)
    b = torch.from_numpy(np.ascontiguousarray(B)).to(dev)
    d = torch.full((TILES, 128, ncols), float("nan"), dtype=torch.float32, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    st = harness.probe_tf32_chain(a.data_ptr(), b.data_ptr(), d.data_ptr(), flag.data_ptr(), nk,
                                  ncols, TILES,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, f"launch failed: cuda error {st}"
    torch.cuda.synchronize()
    assert int(flag.item()) == 0, "a wait for the MMA gave up"
    return d.cpu().numpy()


@pytest.mark.parametrize("name", sorted(SETS))
@pytest.mark.parametrize("ncols", [64, 256])
def test_tf32_chain_error_within_eps_tc(harness, name, ncols):
    gen, nks = SETS[name]
    rng = np.random.default_rng(zlib.crc32(f"{name}/{ncols}".encode()))
    report = []
    for nk in nks:
        A, B = gen(rng, 8 * nk, ncols)
        assert A.shape == (TILES, 128, 8 * nk) and B.shape == (TILES, ncols, 8 * nk)
        # the operands are tf32 values: the tensor core reads them exactly
        assert np.array_equal(tf32(A), A) and np.array_equal(tf32(B), B)
        D = run_chain(harness, A, B, nk, ncols)
        A64, B64 = A.astype(np.float64), B.astype(np.float64)
        exact = np.einsum("tik,tjk->tij", A64, B64)
        mag = np.einsum("tik,tjk->tij", np.abs(A64), np.abs(B64))
        assert np.all(np.isfinite(D))
        err = np.abs(D.astype(np.float64) - exact)
        slack = 8 * nk * 2.0 ** -125 if name == "tiny" else 0.0
        bound = EPS_TC * mag + slack
        bad = err > bound
        assert not bad.any(), (
            f"{name} nk={nk} ncols={ncols}: {int(bad.sum())} scores beyond eps_tc; worst "
            f"err/mag = {float((err / np.where(mag > 0, mag, 1)).max()):.3e}")
        rel = err[mag > 0] / mag[mag > 0]
        worst = float(rel.max()) if rel.size else 0.0
        report.append(f"nk={nk}: worst err/sum|terms| = "
                      f"{'2^%.2f' % math.log2(worst) if worst > 0 else '0'}")
    print(f"[tf32 chain] {name} ncols={ncols}: " + "; ".join(report))

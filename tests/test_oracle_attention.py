"""Pins of the oracle's decode attention over product-VQ codes (CPU only).

The oracle (``oracle.attention_decode``) rebuilds keys and values from their
codes and applies softmax attention in float64.  These pins tie it to things
other than itself: PyTorch's scaled-dot-product attention on independently
gathered keys and values, a hand-worked example, closed forms (one token,
equal scores, a dominant key), and the index conventions (grouped-query head
mapping, sliding window, out-of-range codes).  Every pin takes the function
under test as an argument so that ``test_oracle_mutations.py`` can run them
against planted mistakes.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _case(seed, b=2, hq=4, hkv=2, t=7, d=8, sub=2, n_c=5):
    rng = np.random.default_rng(seed)
    ns = d // sub
    q = rng.standard_normal((b, hq, d))
    kcb = rng.standard_normal((hkv, n_c, sub))
    vcb = rng.standard_normal((hkv, n_c, sub))
    kc = rng.integers(0, n_c, (b, hkv, t, ns), dtype=np.uint8)
    vc = rng.integers(0, n_c, (b, hkv, t, ns), dtype=np.uint8)
    return q, kc, kcb, vc, vcb


def _sdpa(q, kc, kcb, vc, vcb, scale=None):
    """Library attention on keys/values gathered with torch indexing."""
    b, hq, d = q.shape
    _, hkv, t, ns = kc.shape
    kcb_t, vcb_t = torch.from_numpy(kcb), torch.from_numpy(vcb)
    heads = torch.arange(hkv)[None, :, None, None]
    keys = kcb_t[heads, torch.from_numpy(kc.astype(np.int64))].reshape(b, hkv, t, d)
    vals = vcb_t[heads, torch.from_numpy(vc.astype(np.int64))].reshape(b, hkv, t, d)
    rep = hq // hkv
    keys = keys.repeat_interleave(rep, dim=1)
    vals = vals.repeat_interleave(rep, dim=1)
    qt = torch.from_numpy(q)[:, :, None, :]
    out = torch.nn.functional.scaled_dot_product_attention(qt, keys, vals, scale=scale)
    return out[:, :, 0, :].numpy()


def test_matches_library_attention(fn=oracle.attention_decode):
    for seed, shape in ((1, {}), (2, dict(hq=8, hkv=2, d=12, sub=3, t=11, n_c=9)),
                        (3, dict(hq=3, hkv=3, d=4, sub=4, t=1)), (4, dict(b=1, hq=2, hkv=1, t=33))):
        q, kc, kcb, vc, vcb = _case(seed, **shape)
        np.testing.assert_allclose(fn(q, kc, kcb, vc, vcb), _sdpa(q, kc, kcb, vc, vcb),
                                   rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(fn(q, kc, kcb, vc, vcb, scale=0.37),
                                   _sdpa(q, kc, kcb, vc, vcb, scale=0.37), rtol=1e-12, atol=1e-12)


def test_hand_worked_example(fn=oracle.attention_decode):
    # D = 2, sub_dim = 1, scale 1: token 0 scores 0, token 1 scores ln 3, so
    # the weights are 1/4 and 3/4 and the output is 3/4 * [4, 0] = [3, 0].
    q = np.array([[[1.0, 0.0]]])
    kcb = np.array([[[0.0], [math.log(3.0)]]])
    vcb = np.array([[[0.0], [4.0]]])
    kc = np.array([[[[0, 0], [1, 0]]]], dtype=np.uint8)
    vc = np.array([[[[0, 0], [1, 0]]]], dtype=np.uint8)
    np.testing.assert_allclose(fn(q, kc, kcb, vc, vcb, scale=1.0), [[[3.0, 0.0]]], rtol=1e-14)


def test_single_token_returns_its_value_row(fn=oracle.attention_decode):
    q, kc, kcb, vc, vcb = _case(5, t=1)
    out = fn(q, kc, kcb, vc, vcb)
    for bi in range(q.shape[0]):
        for h in range(q.shape[1]):
            hk = h // (q.shape[1] // kc.shape[1])
            np.testing.assert_allclose(out[bi, h], vcb[hk][vc[bi, hk, 0]].reshape(-1), rtol=1e-14)


def test_equal_scores_average_the_values(fn=oracle.attention_decode):
    q, kc, kcb, vc, vcb = _case(6, t=9)
    kc[:] = kc[:, :, :1, :]  # every token has the same key
    out = fn(q, kc, kcb, vc, vcb)
    heads = np.arange(kc.shape[1])[None, :, None, None]
    mean_v = vcb[heads, vc.astype(np.int64)].reshape(*vc.shape[:3], -1).mean(axis=2)
    np.testing.assert_allclose(out, np.repeat(mean_v, 2, axis=1), rtol=1e-12, atol=1e-14)


def test_dominant_key_with_huge_logits(fn=oracle.attention_decode):
    # scores of order 1e4: the softmax must subtract its maximum (exp would
    # overflow otherwise) and put all weight on the dominant token.
    q, kc, kcb, vc, vcb = _case(7, b=1, hq=1, hkv=1, t=6, d=4, sub=2, n_c=4)
    q[:] = 100.0
    kcb[0] = 0.0
    kcb[0, 3] = 100.0
    kc[:] = 0
    kc[0, 0, 4] = 3
    out = fn(q, kc, kcb, vc, vcb, scale=1.0)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], vcb[0][vc[0, 0, 4]].reshape(-1), rtol=1e-14)


def test_window_attends_to_the_last_tokens(fn=oracle.attention_decode):
    q, kc, kcb, vc, vcb = _case(8, t=10)
    for w in (1, 3, 9):
        np.testing.assert_allclose(fn(q, kc, kcb, vc, vcb, window=w),
                                   _sdpa(q, kc[:, :, -w:], kcb, vc[:, :, -w:], vcb),
                                   rtol=1e-12, atol=1e-12)
    for w in (0, 10, 11):
        np.testing.assert_allclose(fn(q, kc, kcb, vc, vcb, window=w), _sdpa(q, kc, kcb, vc, vcb),
                                   rtol=1e-12, atol=1e-12)


def test_grouped_query_head_mapping(fn=oracle.attention_decode):
    # values of KV head k are all k + 1: query head h must return
    # h // (Hq / Hkv) + 1 in every coordinate
    q, kc, kcb, vc, vcb = _case(9, hq=6, hkv=3, d=6, sub=3)
    for k in range(3):
        vcb[k] = k + 1.0
    out = fn(q, kc, kcb, vc, vcb)
    want = (np.arange(6) // 2 + 1.0)[None, :, None] * np.ones_like(out)
    np.testing.assert_allclose(out, want, rtol=1e-14)


def test_out_of_range_codes_are_zero_rows(fn=oracle.attention_decode):
    q, kc, kcb, vc, vcb = _case(10, b=1, hq=1, hkv=1, t=4, d=4, sub=2, n_c=3)
    kc[0, 0, 1, 0] = 200
    vc[0, 0, 2, 1] = 7
    kcb_z = np.concatenate([kcb, np.zeros((1, 250, 2))], axis=1)
    vcb_z = np.concatenate([vcb, np.zeros((1, 250, 2))], axis=1)
    np.testing.assert_allclose(fn(q, kc, kcb, vc, vcb), _sdpa(q, kc, kcb_z, vc, vcb_z),
                               rtol=1e-12, atol=1e-14)


def test_empty_cache_gives_zeros(fn=oracle.attention_decode):
    q, kc, kcb, vc, vcb = _case(11, t=0)
    assert np.array_equal(fn(q, kc, kcb, vc, vcb), np.zeros(q.shape))


def test_token_order_does_not_matter(fn=oracle.attention_decode):
    q, kc, kcb, vc, vcb = _case(12, t=12)
    perm = np.random.default_rng(0).permutation(12)
    np.testing.assert_allclose(fn(q, kc[:, :, perm], kcb, vc[:, :, perm], vcb),
                               fn(q, kc, kcb, vc, vcb), rtol=1e-12, atol=1e-14)


PINS = [test_matches_library_attention, test_hand_worked_example,
        test_single_token_returns_its_value_row, test_equal_scores_average_the_values,
        test_dominant_key_with_huge_logits, test_window_attends_to_the_last_tokens,
        test_grouped_query_head_mapping, test_out_of_range_codes_are_zero_rows,
        test_empty_cache_gives_zeros, test_token_order_does_not_matter]

"""Workload geometry and the input recipes (no GPU needed)."""
import numpy as np
import pytest

import workloads
from conftest import read_golden

GOLD = {row[0]: row[1] for row in read_golden("shape_arithmetic.txt")}


def test_falcon_shape_matches_the_page():
    w = workloads.WORKLOADS["falcon_prefill"]
    assert w.tokens == int(GOLD["falcon_tokens"])
    assert w.kv_heads == int(GOLD["falcon_kv_heads"])
    assert w.sub_vectors_per_head == int(GOLD["falcon_subvectors_per_head"])
    assert w.n_centroids == int(GOLD["falcon_n_centroids"])
    assert w.sub_dim == int(GOLD["falcon_sub_dim"])
    assert w.n == int(GOLD["falcon_n_subvectors"])
    # the materialised [N, n_centroids, sub_dim] fp16 diff tensor of the pure path
    diff_bytes = w.n * w.n_centroids * w.sub_dim * 2
    assert round(diff_bytes / 1e9, 1) == float(GOLD["diff_tensor_gb"])
    # a fused encode holds only its input and output: 8 MiB fp16 in + 4 MiB uint32 out
    assert (w.x_bytes + w.out_bytes) / 2 ** 20 == float(GOLD["metal_peak_mb"])


def test_compression_arithmetic_matches_the_page():
    head_dim, sub_dim = 128, 8
    key_bytes = head_dim * 2
    code_bytes = head_dim // sub_dim  # one 8-bit code per sub-vector (256 centroids)
    assert key_bytes == int(GOLD["key_bytes_fp16_d128"])
    assert code_bytes == int(GOLD["codes_bytes_d128"])
    assert key_bytes // code_bytes == int(GOLD["compression"])


@pytest.mark.parametrize("name,n,groups,sub_dim", [
    ("tiny", 4096, 1, 4),
    ("llama_decode", 262_144, 32, 8),
    ("falcon_prefill", 1_048_576, 1, 4),
    ("long_context", 4_194_304, 8, 8),
    ("grouped_adversarial", 33_554_432, 256, 8),
])
def test_workload_sizes(name, n, groups, sub_dim):
    w = workloads.WORKLOADS[name]
    assert (w.n, w.n_groups, w.sub_dim, w.n_centroids) == (n, groups, sub_dim, 256)
    assert w.n_per_group * w.n_groups == w.n


@pytest.mark.parametrize("name", sorted(workloads.WORKLOADS))
def test_generation_is_seeded_and_shaped(name):
    w = workloads.WORKLOADS[name]
    tokens = min(w.tokens, 64)
    x1, cb1 = workloads.generate(name, tokens=tokens)
    x2, cb2 = workloads.generate(name, tokens=tokens)
    m = tokens * w.layers * w.kv_heads * w.sub_vectors_per_head // w.n_groups
    assert x1.shape == (w.n_groups, m, w.sub_dim) and x1.dtype == np.float16
    assert cb1.shape == (w.n_groups, w.n_centroids, w.sub_dim) and cb1.dtype == np.float16
    assert np.array_equal(x1.view(np.uint16), x2.view(np.uint16))
    assert np.array_equal(cb1.view(np.uint16), cb2.view(np.uint16))
    assert np.isfinite(x1.astype(np.float32)).all() and np.isfinite(cb1.astype(np.float32)).all()


def test_tiny_workload_is_standard_normal():
    x, cb = workloads.generate("tiny")
    assert x.shape == (1, 4096, 4)
    for a in (x, cb):
        v = a.astype(np.float64).ravel()
        assert abs(v.mean()) < 0.1 and abs(v.std() - 1) < 0.1


def test_adversarial_structure():
    x, cb = workloads.generate("grouped_adversarial", tokens=64)
    g, m, _ = x.shape
    n_dup = int(round(0.10 * 256))
    n_copy = int(round(0.01 * m))
    for k in (0, 17, g - 1):
        rows = cb[k].view(np.uint16).reshape(256, -1)
        _, first, counts = np.unique(rows, axis=0, return_index=True, return_counts=True)
        assert 256 - first.size <= n_dup and 256 - first.size >= n_dup // 2
        hits = (x[k][:, None, :] == cb[k][None]).all(-1).any(-1)
        assert hits.sum() >= n_copy


def test_long_context_has_outlier_channels():
    x, _ = workloads.generate("long_context", tokens=256)
    per_channel = x.astype(np.float64).reshape(8, 256, 16 * 8).std(axis=1)
    ratio = per_channel.max(axis=1) / per_channel.min(axis=1)
    assert (ratio > 3).all()

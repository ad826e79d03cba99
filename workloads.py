"""Seeded synthetic inputs for the product-VQ encode workloads.

This module holds the workload shapes and the random input recipes only: no
part of the encode arithmetic.  Both the CUDA path's tests and benchmark and
the CPU oracle's tests draw their inputs from here, so the two sides see the
same bytes.

Shapes follow the key-cache geometry of "I Wrote a Metal Kernel to Stop My Mac
From OOMing" ("What Even Is a KV Cache": keys of length head_dim are split into
head_dim / sub_dim sub-vectors; "What quantize_vq Was Doing Wrong": for the
Falcon3-7B shape N = 4096 tokens x 4 KV heads x 64 sub-vectors = 1,048,576).
The pages publish no calibrated codebooks or model keys, so standard-normal
fp16 keys and codebooks stand in for them (the codebook rows are drawn from the
same distribution as the keys, as a K-means codebook would follow it).

All values are drawn as float32 with NumPy's PCG64 and rounded to fp16
(round-to-nearest-even by ``astype``).
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """One encode workload: ``n_groups`` independent codebooks, each used by a
    contiguous run of ``n_per_group`` sub-vectors."""

    name: str
    description: str
    tokens: int
    layers: int
    kv_heads: int
    head_dim: int
    sub_dim: int
    n_centroids: int
    group_by: str  # "none", "layer" or "head" or "layer_head"

    @property
    def sub_vectors_per_head(self) -> int:
        return self.head_dim // self.sub_dim

    @property
    def n(self) -> int:
        """Total sub-vectors: tokens x layers x kv_heads x head_dim / sub_dim."""
        return self.tokens * self.layers * self.kv_heads * self.sub_vectors_per_head

    @property
    def n_groups(self) -> int:
        return {"none": 1, "layer": self.layers, "head": self.layers * self.kv_heads,
                "layer_head": self.layers * self.kv_heads}[self.group_by]

    @property
    def n_per_group(self) -> int:
        return self.n // self.n_groups

    @property
    def x_bytes(self) -> int:
        return self.n * self.sub_dim * 2

    @property
    def out_bytes(self) -> int:
        return self.n * 4


WORKLOADS = {
    # 4096 fp16 sub-vectors against one 256 x 4 codebook (x seed 0, codebook seed 1).
    "tiny": Workload("tiny", "tiny encode, N=4096, sub_dim=4", tokens=1024, layers=1,
                     kv_heads=1, head_dim=16, sub_dim=4, n_centroids=256, group_by="none"),
    # Llama-3.1-8B decode step, 64 tokens: 32 layers x 8 KV heads x head_dim 128,
    # one codebook per layer.
    "llama_decode": Workload("llama_decode", "Llama-3.1-8B-shape decode, 64 tokens, "
                             "32 per-layer codebooks", tokens=64, layers=32, kv_heads=8,
                             head_dim=128, sub_dim=8, n_centroids=256, group_by="layer"),
    # Falcon3-7B prefill: 4096 tokens x 4 KV heads x head_dim 256, one codebook.
    "falcon_prefill": Workload("falcon_prefill", "Falcon3-7B-shape prefill, 4096 tokens, "
                               "N=1,048,576, sub_dim=4", tokens=4096, layers=1, kv_heads=4,
                               head_dim=256, sub_dim=4, n_centroids=256, group_by="none"),
    # Long context: 32768 tokens x 8 KV heads x head_dim 128, one codebook per head,
    # keys with per-channel outlier scales.
    "long_context": Workload("long_context", "long-context prefill, 32768 tokens x 8 heads, "
                             "per-head codebooks, outlier channels", tokens=32768, layers=1,
                             kv_heads=8, head_dim=128, sub_dim=8, n_centroids=256,
                             group_by="head"),
    # 8192 tokens x 32 layers x 8 heads, one codebook per (layer, head), with
    # duplicated centroid rows and exact centroid copies in x.
    "grouped_adversarial": Workload("grouped_adversarial", "grouped + adversarial, 8192 "
                                    "tokens x 32 layers x 8 heads, 256 codebooks with "
                                    "duplicate rows, 1% exact copies",
                                    tokens=8192, layers=32, kv_heads=8, head_dim=128,
                                    sub_dim=8, n_centroids=256, group_by="layer_head"),
}

# Seeds per workload: (x, codebook, extra-1, extra-2).
SEEDS = {
    "tiny": (0, 1),
    "llama_decode": (2, 3),
    "falcon_prefill": (4, 5),
    "long_context": (6, 8, 7),            # x, codebook, channel scales
    "grouped_adversarial": (9, 10, 11, 12),  # x, codebook, codebook dup, x copies
}

DUP_CENTROID_FRACTION = 0.10
X_COPY_FRACTION = 0.01


def _normal(seed: int, shape) -> np.ndarray:
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape, dtype=np.float32)


def _layout(w: Workload, tokens: int):
    """Shapes of x and the codebooks for a workload with ``tokens`` tokens."""
    n_per_group = tokens * w.layers * w.kv_heads * w.sub_vectors_per_head // w.n_groups
    return (w.n_groups, n_per_group, w.sub_dim), (w.n_groups, w.n_centroids, w.sub_dim)


def generate(name: str, tokens: int | None = None):
    """Return ``(x, codebooks)`` as fp16 arrays ``[G, M, sub_dim]`` and
    ``[G, n_centroids, sub_dim]`` for workload ``name``.

    ``tokens`` shrinks the token count (same recipe, smaller M) for cases the
    CPU oracle must finish in seconds; ``None`` gives the full workload.
    """
    w = WORKLOADS[name]
    tokens = w.tokens if tokens is None else int(tokens)
    x_shape, cb_shape = _layout(w, tokens)
    seeds = SEEDS[name]
    if name == "long_context":
        return _long_context(w, tokens, x_shape, cb_shape, seeds)
    x = _normal(seeds[0], x_shape).astype(np.float16)
    cb = _normal(seeds[1], cb_shape).astype(np.float16)
    if name == "grouped_adversarial":
        _make_adversarial(x, cb, seeds[2], seeds[3])
    return x, cb


@dataclasses.dataclass(frozen=True)
class ScalarWorkload:
    """Keys quantized element by element (sub_dim = 1) against one Lloyd-Max
    codebook, optionally after a randomised Hadamard rotation of each
    head_dim row."""

    name: str
    description: str
    batch: int
    heads: int
    tokens: int
    head_dim: int
    bits: int

    @property
    def n(self) -> int:
        return self.batch * self.heads * self.tokens * self.head_dim

    @property
    def rows(self) -> int:
        return self.batch * self.heads * self.tokens


SCALAR_WORKLOADS = {
    # one layer's keys of a Llama-3.1-8B-shape cache (8 KV heads, head_dim 128)
    # at 32768 tokens, 4-bit codebook
    "turboquant_keys": ScalarWorkload("turboquant_keys", "Llama-3.1-8B-shape key cache, one layer, "
                                      "8 KV heads x 32768 tokens x 128, 4-bit Lloyd-Max codebook",
                                      batch=1, heads=8, tokens=32768, head_dim=128, bits=4),
}

SCALAR_SEEDS = {"turboquant_keys": (19, 20, 21)}  # keys, codebook sample, signs


def lloyd_max_gaussian(bits: int, seed: int, samples: int = 1 << 18, iters: int = 60):
    """Sorted float32 Lloyd-Max centroids of N(0, 1) for 2^bits levels, fitted
    by Lloyd iterations on a seeded sample (an input of the quantizer, not part
    of its arithmetic)."""
    z = np.sort(_normal(seed, (samples,)).astype(np.float64))
    k = 1 << bits
    c = np.quantile(z, (np.arange(k) + 0.5) / k)
    for _ in range(iters):
        edges = np.concatenate([[-np.inf], (c[:-1] + c[1:]) / 2, [np.inf]])
        idx = np.searchsorted(edges, z) - 1
        c = np.array([z[idx == j].mean() for j in range(k)])
    return c.astype(np.float32)


def generate_scalar(name: str, tokens: int | None = None):
    """``(x, centroids, diag)``: fp16 keys ``[B, H, S, D]`` ~ N(0, 1), the
    Lloyd-Max codebook, and random +-1 signs of the Hadamard rotation."""
    w = SCALAR_WORKLOADS[name]
    tokens = w.tokens if tokens is None else int(tokens)
    s = SCALAR_SEEDS[name]
    x = _normal(s[0], (w.batch, w.heads, tokens, w.head_dim)).astype(np.float16)
    c = lloyd_max_gaussian(w.bits, s[1])
    signs = np.random.Generator(np.random.PCG64(s[2])).integers(0, 2, w.head_dim)
    diag = np.where(signs == 1, 1.0, -1.0).astype(np.float32)
    return x, c, diag


SMOOTH_SEED = 18


def generate_smooth(name: str, tokens: int | None = None):
    """``(x, smooth, codebooks)`` for the smoothed encode of workload ``name``:
    ``smooth`` is ``[G, head_dim]`` float32, one factor per channel.

    For ``long_context`` the factors are the workload's own per-(head,
    channel) outlier scales, so the smoothed keys are about N(0, 1), and the
    codebooks are N(0, 1) rows (a codebook of the smoothed space).  For the
    other workloads x and the codebooks are those of :func:`generate` and the
    factors are exp(0.5 z), z ~ N(0, 1), per (group, channel).
    """
    w = WORKLOADS[name]
    head_dim = w.sub_vectors_per_head * w.sub_dim
    x, cb = generate(name, tokens)
    if name == "long_context":
        g = w.n_groups
        seeds = SEEDS[name]
        smooth = np.exp(np.float32(0.5) * _normal(seeds[2], (g, w.sub_vectors_per_head, w.sub_dim)))
        smooth = smooth.astype(np.float32).reshape(g, head_dim)
        cb = _normal(SMOOTH_SEED, cb.shape).astype(np.float16)
        return x, smooth, cb
    smooth = np.exp(np.float32(0.5) * _normal(SMOOTH_SEED, (w.n_groups, head_dim))).astype(np.float32)
    return x, smooth, cb


def _long_context(w, tokens, x_shape, cb_shape, seeds):
    """Keys with per-(head, channel) scale s = exp(0.5 z), z ~ N(0, 1), so a few
    channels are outliers; each head's codebook row r is N(0, 1) scaled by the
    channel scales of one uniformly chosen sub-vector slot p_r of that head."""
    g, m, sub = x_shape
    slots = w.sub_vectors_per_head
    scales = np.exp(np.float32(0.5) * _normal(seeds[2], (g, slots, sub))).astype(np.float32)
    z = _normal(seeds[0], (g, tokens, slots, sub))
    x = (z * scales[:, None, :, :]).reshape(x_shape).astype(np.float16)
    rng = np.random.Generator(np.random.PCG64(seeds[1]))
    rows = rng.standard_normal(cb_shape, dtype=np.float32)
    slot_of_row = rng.integers(0, slots, size=cb_shape[:2])
    cb_scale = np.take_along_axis(scales, slot_of_row[:, :, None], axis=1)
    cb = (rows * cb_scale).astype(np.float16)
    return x, cb


def _make_adversarial(x, cb, dup_seed, copy_seed):
    """In place: per group, overwrite round(10% n_c) distinct destination
    centroid rows with copies of uniformly chosen non-destination rows (so
    about half the duplicates sit below their source), then overwrite
    round(1% M) distinct rows of x with exact copies of uniformly chosen rows
    of that group's (final) codebook."""
    g, n_c, _ = cb.shape
    m = x.shape[1]
    n_dup = int(round(DUP_CENTROID_FRACTION * n_c))
    n_copy = int(round(X_COPY_FRACTION * m))
    rng_dup = np.random.Generator(np.random.PCG64(dup_seed))
    rng_copy = np.random.Generator(np.random.PCG64(copy_seed))
    for k in range(g):
        if n_dup:
            dest = rng_dup.choice(n_c, size=n_dup, replace=False)
            keep = np.setdiff1d(np.arange(n_c), dest)
            src = rng_dup.choice(keep, size=n_dup, replace=True)
            cb[k, dest] = cb[k, src]
        if n_copy:
            rows = rng_copy.choice(m, size=n_copy, replace=False)
            src = rng_copy.integers(0, n_c, size=n_copy)
            x[k, rows] = cb[k, src]


@dataclasses.dataclass(frozen=True)
class AttentionWorkload:
    """One decode step of attention over an 8-bit product-VQ KV cache."""

    name: str
    description: str
    batch: int
    heads_q: int
    heads_kv: int
    tokens: int
    head_dim: int
    sub_dim: int
    n_centroids: int
    window: int = 0

    @property
    def code_bytes(self) -> int:
        """Bytes of key + value codes read per step."""
        return 2 * self.batch * self.heads_kv * self.tokens * (self.head_dim // self.sub_dim)


ATTENTION_WORKLOADS = {
    # Llama-3.1-8B decode step: 32 query heads, 8 KV heads, head_dim 128,
    # sub_dim 8 (16 codes per token and head), batch 8, 32k cached tokens.
    "llama_attention": AttentionWorkload("llama_attention", "Llama-3.1-8B-shape decode "
                                         "attention, batch 8, 32768 cached tokens",
                                         batch=8, heads_q=32, heads_kv=8, tokens=32768,
                                         head_dim=128, sub_dim=8, n_centroids=256),
}

ATTENTION_SEEDS = {"llama_attention": (13, 14, 15, 16, 17)}


def generate_attention(name: str, tokens: int | None = None, batch: int | None = None):
    """``(q, k_codes, k_codebooks, v_codes, v_codebooks)`` for an attention
    workload: fp16 queries and codebooks ~ N(0, 1), codes uniform in
    [0, n_centroids) (keys and values of a cache encoded elsewhere)."""
    w = ATTENTION_WORKLOADS[name]
    tokens = w.tokens if tokens is None else int(tokens)
    batch = w.batch if batch is None else int(batch)
    s = ATTENTION_SEEDS[name]
    ns = w.head_dim // w.sub_dim
    q = _normal(s[0], (batch, w.heads_q, w.head_dim)).astype(np.float16)
    kcb = _normal(s[1], (w.heads_kv, w.n_centroids, w.sub_dim)).astype(np.float16)
    vcb = _normal(s[2], (w.heads_kv, w.n_centroids, w.sub_dim)).astype(np.float16)
    shape = (batch, w.heads_kv, tokens, ns)
    kc = np.random.Generator(np.random.PCG64(s[3])).integers(0, w.n_centroids, shape, dtype=np.uint8)
    vc = np.random.Generator(np.random.PCG64(s[4])).integers(0, w.n_centroids, shape, dtype=np.uint8)
    return q, kc, kcb, vc, vcb


def flat(x: np.ndarray) -> np.ndarray:
    """View ``[G, M, sub]`` as ``[G*M, sub]``."""
    return x.reshape(-1, x.shape[-1])

"""GPU parity of decode attention over 8-bit product-VQ codes.

The CUDA path (``vq_attention_decode`` through the C ABI) is compared element
by element with the float64 oracle on the same seeded inputs.  The kernel
computes in fp32 with a reordered (per-code) value sum and split-token
partials, so agreement is within a tolerance derived from its arithmetic
(``attention_tolerance``), not bit-exact.

Error bound, per output row (u = 2^-24, kappa = scale * log2 e, S_t = kappa *
q . K^_t the token's score in log2 units, M = max_t S_t, A_t = sum_i |q_i
K^_ti|, NS sub-spaces of SUB elements):
  * the table entry (a SUB-term fp32 dot product times kappa) and the score (a
    sum of NS entries) are off by at most delta_t = (SUB + NS + 3) u kappa A_t;
  * the weight 2^(S_t - m) of a token, with the subtraction, the exp2 (2 ulp),
    the rescales of the running sums and the merge factor, is off by a
    relative eps_t <= ln2 (delta_t + 2u (M - S_t)) + 2^-23 (4 + 3 * chunks);
  * the sums of weights (l) and of weighted value rows (fp32, per thread,
    then over at most 64 token streams, then over the slices) add at most
    (T + 80) u of l, resp. of l * max|V^|.
  Perturbing each weight by eps_t moves the normalised output by at most
  2 * (sum_t p_t eps_t / sum_t p_t) * max|V^|, so
    |out - exact| <= 1.1 * max|V^| * (2 * eps_bar + 4 * (T + 80) u)
  plus half an ulp of the output type (f16 2^-11, bf16 2^-8 relative).
"""
import math
import zlib

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
CHUNK = 512  # tokens per chunk of the kernel for up to 16 sub-spaces


def chunk_tokens(ns):
    """Tokens per chunk: 256 threads x (2 or 1) tokens."""
    return 256 * (2 if ns <= 16 else 1)


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


def to_dtype(a, dtype):
    """(numpy values exactly as the kernel sees them in float64, device tensor)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    t = t.to({"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[dtype])
    return t.to(torch.float64).numpy(), t.cuda()


def make_case(seed, b, hq, hkv, t, d, sub, n_c, dtype, q_gain=1.0):
    rng = np.random.default_rng(seed)
    ns = d // sub
    q, qd = to_dtype(q_gain * rng.standard_normal((b, hq, d)), dtype)
    kcb, kcbd = to_dtype(rng.standard_normal((hkv, n_c, sub)), dtype)
    vcb, vcbd = to_dtype(rng.standard_normal((hkv, n_c, sub)), dtype)
    kc = rng.integers(0, n_c, (b, hkv, t, ns), dtype=np.uint8)
    vc = rng.integers(0, n_c, (b, hkv, t, ns), dtype=np.uint8)
    host = (q, kc, kcb, vc, vcb)
    dev = (qd, torch.from_numpy(kc).cuda(), kcbd, torch.from_numpy(vc).cuda(), vcbd)
    return host, dev


def attention_tolerance(q, kc, kcb, vc, vcb, window=0, scale=0.0, dtype="f32"):
    """Per-element bound of the module docstring, shape [B, Hq, 1]."""
    b, hq, d = q.shape
    _, hkv, t, ns = kc.shape
    n_c, sub = kcb.shape[1], kcb.shape[2]
    first = t - window if 0 < window < t else 0
    n = t - first
    scale = scale if scale > 0 else 1.0 / math.sqrt(d)
    kappa = scale / math.log(2.0)
    chunks = max(1, -(-n // chunk_tokens(ns)))
    tol = np.zeros((b, hq, 1))
    if n == 0:
        return tol
    qpk = hq // hkv
    for bi in range(b):
        for h in range(hkv):
            idx_k = kc[bi, h, first:].astype(np.int64)
            idx_v = vc[bi, h, first:].astype(np.int64)
            kz = np.concatenate([kcb[h], np.zeros((256, sub))])  # codes >= n_c: zero rows
            vz = np.concatenate([vcb[h], np.zeros((256, sub))])
            keys = kz[idx_k].reshape(n, d)
            vmax = np.abs(vz[idx_v]).max()
            for g in range(qpk):
                qv = q[bi, h * qpk + g]
                s = kappa * (keys @ qv)
                a = np.abs(keys) @ np.abs(qv)
                p = np.exp2(s - s.max())
                delta = (sub + ns + 3) * U * kappa * a
                eps = math.log(2.0) * (delta + 2 * U * (s.max() - s)) + 2.0 ** -23 * (4 + 3 * chunks)
                eps_bar = float((p * eps).sum() / p.sum())
                tol[bi, h * qpk + g] = 1.1 * vmax * (2 * eps_bar + 4 * (n + 80) * U)
    return tol


def check(vq, oracle_mod, host, dev, dtype, window=0, scale=0.0, workspace=None):
    out = vq.vq_attention_decode(*dev, window=window, scale=scale, workspace=workspace)
    torch.cuda.synchronize()
    got = out.to(torch.float64).cpu().numpy()
    want = oracle_mod.attention_decode(*host, window=window, scale=scale)
    tol = attention_tolerance(*host, window=window, scale=scale, dtype=dtype)
    rel_out = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8, "f32": 0.0}[dtype]
    bound = tol + rel_out * np.abs(want) + 1e-30
    err = np.abs(got - want)
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert np.all(err <= bound), (
        f"max err/bound {float((err / bound)[worst]):.3g} at {worst}: got {got[worst]}, "
        f"want {want[worst]}, bound {bound[worst]}")
    return got


CASES = [
    # (b, hq, hkv, tokens, head_dim, sub_dim, n_centroids, dtype)
    (2, 8, 2, 3000, 128, 8, 256, "f16"),    # GQA 4, 16 sub-spaces, ragged last chunk
    (1, 32, 8, 5000, 128, 4, 256, "bf16"),  # 32 sub-spaces
    (2, 8, 8, 1500, 64, 8, 256, "f32"),     # multi-head, 8 sub-spaces
    (1, 16, 2, 2500, 256, 8, 256, "f16"),   # GQA 8, head_dim 256
    (1, 4, 1, 4100, 256, 4, 256, "f16"),    # 64 sub-spaces
    (1, 8, 2, 3000, 128, 32, 256, "f32"),   # 4 sub-spaces of 32
    (2, 6, 2, 2049, 64, 4, 256, "bf16"),    # GQA 3 (three heads per block)
    (1, 32, 2, 2000, 128, 8, 256, "f16"),   # GQA 16: two head groups per KV head
    (3, 4, 4, 777, 128, 8, 100, "f32"),     # 100 centroids; codes up to 99
    (1, 8, 1, 2000, 512, 8, 256, "f16"),    # head_dim 512 (the maximum), 64 sub-spaces
    (1, 4, 4, 1000, 512, 32, 256, "bf16"),  # head_dim 512, sub_dim 32
    (2, 16, 2, 1500, 64, 16, 256, "f32"),   # 4 sub-spaces of 16, GQA 8
    (1, 64, 8, 700, 128, 8, 256, "f16"),    # 64 query heads
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_attention_matches_oracle(vq, oracle_mod, case):
    b, hq, hkv, t, d, sub, n_c, dtype = case
    host, dev = make_case(zlib.crc32(repr(case).encode()), b, hq, hkv, t, d, sub, n_c, dtype)
    check(vq, oracle_mod, host, dev, dtype)


@pytest.mark.parametrize("window", [1, 1000, 1023, 1025, 4999, 5000, 7000])
def test_sliding_window(vq, oracle_mod, window):
    host, dev = make_case(window, 2, 8, 2, 5000, 128, 8, 256, "f16")
    check(vq, oracle_mod, host, dev, "f16", window=window)


def test_explicit_scale_and_large_logits(vq, oracle_mod):
    # queries 30x larger: scores spread over hundreds of log2 units, so later
    # chunks raise the running maximum and rescale the value weights
    host, dev = make_case(21, 2, 8, 2, 6000, 128, 8, 256, "f32", q_gain=30.0)
    check(vq, oracle_mod, host, dev, "f32")
    check(vq, oracle_mod, host, dev, "f32", scale=0.05)


def test_rising_scores_force_rescales(vq, oracle_mod):
    # key codes chosen so the best score rises chunk after chunk
    host, dev = make_case(22, 1, 4, 1, 8 * CHUNK, 64, 8, 256, "f32", q_gain=4.0)
    q, kc, kcb, vc, vcb = host
    ns = kc.shape[-1]
    order = np.argsort((kcb[0] @ q[0, 0].reshape(ns, 8).T).T, axis=1)  # [ns][n_c] by score
    t = kc.shape[2]
    rank = (np.arange(t) * 255 // (t - 1)).astype(np.int64)
    kc[0, 0] = order[np.arange(ns)[None, :], rank[:, None]].astype(np.uint8)
    dev = (dev[0], torch.from_numpy(kc).cuda(), dev[2], dev[3], dev[4])
    check(vq, oracle_mod, (q, kc, kcb, vc, vcb), dev, "f32")


def test_out_of_range_codes_read_zero_rows(vq, oracle_mod):
    host, dev = make_case(23, 1, 4, 2, 2000, 64, 8, 50, "f16")
    q, kc, kcb, vc, vcb = host
    rng = np.random.default_rng(5)
    kc[rng.random(kc.shape) < 0.05] = 200
    vc[rng.random(vc.shape) < 0.05] = 255
    dev = (dev[0], torch.from_numpy(kc).cuda(), dev[2], torch.from_numpy(vc).cuda(), dev[4])
    check(vq, oracle_mod, (q, kc, kcb, vc, vcb), dev, "f16")


@pytest.mark.parametrize("tokens", [0, 1, 2, 1023, 1024, 1025])
def test_short_and_empty_caches(vq, oracle_mod, tokens):
    host, dev = make_case(100 + tokens, 2, 8, 2, tokens, 128, 8, 256, "f16")
    got = check(vq, oracle_mod, host, dev, "f16")
    if tokens == 0:
        assert not np.any(got)


def test_small_workspace_uses_fewer_slices(vq, oracle_mod):
    host, dev = make_case(31, 2, 8, 2, 20000, 128, 8, 256, "f16")
    b, hq, d = host[0].shape
    full = vq.vq_attention_workspace_bytes(b, hq, 2, 20000, d, 8, 256)
    per_slice = b * hq * (d + 2) * 4
    assert full % per_slice == 0 and full // per_slice > 1
    for slices in (1, 2, 3):
        ws = torch.empty(slices * per_slice, dtype=torch.uint8, device="cuda")
        check(vq, oracle_mod, host, dev, "f16", workspace=ws)
    with pytest.raises(vq.VQError):
        vq.vq_attention_decode(*dev, workspace=torch.empty(per_slice - 16, dtype=torch.uint8,
                                                           device="cuda"))


def test_long_cache_many_slices(vq, oracle_mod):
    """A quarter-million-token cache of one sequence: hundreds of chunks,
    many token slices merged."""
    host, dev = make_case(51, 1, 8, 2, 262144, 128, 8, 256, "f16")
    check(vq, oracle_mod, host, dev, "f16")


def test_repeated_calls_agree(vq):
    _, dev = make_case(41, 2, 8, 2, 9000, 128, 8, 256, "f32")
    a = vq.vq_attention_decode(*dev)
    b = vq.vq_attention_decode(*dev)
    torch.cuda.synchronize()
    # no atomics: every sum has a fixed order, so repeated calls agree bit for bit
    assert torch.equal(a, b)


def test_llama_attention_full_size(vq, oracle_mod):
    """The benchmarked decode step (batch 8, 32 query / 8 KV heads, head_dim
    128, sub_dim 8, 32768 tokens), every output against the oracle."""
    q, kc, kcb, vc, vcb = workloads.generate_attention("llama_attention")
    dev = tuple(torch.from_numpy(a).cuda() for a in (q, kc, kcb, vc, vcb))
    host = (q.astype(np.float64), kc, kcb.astype(np.float64), vc, vcb.astype(np.float64))
    check(vq, oracle_mod, host, dev, "f16")

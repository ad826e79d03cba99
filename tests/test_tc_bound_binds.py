"""Bit-exact parity of the tensor-core encode where its screening bound
decides.

The tensor-core encode screens centroids with tf32 MMA scores and evaluates
the exact fp32 formula only for the centroid groups whose screened minimum
lies within a threshold of the least one; rows with more than two such groups
go to an exact scan.  The threshold comes from a bound on the scores' error
that grows with C2 + sum_i |x_i| A_i (the largest |c|^2 of the codebook, and
the row against the largest |c_i|).  When keys and codebook share a common
offset O, that bound grows as O^2 while the distances and their gaps do not.
Sweeping O moves the rows from one candidate group (small O), through one or
two groups with the nearest excluded group close to the threshold, to the
exact scan (large O).  In the middle of the sweep the choice of groups rests
on the bound: were the tensor core's error larger than the bound assumes, a
true nearest centroid could be screened out there.

The sweep runs for fp16, bf16 and fp32 keys and for smoothed fp16 keys, at
sub_dim 4 and 8, one offset per codebook group:
  * through the library (``vq_encode_grouped`` / ``vq_encode_grouped_smooth``),
    bit-exact against the oracle on every row;
  * through the same kernel built with screening statistics
    (``tests/harness/tc_stats.cu``), equally bit-exact, whose histogram of
    outcomes per offset is printed (``pytest -s``) and must show rows decided
    at the threshold: at some offset at least 1% of the rows have their
    nearest excluded group within one bound of the threshold while fewer
    than half go to the exact scan.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

OFFSETS = [0.0, 4.0, 8.0, 12.0, 16.0, 24.0, 32.0, 48.0, 64.0, 128.0]
HEAD_DIM = 64
N_C = 256
CASES = [("f16", 4, False), ("f16", 8, False), ("bf16", 4, False), ("bf16", 8, False),
         ("f32", 4, False), ("f32", 8, False), ("f16", 4, True), ("f16", 8, True)]
DTYPE_CODE = {"f16": 0, "bf16": 1, "f32": 2}
TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


@pytest.fixture(scope="module")
def harness():
    import tc_harness

    return tc_harness.load()


def make_case(dtype, sub, smooth, seed):
    """Keys and codebooks sharing offset OFFSETS[g] in group g; with smooth,
    keys are scaled per channel by factors exp(0.25 z) so that the divided
    keys sit at the offset."""
    rng = np.random.default_rng(seed)
    g = len(OFFSETS)
    m = (HEAD_DIM // sub) * 801  # whole keys, a ragged last tile
    off = np.asarray(OFFSETS, np.float64)[:, None, None]
    x = off + rng.standard_normal((g, m, sub))
    cb = off + rng.standard_normal((g, N_C, sub))
    factors = None
    if smooth:
        factors = np.exp(0.25 * rng.standard_normal((g, HEAD_DIM))).astype(np.float32)
        ch = (np.arange(m)[:, None] % (HEAD_DIM // sub)) * sub + np.arange(sub)[None, :]
        x = x * factors[:, ch]
    tdt = TORCH_DTYPE[dtype]
    xt = torch.from_numpy(x.astype(np.float32)).to(tdt)
    cbt = torch.from_numpy(cb.astype(np.float32)).to(tdt)
    if dtype == "bf16":  # the oracle takes bf16 as its raw bits
        xh = xt.view(torch.int16).numpy().view(np.uint16)
        cbh = cbt.view(torch.int16).numpy().view(np.uint16)
    else:
        xh, cbh = xt.numpy(), cbt.numpy()
    return xt, cbt, factors, xh, cbh


@pytest.mark.parametrize("dtype,sub,smooth", CASES,
                         ids=[f"{d}-sub{s}{'-smooth' if sm else ''}" for d, s, sm in CASES])
def test_offset_sweep_is_bit_exact_where_the_bound_decides(vq, oracle_mod, harness, dtype, sub,
                                                           smooth):
    import os

    import tc_harness

    xt, cbt, factors, xh, cbh = make_case(dtype, sub, smooth, seed=900 + 10 * sub + len(dtype))
    g, m, _ = xt.shape
    threads = os.cpu_count() or 1
    if smooth:
        want = oracle_mod.encode_smooth(xh, factors, cbh, HEAD_DIM, bf16=dtype == "bf16",
                                        n_threads=threads)
    else:
        want = oracle_mod.encode(xh, cbh, bf16=dtype == "bf16", n_threads=threads)
    dev = torch.device("cuda")
    xd, cbd = xt.to(dev), cbt.to(dev)
    fd = torch.from_numpy(factors).to(dev) if smooth else None
    desc = vq.vq_describe_launch(g, m, N_C, sub, TORCH_DTYPE[dtype], xd.data_ptr())
    assert desc.startswith("kernel=encode_tc"), desc
    if smooth:
        got = vq.vq_encode_grouped_smooth(xd, fd, cbd, HEAD_DIM, index_bytes=4)
    else:
        got = vq.vq_encode_grouped(xd, cbd)
    got = got.view(torch.int32).cpu().numpy().view(np.uint32)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} rows differ, first (group, row) {bad[:5].tolist()}"

    # the same kernel with screening statistics, one offset per launch
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    tc_harness.read_stats(clear=True)
    tc_harness.status("stats", clear=True)
    lines, decided = [], []
    for gi, offset in enumerate(OFFSETS):
        out = torch.full((m,), 0x7fffffff, dtype=torch.int32, device=dev)
        st = harness.stats_encode(DTYPE_CODE[dtype], sub, 1 if smooth else 0,
                                  xd[gi].data_ptr(), cbd[gi].data_ptr(), 1, m, N_C, 2,
                                  out.data_ptr(), fd[gi].data_ptr() if smooth else None,
                                  HEAD_DIM, stream)
        assert st == 0, f"stats launch failed: cuda error {st}"
        h = tc_harness.read_stats(clear=True)
        assert sum(h) == m
        assert np.array_equal(out.cpu().numpy().view(np.uint32), want[gi])
        one, one_tight, two, two_tight, queued = (v / m for v in h)
        decided.append((one_tight + two_tight, queued))
        lines.append(f"  offset {offset:6.1f}: 1 group {one:6.1%} (tight {one_tight:6.1%})  "
                     f"2 groups {two:6.1%} (tight {two_tight:6.1%})  exact scan {queued:6.1%}")
    assert tc_harness.status("stats") == 0
    print(f"[screening outcomes] {dtype} sub_dim {sub}{' smoothed' if smooth else ''}, "
          f"{m} rows per offset:\n" + "\n".join(lines))
    assert any(t >= 0.01 and q < 0.5 for t, q in decided), decided

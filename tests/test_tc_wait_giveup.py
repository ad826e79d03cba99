"""The give-up path of the tensor-core encode's bounded waits, on the GPU.

The encode waits for each MMA on an mbarrier with a bounded number of polls.
Should a wait give up, the block must not free its tensor memory, or exit,
while an MMA it issued may still be writing it; it marks every row it has not
encoded (0xFFFFFFFF, or 0xFF as 8-bit codes) and records the failure in the
device status word.  In the library the limit is 2^22 polls and has never been
reached; ``tests/harness/tc_polls.cu`` builds the same kernel with 0 or 1
polls per pass, so the waits give up while every MMA still completes (the
final wait before the memory is freed keeps the full limit).  No wait is left
unbounded and no access differs from the library's: the waits only run out
early.

Checked here:
  * with 0 polls every row of every block is marked and the status word says
    so (with 8-bit codes at 256 centroids the marker is a valid code, and
    only the status word tells);
  * with 1 poll each block's rows are correct up to the tile whose wait gave
    up and marked from there on, and the status bit is set exactly when some
    row is marked;
  * a normal library call afterwards, on the same device, is bit-exact and
    leaves the library's status word clear (``vq_kernel_status``).
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

N_C = 256
TILES_PER_BLOCK = 3


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


def make(sub, seed, g=3, m=5000):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((g, m, sub)).astype(np.float16)
    cb = rng.standard_normal((g, N_C, sub)).astype(np.float16)
    return x, cb


def run_polls(harness, polls, sub, out_bytes, xd, cbd):
    g, m, _ = xd.shape
    dt = torch.int32 if out_bytes == 4 else torch.uint8
    out = torch.full((g, m), 7, dtype=dt, device=xd.device)
    st = harness.polls_encode(polls, sub, out_bytes, xd.data_ptr(), cbd.data_ptr(), g, m, N_C,
                              TILES_PER_BLOCK, out.data_ptr(),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, f"launch failed: cuda error {st}"
    torch.cuda.synchronize()
    res = out.cpu().numpy()
    return res.view(np.uint32) if out_bytes == 4 else res.astype(np.uint32)


def library_call_is_exact(vq, oracle_mod, xd, cbd, x, cb):
    assert vq.vq_kernel_status(clear=True) == 0
    got = vq.vq_encode_grouped(xd, cbd).view(torch.int32).cpu().numpy().view(np.uint32)
    assert np.array_equal(got, oracle_mod.encode(x, cb, n_threads=8))
    assert vq.vq_kernel_status() == 0


@pytest.mark.parametrize("sub,out_bytes", [(4, 4), (4, 1), (8, 4)])
def test_zero_polls_mark_every_row_and_set_the_status(vq, oracle_mod, harness, sub, out_bytes):
    import tc_harness

    x, cb = make(sub, seed=31 + sub + out_bytes)
    xd, cbd = torch.from_numpy(x).cuda(), torch.from_numpy(cb).cuda()
    tc_harness.status("polls", clear=True)
    got = run_polls(harness, 0, sub, out_bytes, xd, cbd)
    marker = 0xFFFFFFFF if out_bytes == 4 else 0xFF
    assert np.all(got == marker)
    assert tc_harness.status("polls") & vq.VQ_KSTATUS_WAIT_GAVE_UP
    assert tc_harness.status("polls") == 0  # cleared by the read above
    library_call_is_exact(vq, oracle_mod, xd, cbd, x, cb)


@pytest.mark.parametrize("sub", [4, 8])
def test_one_poll_marks_a_suffix_of_tiles_per_block(vq, oracle_mod, harness, sub):
    import tc_harness

    x, cb = make(sub, seed=47 + sub, m=40000)
    want = oracle_mod.encode(x, cb, n_threads=8)
    xd, cbd = torch.from_numpy(x).cuda(), torch.from_numpy(cb).cuda()
    g, m = want.shape
    marked_any = False
    for _ in range(3):
        tc_harness.status("polls", clear=True)
        got = run_polls(harness, 1, sub, 4, xd, cbd)
        marked = got == 0xFFFFFFFF
        assert np.array_equal(got[~marked], want[~marked])
        # per block (TILES_PER_BLOCK tiles of 128 rows of one group): correct
        # tiles first, then marked tiles to the block's end
        rows_per_block = 128 * TILES_PER_BLOCK
        for gi in range(g):
            for b0 in range(0, m, rows_per_block):
                blk = marked[gi, b0:b0 + rows_per_block]
                tiles = [blk[t:t + 128] for t in range(0, blk.size, 128)]
                states = [bool(t.all()) if t.any() else False for t in tiles]
                assert all(t.all() or not t.any() for t in tiles), "a tile partly marked"
                first = states.index(True) if True in states else len(states)
                assert all(states[first:]), f"group {gi} block at row {b0}: {states}"
        bits = tc_harness.status("polls")
        assert bool(bits & vq.VQ_KSTATUS_WAIT_GAVE_UP) == bool(marked.any())
        marked_any |= bool(marked.any())
    print(f"[one poll] sub_dim {sub}: some wait gave up: {marked_any}")
    library_call_is_exact(vq, oracle_mod, xd, cbd, x, cb)


def test_kernel_status_reads_clean_after_normal_work(vq):
    x = torch.randn(2, 3000, 8, device="cuda").half()
    cb = torch.randn(2, 256, 8, device="cuda").half()
    vq.vq_kernel_status(clear=True)
    vq.vq_encode_grouped(x, cb)
    vq.vq_encode_grouped_u8(x, cb)
    assert vq.vq_kernel_status() == 0

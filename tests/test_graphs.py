"""The device entry points can be captured in a CUDA graph and replayed.

A decode loop that encodes each step's new keys and attends over the codes
issues a handful of small launches per step; capturing them once into a CUDA
graph and replaying removes the host overhead of every launch.  Each case
captures one call on a side stream (torch.cuda.graph), writes new inputs into
the captured buffers, replays, and compares with a direct call on the same
inputs.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


def capture_and_replay(fn, inputs, fresh):
    """Capture fn(*inputs) into a graph, copy `fresh` into `inputs`, replay;
    return (replayed output, direct output on the fresh inputs)."""
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn(*inputs)  # warm-up outside the capture (kernel attributes, workspace)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = fn(*inputs)
    for dst, src in zip(inputs, fresh):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    replayed = out.clone()
    direct = fn(*fresh)
    torch.cuda.synchronize()
    return replayed, direct


def test_encode_in_a_graph(vq):
    rng = np.random.default_rng(1)
    mk = lambda: torch.from_numpy(rng.standard_normal((4, 5000, 8)).astype(np.float16)).cuda()
    cb = torch.from_numpy(rng.standard_normal((4, 256, 8)).astype(np.float16)).cuda()
    a, b = capture_and_replay(lambda x, c: vq.vq_encode_grouped(x, c), (mk(), cb), (mk(), cb))
    assert torch.equal(a, b)
    a, b = capture_and_replay(lambda x, c: vq.vq_encode_grouped_u8(x, c), (mk(), cb), (mk(), cb))
    assert torch.equal(a, b)
    codes = vq.vq_encode_grouped_u8(mk(), cb)
    a, b = capture_and_replay(lambda i, c: vq.vq_dequantize_grouped(i, c), (codes.clone(), cb),
                              (vq.vq_encode_grouped_u8(mk(), cb), cb))
    assert torch.equal(a, b)


def test_smoothed_encode_in_a_graph(vq):
    x, s, cb = workloads.generate_smooth("llama_decode")
    x2, _, _ = workloads.generate_smooth("llama_decode")
    x2 = np.ascontiguousarray(x2[:, ::-1])  # other rows
    xs = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (x, x2)]
    sd, cbd = torch.from_numpy(s).cuda(), torch.from_numpy(cb).cuda()
    a, b = capture_and_replay(lambda xx: vq.vq_encode_grouped_smooth(xx, sd, cbd, 128), (xs[0],),
                              (xs[1],))
    assert torch.equal(a, b)


def test_attention_in_a_graph(vq):
    arrays = workloads.generate_attention("llama_attention", tokens=3000, batch=2)
    dev = [torch.from_numpy(a).cuda() for a in arrays]
    q2 = torch.flip(dev[0], dims=[1]).contiguous()
    ws = torch.empty(vq.vq_attention_workspace_bytes(2, 32, 8, 3000, 128, 8, 256),
                     dtype=torch.uint8, device="cuda")
    fn = lambda q: vq.vq_attention_decode(q, *dev[1:], workspace=ws)
    a, b = capture_and_replay(fn, (dev[0].clone(),), (q2,))
    assert torch.equal(a, b)  # same plan, no atomics: the same bits


def test_scalar_and_hadamard_in_a_graph(vq):
    x, c, diag = workloads.generate_scalar("turboquant_keys", tokens=256)
    xd = torch.from_numpy(x).cuda()
    x2 = (xd * 0.5).contiguous()
    cd, dd = torch.from_numpy(c).cuda(), torch.from_numpy(diag).cuda()
    ws = torch.empty(65536, dtype=torch.uint8, device="cuda")
    a, b = capture_and_replay(lambda xx: vq.vq_scalar_quantize(xx, cd, workspace=ws), (xd.clone(),), (x2,))
    assert torch.equal(a, b)
    a, b = capture_and_replay(lambda xx: vq.vq_hadamard_quantize(xx, dd, cd), (xd.clone(),), (x2,))
    assert torch.equal(a, b)

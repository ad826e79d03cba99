"""The bounds-checked build (``libvqenc_checked.so``), on the GPU.

``compute-sanitizer`` may not run on these machines, so the library is built a
second time with ``-DVQ_CHECKED`` (``csrc/vq_check.cuh``): every index the
encode (tensor-core, filter), attention, scalar-lookup and Hadamard kernels
compute into a global or shared buffer is checked against that buffer before
the access, and a span outside it sets an out-of-bounds bit in the device
status word instead of being made.  Its entry points wait for their launches
and return ``VQ_ERR_INTERNAL`` when the bit is set.

Checked here:
  * the check primitives themselves, evaluated by a probe kernel on spans it
    describes but never touches (``tests/harness/check_probe.cu``): spans
    inside, straddling the end, before the start and misaligned;
  * every entry point of the checked build on ragged sizes, tile boundaries,
    every kernel of the dispatch and every attention head grouping: each call
    returns ``VQ_OK`` and its output is bit-identical to the library
    build's, and the status word stays clear.
"""
import contextlib
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    from product_vq_kv_gb300 import build as b
    import product_vq_kv_gb300._binding as bind

    b.build()
    b.build(checked=True)
    normal = bind.load_library()
    checked = bind._configure(ctypes.CDLL(b.CHECKED_LIB_PATH))
    return bind, normal, checked


@contextlib.contextmanager
def using(bind, lib):
    saved = bind._lib
    bind._lib = lib
    try:
        yield
    finally:
        bind._lib = saved


def both(libs, fn):
    """fn() through the library and through the checked build; the checked
    build's status word must stay clear."""
    bind, normal, checked = libs
    with using(bind, normal):
        want = fn()
    with using(bind, checked):
        bind.vq_kernel_status(clear=True)
        got = fn()
        torch.cuda.synchronize()
        assert bind.vq_kernel_status() == 0
    return want, got


BITS = {torch.float16: torch.int16, torch.bfloat16: torch.int16, torch.float32: torch.int32,
        torch.uint32: torch.int32, torch.uint8: torch.uint8}


def same(want, got):
    """Bit-identical outputs (compared through integer views)."""
    assert want.dtype == got.dtype and want.shape == got.shape
    assert torch.equal(want.view(BITS[want.dtype]), got.view(BITS[got.dtype]))


def test_check_primitives_accept_and_reject_spans():
    import tc_harness

    lib = tc_harness.load()
    smem = 1024
    big = 1 << 40
    cases = [  # (kind, offset, bytes, region, accepted)
        (0, 0, 16, 0, True), (0, 1008, 16, 0, True), (0, 1016, 16, 0, False),
        (0, 1024, 0, 0, True), (0, 1024, 4, 0, False), (0, -16, 16, 0, False),
        (0, 4, 16, 0, False), (0, 4, 4, 0, True), (0, 2, 4, 0, False), (0, 1020, 8, 0, False),
        (0, 512, 512, 0, True), (0, 512, 513, 0, False),
        (1, 0, 4096, 4096, True), (1, 16, 4096, 4096, False), (1, 4088, 8, 4096, True),
        (1, 4092, 8, 4096, False), (1, -8, 8, 4096, False), (1, 6, 2, 8, True),
        (1, 6, 4, 8, False), (1, big, 8, 2 * big, True), (1, 2 * big, 1, 2 * big, False),
        (2, 5, 0, 6, True), (2, 6, 0, 6, False), (2, -1, 0, 6, False), (2, 0, 0, 0, False),
    ]
    dev = torch.device("cuda")
    kind = torch.tensor([c[0] for c in cases], dtype=torch.int32, device=dev)
    off = torch.tensor([c[1] for c in cases], dtype=torch.int64, device=dev)
    nbytes = torch.tensor([c[2] for c in cases], dtype=torch.int64, device=dev)
    region = torch.tensor([c[3] for c in cases], dtype=torch.int64, device=dev)
    gbuf = torch.zeros(16, dtype=torch.uint8, device=dev)
    result = torch.full((len(cases),), -1, dtype=torch.int32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    tc_harness.status("check", clear=True)
    assert lib.check_probe(kind.data_ptr(), off.data_ptr(), nbytes.data_ptr(), region.data_ptr(),
                           len(cases), gbuf.data_ptr(), result.data_ptr(), smem, stream) == 0
    got = result.cpu().tolist()
    assert got == [int(c[4]) for c in cases], [(c, g) for c, g in zip(cases, got) if int(c[4]) != g]
    assert tc_harness.status("check") & 2  # the rejected spans were recorded
    # only accepted spans: the word stays clear
    ok = [c for c in cases if c[4]]
    kind, off, nbytes, region = (torch.tensor([c[i] for c in ok], dtype=dt, device=dev)
                                 for i, dt in ((0, torch.int32), (1, torch.int64),
                                               (2, torch.int64), (3, torch.int64)))
    assert lib.check_probe(kind.data_ptr(), off.data_ptr(), nbytes.data_ptr(), region.data_ptr(),
                           len(ok), gbuf.data_ptr(), result.data_ptr(), smem, stream) == 0
    assert tc_harness.status("check") == 0


TDT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("sub", [4, 8])
@pytest.mark.parametrize("n_c", [33, 64, 100, 256, 300, 1000])
def test_encode_checked_matches(libs, dtype, sub, n_c):
    bind = libs[0]
    g = torch.Generator().manual_seed(7 * n_c + sub)
    for groups, m in [(1, 1), (1, 127), (1, 129), (3, 1000), (2, 128 * 7 + 5)]:
        x = torch.randn(groups, m, sub, generator=g).to(TDT[dtype]).cuda()
        cb = torch.randn(groups, n_c, sub, generator=g).to(TDT[dtype]).cuda()
        want, got = both(libs, lambda: bind.vq_encode_grouped(x, cb))
        same(want, got)
        if n_c <= 256:
            want, got = both(libs, lambda: bind.vq_encode_grouped_u8(x, cb))
            same(want, got)


def test_encode_general_paths_checked_match(libs):
    bind = libs[0]
    g = torch.Generator().manual_seed(3)
    # misaligned rows (one element in) and sub_dim 5 take the general kernel
    base = torch.randn(1 + 2000 * 8, generator=g).half().cuda()
    x = base[1:].view(1, 2000, 8)
    cb = torch.randn(1, 256, 8, generator=g).half().cuda()
    assert bind.vq_describe_launch(1, 2000, 256, 8, torch.float16, x.data_ptr()).startswith(
        "kernel=encode_general")
    want, got = both(libs, lambda: bind.vq_encode_grouped(x, cb))
    same(want, got)
    x5 = torch.randn(2, 777, 5, generator=g).half().cuda()
    cb5 = torch.randn(2, 99, 5, generator=g).half().cuda()
    want, got = both(libs, lambda: bind.vq_encode_grouped(x5, cb5))
    same(want, got)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("sub", [4, 8])
@pytest.mark.parametrize("n_c", [256, 300])
def test_smooth_checked_matches(libs, dtype, sub, n_c):
    bind = libs[0]
    g = torch.Generator().manual_seed(11 * n_c + sub)
    hd = 64
    m = (hd // sub) * 37
    x = torch.randn(3, m, sub, generator=g).to(TDT[dtype]).cuda()
    cb = torch.randn(3, n_c, sub, generator=g).to(TDT[dtype]).cuda()
    f = torch.exp(0.5 * torch.randn(3, hd, generator=g)).cuda()
    for ib in ((1, 4) if n_c <= 256 else (4,)):
        want, got = both(libs, lambda: bind.vq_encode_grouped_smooth(x, f, cb, hd, index_bytes=ib))
        same(want, got)


@pytest.mark.parametrize("sub", [3, 4, 8, 16])
def test_dequantize_checked_matches(libs, sub):
    bind = libs[0]
    g = torch.Generator().manual_seed(sub)
    cb = torch.randn(3, 200, sub, generator=g).half().cuda()
    idx = torch.randint(0, 256, (3, 1001), generator=g, dtype=torch.int32).cuda()  # some >= 200
    for codes in (idx.view(torch.uint32), idx.to(torch.uint8)):
        want, got = both(libs, lambda: bind.vq_dequantize_grouped(codes, cb))
        same(want, got)


ATTN = [  # (b, hq, hkv, tokens, head_dim, sub_dim, n_c, dtype, window)
    (2, 8, 8, 1, 128, 8, 256, "f16", 0),        # one head per KV head, one token
    (1, 16, 8, 255, 64, 16, 200, "bf16", 0),    # 4 sub-spaces, 200 centroids
    (2, 8, 2, 1000, 128, 8, 256, "f16", 300),   # 4 heads per KV head, window
    (1, 16, 2, 3001, 128, 4, 256, "f32", 0),    # 8 heads per KV head, 32 sub-spaces
    (3, 4, 2, 777, 256, 8, 100, "f16", 0),      # 2 heads per KV head
    (1, 8, 1, 2048, 512, 8, 256, "f16", 0),     # 64 sub-spaces
    (4, 32, 8, 5000, 128, 8, 256, "bf16", 0),   # the benchmark grouping
]


@pytest.mark.parametrize("shape", ATTN, ids=lambda s: "-".join(map(str, s)))
def test_attention_checked_matches(libs, shape):
    import test_attention as ta

    bind = libs[0]
    b, hq, hkv, t, d, sub, n_c, dtype, window = shape
    _, dev = ta.make_case(500 + t, b, hq, hkv, t, d, sub, n_c, dtype)
    want, got = both(libs, lambda: bind.vq_attention_decode(*dev, window=window))
    same(want, got)
    want, got = both(libs, lambda: bind.vq_attention_decode_static(*dev, window=window))
    same(want, got)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_scalar_checked_matches(libs, dtype):
    bind = libs[0]
    g = torch.Generator().manual_seed(5)
    x = torch.randn(8 * 4099 + 3, generator=g).to(TDT[dtype]).cuda()
    for n_c in (16, 100):
        c = torch.sort(torch.randn(n_c, generator=g)).values.cuda()
        for use_table in (True, False):
            want, got = both(libs, lambda: bind.vq_scalar_quantize(x, c, use_table=use_table))
            same(want, got)
        codes = bind.vq_scalar_quantize(x, c)
        want, got = both(libs, lambda: bind.vq_scalar_dequantize(codes, c, dtype=TDT[dtype]))
        same(want, got)
    # an odd offset: the element-by-element tail paths
    xo = x[1:]
    want, got = both(libs, lambda: bind.vq_scalar_quantize(xo, c))
    same(want, got)


@pytest.mark.parametrize("dim", [1, 2, 32, 64, 128, 256, 1024])
@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_hadamard_checked_matches(libs, dim, dtype):
    bind = libs[0]
    g = torch.Generator().manual_seed(dim)
    x = torch.randn(37, dim, generator=g).to(TDT[dtype]).cuda()
    diag = torch.where(torch.rand(dim, generator=g) < 0.5, -1.0, 1.0).cuda()
    want, got = both(libs, lambda: bind.vq_hadamard_rotate(x, diag))
    same(want, got)
    for n_c in (2, 16, 100):
        c = torch.sort(torch.randn(n_c, generator=g)).values.cuda()
        want, got = both(libs, lambda: bind.vq_hadamard_quantize(x, diag, c))
        same(want, got)

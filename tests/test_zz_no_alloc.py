"""fvx_sparse_conv_noalloc: the convolution for callers that cannot allocate
device memory while they run (for example a runtime whose device memory is
reserved once at load time).  Its scratch lives in a fixed array in the
library's device image instead of coming from an allocator.

Called here through the C ABI (ctypes) and compared with fvx_sparse_conv on
the same grids, kernel map and inputs, on two calls in a row (the second call
reuses the array the first one left behind).  This file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _grid_and_map(seed):
    import torch

    import sparse_convolution_gb300 as fvx

    rng = np.random.default_rng(seed)
    c = rng.integers(-30, 30, size=(12000, 3)).astype(np.int32)
    c = np.concatenate([c, c[:1500]])
    g = fvx.Grid.build(torch.from_numpy(c).cuda(), [0, 7000, len(c)])
    return g, fvx.KernelMap(g, g, 1)


def _call(fn, g, km, dt, x, W, out):
    import torch

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(g._h, g._h, km._h, dt, ctypes.c_void_p(x.data_ptr()), W.shape[1], ctypes.c_void_p(W.data_ptr()),
              W.shape[2], ctypes.c_void_p(out.data_ptr()), stream)


@pytest.mark.parametrize("cin,cout,out_bf16", [(8, 16, False), (64, 64, False), (128, 128, True), (16, 8, False),
                                              (24, 40, True)])
def test_noalloc_matches_allocating_conv(cuda_device, cin, cout, out_bf16):
    import torch

    import sparse_convolution_gb300 as fvx

    lib = fvx.load()
    g, km = _grid_and_map(cin + cout)
    dt = fvx.FVX_BF16_OUT_BF16 if out_bf16 else fvx.FVX_BF16
    odt = torch.bfloat16 if out_bf16 else torch.float32
    for call in range(2):  # two calls in a row: the shared array keeps the first call's contents
        gen = torch.Generator(device="cuda").manual_seed(100 * call + cin)
        x = torch.randn(g.n_active, cin, device="cuda", generator=gen).bfloat16()
        W = (torch.randn(27, cin, cout, device="cuda", generator=gen) / (27 * cin) ** 0.5).bfloat16()
        ref = torch.empty(g.n_active, cout, device="cuda", dtype=odt)
        got = torch.full((g.n_active, cout), float("nan"), device="cuda", dtype=odt)
        assert _call(lib.fvx_sparse_conv, g, km, dt, x, W, ref) == 0, lib.fvx_last_error()
        assert _call(lib.fvx_sparse_conv_noalloc, g, km, dt, x, W, got) == 0, lib.fvx_last_error()
        assert lib.fvx_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
        torch.cuda.synchronize()
        # same kernel and arithmetic: within the conv tolerance (2e-3 * sum|w*x|),
        # and in fact identical
        a = (x.float().abs().double().cpu().numpy(), W.float().abs().double().cpu().numpy())
        scale = np.zeros((g.n_active, cout))
        ii, oo, _ = (t.cpu().numpy() for t in km.pairs())
        for s in range(27):
            lo, hi = km.offsets[s], km.offsets[s + 1]
            np.add.at(scale, oo[lo:hi], a[0][ii[lo:hi]] @ a[1][s])
        err = np.abs(got.double().cpu().numpy() - ref.double().cpu().numpy())
        assert np.all(err <= 2e-3 * scale)
        assert torch.equal(got, ref)


def test_noalloc_fp32_and_limits(cuda_device):
    import torch

    import sparse_convolution_gb300 as fvx

    lib = fvx.load()
    g, km = _grid_and_map(7)
    x = torch.randn(g.n_active, 16, device="cuda")
    W = torch.randn(27, 16, 16, device="cuda") / 20.0
    ref = torch.empty(g.n_active, 16, device="cuda")
    got = torch.empty(g.n_active, 16, device="cuda")
    assert _call(lib.fvx_sparse_conv, g, km, fvx.FVX_F32, x, W, ref) == 0
    assert _call(lib.fvx_sparse_conv_noalloc, g, km, fvx.FVX_F32, x, W, got) == 0
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    # weights beyond the fixed scratch are refused before any device work
    xb = torch.zeros(g.n_active, 256, device="cuda", dtype=torch.bfloat16)
    Wb = torch.zeros(27, 256, 256, device="cuda", dtype=torch.bfloat16)
    ob = torch.empty(g.n_active, 256, device="cuda")
    assert _call(lib.fvx_sparse_conv_noalloc, g, km, fvx.FVX_BF16, xb, Wb, ob) == 2  # FVX_ERR_RANGE
    assert b"fixed" in lib.fvx_last_error()


def test_noalloc_leaf_kernel(cuda_device):
    """The leaf-densified kernel through the allocation-free entry point."""
    import torch

    import sparse_convolution_gb300 as fvx

    lib = fvx.load()
    g, km = _grid_and_map(5)
    fvx.set_conv_algo(fvx.FVX_CONV_LEAF)
    try:
        for call in range(2):
            gen = torch.Generator(device="cuda").manual_seed(200 + call)
            x = torch.randn(g.n_active, 16, device="cuda", generator=gen).bfloat16()
            W = (torch.randn(27, 16, 32, device="cuda", generator=gen) / 20.0).bfloat16()
            ref = torch.empty(g.n_active, 32, device="cuda")
            got = torch.full((g.n_active, 32), float("nan"), device="cuda")
            assert _call(lib.fvx_sparse_conv, g, km, fvx.FVX_BF16, x, W, ref) == 0, lib.fvx_last_error()
            assert _call(lib.fvx_sparse_conv_noalloc, g, km, fvx.FVX_BF16, x, W, got) == 0, lib.fvx_last_error()
            assert fvx.last_conv_algo() == fvx.FVX_CONV_LEAF
            torch.cuda.synchronize()
            assert torch.equal(got, ref)
    finally:
        fvx.set_conv_algo(fvx.FVX_CONV_AUTO)


def test_noalloc_halo_passes(cuda_device):
    """The halo-staged kernel through the allocation-free entry point, on a
    grid whose leaves hold enough outputs for the automatic choice to take
    it, with 64 input channels: two 32-channel launches, the second adding to
    the fp32 output; equal to the allocating call, twice in a row."""
    import torch

    import sparse_convolution_gb300 as fvx

    lib = fvx.load()
    rng = np.random.default_rng(11)
    c = rng.integers(-12, 12, size=(14000, 3)).astype(np.int32)  # about 64% of a 24^3 box
    g = fvx.Grid.build(torch.from_numpy(c).cuda(), [0, len(c)])
    km = fvx.KernelMap(g, g, 1)
    for call in range(2):
        gen = torch.Generator(device="cuda").manual_seed(300 + call)
        x = torch.randn(g.n_active, 64, device="cuda", generator=gen).bfloat16()
        W = (torch.randn(27, 64, 64, device="cuda", generator=gen) / 40.0).bfloat16()
        ref = torch.empty(g.n_active, 64, device="cuda")
        got = torch.full((g.n_active, 64), float("nan"), device="cuda")
        assert _call(lib.fvx_sparse_conv, g, km, fvx.FVX_BF16, x, W, ref) == 0, lib.fvx_last_error()
        assert fvx.last_conv_kernel() == "conv_halo"
        assert _call(lib.fvx_sparse_conv_noalloc, g, km, fvx.FVX_BF16, x, W, got) == 0, lib.fvx_last_error()
        assert fvx.last_conv_kernel() == "conv_halo"
        assert lib.fvx_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)


def test_noalloc_calls_no_allocator(cuda_device):
    """With an allocator installed that refuses every request and counts
    them, the no-alloc entry point (called here before any allocating
    convolution in this test) runs, is never asked for memory, and matches
    fvx_sparse_conv called afterwards with the default allocator."""
    import torch

    import sparse_convolution_gb300 as fvx

    lib = fvx.load()
    g, km = _grid_and_map(31)
    gen = torch.Generator(device="cuda").manual_seed(31)
    x = torch.randn(g.n_active, 32, device="cuda", generator=gen).bfloat16()
    W = (torch.randn(27, 32, 64, device="cuda", generator=gen) / 30.0).bfloat16()
    got = [torch.full((g.n_active, 64), float("nan"), device="cuda") for _ in range(2)]
    calls = []
    refuse = ALLOC_FN(lambda n, s, c: calls.append(n) or None)
    no_free = FREE_FN(lambda p, s, c: calls.append(-1))
    torch.cuda.synchronize()
    assert lib.fvx_set_allocator(ctypes.cast(refuse, ctypes.c_void_p), ctypes.cast(no_free, ctypes.c_void_p),
                                 None) == 0
    try:
        for out in got:  # two calls in a row
            assert _call(lib.fvx_sparse_conv_noalloc, g, km, fvx.FVX_BF16, x, W, out) == 0, lib.fvx_last_error()
            assert lib.fvx_noalloc_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
        torch.cuda.synchronize()
    finally:
        lib.fvx_set_allocator(None, None, None)
    assert calls == [], calls
    ref = torch.empty(g.n_active, 64, device="cuda")
    assert _call(lib.fvx_sparse_conv, g, km, fvx.FVX_BF16, x, W, ref) == 0, lib.fvx_last_error()
    torch.cuda.synchronize()
    assert torch.equal(got[0], ref) and torch.equal(got[1], ref)


def test_noalloc_empty_output_and_errors_match(cuda_device):
    """An empty output grid returns FVX_OK from both entry points, whatever
    the channel counts, as fvx_sparse_conv does."""
    import torch

    import sparse_convolution_gb300 as fvx

    lib = fvx.load()
    g = fvx.Grid.build(torch.zeros((0, 3), dtype=torch.int32, device="cuda"), [0, 0])
    km = fvx.KernelMap(g, g, 1)
    x = torch.zeros(1, 8, device="cuda", dtype=torch.bfloat16)
    W = torch.zeros(27, 8, 12, device="cuda", dtype=torch.bfloat16)  # 12: not a multiple of 8
    out = torch.zeros(1, 12, device="cuda")
    assert _call(lib.fvx_sparse_conv, g, km, fvx.FVX_BF16, x, W, out) == 0
    assert _call(lib.fvx_sparse_conv_noalloc, g, km, fvx.FVX_BF16, x, W, out) == 0

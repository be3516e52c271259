"""The halo-staged bf16 convolution (stride 1, 32 input channels per pass:
each output leaf's 10^3 input window fetched once into shared memory at the
positions that hold an input voxel, the operands of the leaf's active outputs
built from there, 128 outputs per tile; wider inputs in several passes that
add to the fp32 output) against the CPU oracle and against the direct
pair-list kernel, forced through fvx_set_conv_algo.

Narrow-band, random-sparse and solid grids (one to four tiles per leaf, tiles
that take the tail of one leaf and the head of the next, the persistent loop
over many leaves per block and the window pool wrapping around), two batches
with negative coordinates, unrelated input/output grids (windows with no input
voxel), cout 8 to 64 (including an MMA N padded past the stored columns), bf16
and fp32 output, the identity and single-offset stencils, the automatic choice
and the refusals.
"""
import numpy as np
import pytest

import oracle
from sparse_convolution_gb300 import synth
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


def _grid(seed, n, span, lo=-20, B=2):
    rng = np.random.default_rng(seed)
    c = rng.integers(lo, lo + span, size=(n, 3)).astype(np.int32)
    cuts = np.sort(rng.choice(np.arange(1, n), size=B - 1, replace=False)) if B > 1 else []
    return c, np.array([0, *cuts, n], np.int64)


def _solid(lo=-13, side=27):
    """A solid cube: every leaf inside holds 512 outputs (four tiles)."""
    ax = np.arange(lo, lo + side)
    c = np.stack(np.meshgrid(ax, ax, ax, indexing="ij"), -1).reshape(-1, 3).astype(np.int32)
    c = c[np.random.default_rng(9).permutation(len(c))]
    return c, np.array([0, len(c)], np.int64)


def _conv_with(algo, g, gout, km, x, W, out_dtype=None):
    import sparse_convolution_gb300 as fvx

    fvx.set_conv_algo(algo)
    try:
        y = fvx.sparse_conv(g, gout, km, x, W, out_dtype=out_dtype)
        kern = fvx.last_conv_kernel()
        fvx.device_status()
    finally:
        fvx.set_conv_algo(fvx.FVX_CONV_AUTO)
    return y, kern


def _coords(case):
    if case == "dense":
        return _grid(1, 30000, 28)
    if case == "sparse":  # ~10% occupancy: windows of a few dozen voxels
        return _grid(2, 25000, 64)
    if case == "solid":
        return _solid()
    w = synth.narrow_band(scale=0.06)
    return w["coords"], w["batch_offsets"]


@pytest.mark.parametrize("case,cout", [("band", 64), ("dense", 64), ("solid", 64), ("sparse", 64), ("band", 16),
                                       ("dense", 48), ("band", 8), ("solid", 24), ("sparse", 32)])
def test_halo_matches_oracle_and_direct(cuda_device, case, cout):
    import torch

    import sparse_convolution_gb300 as fvx

    coords, offs = _coords(case)
    g = G.gpu_grid(coords, offs)
    og = oracle.Grid.build(coords, offs)
    km = fvx.KernelMap(g, g, 1)
    okm = oracle.KernelMap(og, og, 1)
    x, W = G.bf16_inputs(32 + cout, g.n_active, 32, cout)
    y, kern = _conv_with(fvx.FVX_CONV_HALO, g, g, km, x, W)
    assert kern == "conv_halo" and fvx.last_conv_algo() == fvx.FVX_CONV_HALO
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y), yo, ao, G.BF16_TOL)
    yd, kd = _conv_with(fvx.FVX_CONV_DIRECT, g, g, km, x, W)
    assert kd == "conv_bf16_tma"
    G.assert_conv_close(G.np_(yd), yo, ao, G.BF16_TOL)
    # the same products, summed in fp32 in offset order by both kernels (the
    # direct kernel skips offsets absent from a whole tile): equal up to fp32
    # rounding (relative to sum|w*x|)
    assert np.all(np.abs(G.np_(y) - G.np_(yd)) <= 1e-5 * ao + 1e-30)
    yb, _ = _conv_with(fvx.FVX_CONV_HALO, g, g, km, x, W, out_dtype=torch.bfloat16)
    assert torch.equal(yb, y.bfloat16())


@pytest.mark.parametrize("case,cin,cout", [("band", 64, 64), ("dense", 64, 32), ("solid", 96, 64), ("sparse", 64, 48),
                                            ("band", 128, 16)])
def test_halo_passes_match_oracle_and_direct(cuda_device, case, cin, cout):
    """cin a multiple of 32 above 32: one pass per 32 input channels, the later
    passes adding to the fp32 output."""
    import torch

    import sparse_convolution_gb300 as fvx

    coords, offs = _coords(case)
    g = G.gpu_grid(coords, offs)
    og = oracle.Grid.build(coords, offs)
    km = fvx.KernelMap(g, g, 1)
    okm = oracle.KernelMap(og, og, 1)
    x, W = G.bf16_inputs(7 + cin + cout, g.n_active, cin, cout)
    y, kern = _conv_with(fvx.FVX_CONV_HALO, g, g, km, x, W)
    assert kern == "conv_halo" and y.dtype == torch.float32
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y), yo, ao, G.BF16_TOL)
    yd, kd = _conv_with(fvx.FVX_CONV_DIRECT, g, g, km, x, W)
    assert kd == "conv_bf16_tma"
    assert np.all(np.abs(G.np_(y) - G.np_(yd)) <= 1e-5 * ao + 1e-30)
    # the sum of the 32-channel passes, each run on its own
    parts = [_conv_with(fvx.FVX_CONV_HALO, g, g, km, x[:, c:c + 32].contiguous(), W[:, c:c + 32].contiguous())[0]
             for c in range(0, cin, 32)]
    acc = parts[0].clone()
    for p_ in parts[1:]:
        acc += p_
    assert torch.equal(acc, y)


def test_halo_unrelated_grids_and_identity(cuda_device):
    """Outputs whose windows hold no input voxel are zero; W[13] = I copies x."""
    import torch

    import sparse_convolution_gb300 as fvx

    a, oa = _grid(4, 6000, 30, lo=0, B=1)
    b, ob = _grid(5, 6000, 30, lo=200, B=1)  # far away: no output has a neighbour
    bo = np.concatenate([b, a[:500]])
    ga, gb = G.gpu_grid(a, oa), G.gpu_grid(bo, [0, len(bo)])
    km = fvx.KernelMap(ga, gb, 1)
    x, W = G.bf16_inputs(3, ga.n_active, 32, 64)
    y, kern = _conv_with(fvx.FVX_CONV_HALO, ga, gb, km, x, W)
    assert kern == "conv_halo"
    okm = oracle.KernelMap(oracle.Grid.build(a, oa), oracle.Grid.build(bo, np.array([0, len(bo)], np.int64)), 1)
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y), yo, ao, G.BF16_TOL)
    assert int((np.abs(yo).sum(1) == 0).sum()) > 1000 and np.all(G.np_(y)[np.abs(yo).sum(1) == 0] == 0)
    g = G.gpu_grid(a, oa)
    km2 = fvx.KernelMap(g, g, 1)
    Wi = torch.zeros(27, 32, 32, device="cuda", dtype=torch.bfloat16)
    Wi[13] = torch.eye(32, device="cuda", dtype=torch.bfloat16)
    xi = torch.randn(g.n_active, 32, device="cuda").bfloat16()
    yi, _ = _conv_with(fvx.FVX_CONV_HALO, g, g, km2, xi, Wi)
    assert torch.equal(yi, xi.float())


def test_halo_single_voxel_shift_stencils(cuda_device):
    """One-hot stencils: W[s] = I for a single offset s moves every feature by
    that offset (output p reads input p + d_s, zero where absent), on a grid
    that crosses leaf and window boundaries in every direction."""
    import torch

    import sparse_convolution_gb300 as fvx

    coords, offs = _grid(7, 9000, 34, lo=-17, B=1)
    g = G.gpu_grid(coords, offs)
    km = fvx.KernelMap(g, g, 1)
    ijk = G.np_(g.ijk()).astype(np.int64)
    index = {tuple(c): i for i, c in enumerate(ijk)}
    xi = torch.randn(g.n_active, 32, device="cuda").bfloat16()
    xh = xi.float().cpu().numpy()
    for s in (0, 5, 13, 21, 26):
        d = np.array([s // 9 - 1, (s // 3) % 3 - 1, s % 3 - 1])
        Wi = torch.zeros(27, 32, 32, device="cuda", dtype=torch.bfloat16)
        Wi[s] = torch.eye(32, device="cuda", dtype=torch.bfloat16)
        y, kern = _conv_with(fvx.FVX_CONV_HALO, g, g, km, xi, Wi)
        assert kern == "conv_halo"
        src = np.array([index.get(tuple(c + d), -1) for c in ijk])
        exp = np.where(src[:, None] >= 0, xh[np.maximum(src, 0)], 0.0)
        assert np.array_equal(G.np_(y), exp), s


def test_halo_auto_choice(cuda_device):
    import torch

    import sparse_convolution_gb300 as fvx

    w = synth.narrow_band(scale=0.06)
    g = G.gpu_grid(w["coords"], w["batch_offsets"])
    km = fvx.KernelMap(g, g, 1)
    x, W = G.bf16_inputs(1, g.n_active, 32, 64)
    _, kern = _conv_with(fvx.FVX_CONV_AUTO, g, g, km, x, W)
    assert kern == "conv_halo"  # about 100 outputs per leaf
    x64, W64 = G.bf16_inputs(1, g.n_active, 64, 64)
    _, kern = _conv_with(fvx.FVX_CONV_AUTO, g, g, km, x64, W64)
    assert kern == "conv_halo"  # two 32-channel passes, fp32 output
    _, kern = _conv_with(fvx.FVX_CONV_AUTO, g, g, km, x64, W64, out_dtype=torch.bfloat16)
    assert kern == "conv_bf16_tma"
    _, kern = _conv_with(fvx.FVX_CONV_GATHER, g, g, km, x, W)
    assert kern == "conv_bf16_tma"
    coords, offs = _grid(2, 4000, 120)  # a few outputs per leaf
    gs = G.gpu_grid(coords, offs)
    kms = fvx.KernelMap(gs, gs, 1)
    xs, Ws = G.bf16_inputs(1, gs.n_active, 32, 64)
    _, kern = _conv_with(fvx.FVX_CONV_AUTO, gs, gs, kms, xs, Ws)
    assert kern == "conv_bf16_tma"


def test_halo_refusals(cuda_device):
    import torch

    import sparse_convolution_gb300 as fvx

    coords, offs = _grid(6, 3000, 20, B=1)
    g = G.gpu_grid(coords, offs)
    km = fvx.KernelMap(g, g, 1)
    for cin, cout, od in [(16, 32, None), (48, 64, None), (32, 128, None), (32, 256, None),
                          (64, 64, torch.bfloat16)]:
        x, W = G.bf16_inputs(1, g.n_active, cin, cout)
        with pytest.raises(fvx.FvxError) as e:
            _conv_with(fvx.FVX_CONV_HALO, g, g, km, x, W, out_dtype=od)
        assert e.value.status == "FVX_ERR_INVALID_ARG"
    x, W = G.bf16_inputs(1, g.n_active, 32, 32)
    coarse = g.coarsen(2)
    for kmap, gi, go in [(fvx.KernelMap(g, coarse, 2), g, coarse), (fvx.KernelMap(g, g, 1, transposed=True), g, g)]:
        with pytest.raises(fvx.FvxError) as e:
            _conv_with(fvx.FVX_CONV_HALO, gi, go, kmap, x, W)
        assert e.value.status == "FVX_ERR_INVALID_ARG"

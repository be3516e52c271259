"""The union-staged pair-list convolution (each distinct input row of a tile
fetched once into shared memory, the tensor-core operands built from there)
against the CPU oracle and against the direct pair-list kernel, forced through
fvx_set_conv_algo.

Dense and narrow-band grids (unions of a few hundred rows per tile), sparse
grids whose tiles need more distinct rows than a union buffer holds (the tile
is split into groups of offsets), stride-2 and transposed maps, cin 32 and 64,
cout 8 to 128, empty tiles, bf16 and fp32 output.
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


@pytest.mark.parametrize("case,cin,cout", [("dense", 32, 64), ("dense", 64, 64), ("dense", 64, 128),
                                           ("sparse", 64, 64), ("sparse", 32, 16), ("band", 32, 64),
                                           ("band", 64, 8), ("sparse", 64, 128)])
def test_union_matches_oracle_and_direct(cuda_device, case, cin, cout):
    import sparse_convolution_gb300 as fvx

    if case == "dense":
        coords, offs = _grid(1, 30000, 28)
    elif case == "sparse":  # ~10% occupancy: a tile names over a thousand distinct rows
        coords, offs = _grid(2, 25000, 64)
    else:
        w = synth.narrow_band(scale=0.06)
        coords, offs = w["coords"], w["batch_offsets"]
    g = G.gpu_grid(coords, offs)
    og = oracle.Grid.build(coords, offs)
    km = fvx.KernelMap(g, g, 1)
    okm = oracle.KernelMap(og, og, 1)
    x, W = G.bf16_inputs(cin + cout, g.n_active, cin, cout)
    y, kern = _conv_with(fvx.FVX_CONV_UNION, g, g, km, x, W)
    assert kern == "conv_union"
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y), yo, ao, G.BF16_TOL)
    yd, kd = _conv_with(fvx.FVX_CONV_DIRECT, g, g, km, x, W)
    assert kd == "conv_bf16_tma"
    G.assert_conv_close(G.np_(yd), yo, ao, G.BF16_TOL)
    assert (yd == y).all()  # same products, same order of accumulation
    # bf16 output: the fp32 result rounded
    yb, _ = _conv_with(fvx.FVX_CONV_UNION, g, g, km, x, W, out_dtype=__import__("torch").bfloat16)
    assert (yb == y.bfloat16()).all()


@pytest.mark.parametrize("stride,transposed", [(2, False), (2, True), (1, True)])
def test_union_strided_and_transposed_maps(cuda_device, stride, transposed):
    import sparse_convolution_gb300 as fvx

    coords, offs = _grid(3, 20000, 40, lo=-19)
    fine = G.gpu_grid(coords, offs)
    ofine = oracle.Grid.build(coords, offs)
    coarse = fine if stride == 1 else fine.coarsen(2)
    ocoarse = ofine if stride == 1 else ofine.coarsen(2)
    gi, go = (coarse, fine) if transposed else (fine, coarse)
    ogi, ogo = (ocoarse, ofine) if transposed else (ofine, ocoarse)
    km = fvx.KernelMap(gi, go, stride, transposed=transposed)
    okm = oracle.KernelMap(ogi, ogo, stride, transposed=transposed)
    x, W = G.bf16_inputs(7, gi.n_active, 64, 32)
    y, kern = _conv_with(fvx.FVX_CONV_UNION, gi, go, km, x, W)
    assert kern == "conv_union"
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y), yo, ao, G.BF16_TOL)


def test_union_unrelated_grids_and_identity(cuda_device):
    """Outputs with no pairs (all-empty tiles) are zero; W[13] = I copies x."""
    import torch

    import sparse_convolution_gb300 as fvx

    a, oa = _grid(4, 6000, 30, lo=0, B=1)
    b, ob = _grid(5, 6000, 30, lo=200, B=1)  # far away: no output has a neighbour
    ga, gb = G.gpu_grid(a, oa), G.gpu_grid(np.concatenate([b, a[:500]]), [0, len(b) + 500])
    km = fvx.KernelMap(ga, gb, 1)
    x, W = G.bf16_inputs(3, ga.n_active, 32, 64)
    y, _ = _conv_with(fvx.FVX_CONV_UNION, ga, gb, km, x, W)
    ogb = oracle.Grid.build(np.concatenate([b, a[:500]]), np.array([0, len(b) + 500], np.int64))
    okm = oracle.KernelMap(oracle.Grid.build(a, oa), ogb, 1)
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y), yo, ao, G.BF16_TOL)
    g = G.gpu_grid(a, oa)
    km2 = fvx.KernelMap(g, g, 1)
    Wi = torch.zeros(27, 64, 64, device="cuda", dtype=torch.bfloat16)
    Wi[13] = torch.eye(64, device="cuda", dtype=torch.bfloat16)
    xi = torch.randn(g.n_active, 64, device="cuda").bfloat16()
    yi, _ = _conv_with(fvx.FVX_CONV_UNION, g, g, km2, xi, Wi)
    assert torch.equal(yi, xi.float())


def test_union_refusals(cuda_device):
    import sparse_convolution_gb300 as fvx

    coords, offs = _grid(6, 3000, 20, B=1)
    g = G.gpu_grid(coords, offs)
    km = fvx.KernelMap(g, g, 1)
    for cin, cout in [(16, 32), (128, 64), (32, 256)]:
        x, W = G.bf16_inputs(1, g.n_active, cin, cout)
        with pytest.raises(fvx.FvxError) as e:
            _conv_with(fvx.FVX_CONV_UNION, g, g, km, x, W)
        assert e.value.status == "FVX_ERR_INVALID_ARG"
    x, W = G.bf16_inputs(1, g.n_active, 64, 64)
    _, kern = _conv_with(fvx.FVX_CONV_AUTO, g, g, km, x, W)
    assert kern == "conv_halo"  # the automatic choice never takes the union-staged kernel (here: two halo passes)
    x, W = G.bf16_inputs(1, g.n_active, 32, 64)
    _, kern = _conv_with(fvx.FVX_CONV_AUTO, g, g, km, x, W)
    assert kern == "conv_halo"  # 32 channels on leaves this full: the halo-staged kernel

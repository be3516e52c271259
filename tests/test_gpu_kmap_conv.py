"""GPU kernel map and sparse conv vs the CPU oracle.

Kernel map: bit-exact ("DriveRT", Shared neighbour maps).  Conv: within
2e-3 * sum|w*x| per output element for bf16 (bf16-rounded inputs, fp32
accumulation, fp32 output; a bf16 output adds one 2^-8 |y| rounding) and
1e-5 * sum|w*x| for fp32 ("fVDB: A Deep-Learning Framework for Sparse, Large
Scale, and High Performance Spatial Intelligence" notes, Sparse-convolution
operators)."""
import numpy as np
import pytest

import oracle
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


def _random(seed, n, lo, span, B, dup=0.1):
    rng = np.random.default_rng(seed)
    rows, offs = [], [0]
    for _ in range(B):
        c = rng.integers(lo, lo + span, size=(n, 3)).astype(np.int32)
        c = np.concatenate([c, c[rng.integers(0, n, size=int(dup * n))]])
        rows.append(c[rng.permutation(len(c))])
        offs.append(offs[-1] + len(c))
    return np.concatenate(rows), np.array(offs, np.int64)


@pytest.fixture(scope="module")
def grids():
    c, offs = _random(3, 9000, -25, 50, 2)
    import sparse_convolution_gb300 as fvx  # noqa: F401

    g = G.gpu_grid(c, offs)
    og = oracle.Grid.build(c, offs)
    gc = g.coarsen(2)
    ogc = og.coarsen(2)
    return dict(g=g, og=og, gc=gc, ogc=ogc)


def _maps(grids, stride):
    import sparse_convolution_gb300 as fvx

    if stride == 1:
        return grids["g"], grids["g"], fvx.KernelMap(grids["g"], grids["g"], 1), oracle.KernelMap(
            grids["og"], grids["og"], 1)
    return grids["g"], grids["gc"], fvx.KernelMap(grids["g"], grids["gc"], 2), oracle.KernelMap(
        grids["og"], grids["ogc"], 2)


@pytest.mark.parametrize("stride", [1, 2])
def test_kmap_matches_oracle(cuda_device, grids, stride):
    _, _, km, okm = _maps(grids, stride)
    G.assert_kmap_equal(km, okm)


def test_kmap_between_unrelated_grids(cuda_device):
    """Stride-1 map from one grid to a different output grid: outputs far from
    every input get no pairs (and a zero conv output)."""
    import sparse_convolution_gb300 as fvx

    a, oa = _random(41, 3000, 0, 30, 1)
    b, ob = _random(42, 3000, 20, 40, 1)
    ga, gb = G.gpu_grid(a, oa), G.gpu_grid(b, ob)
    oga, ogb = oracle.Grid.build(a, oa), oracle.Grid.build(b, ob)
    km = fvx.KernelMap(ga, gb, 1)
    okm = oracle.KernelMap(oga, ogb, 1)
    G.assert_kmap_equal(km, okm)
    x, W = G.bf16_inputs(5, ga.n_active, 16, 32)
    y = fvx.sparse_conv(ga, gb, km, x, W)
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    assert (okm.mask == 0).any()
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL)
    assert np.all(G.np_(y.float())[okm.mask == 0] == 0)


@pytest.mark.parametrize("cin,cout", [(16, 16), (5, 7), (3, 33), (32, 8)])
@pytest.mark.parametrize("stride", [1, 2])
def test_conv_f32_matches_oracle(cuda_device, grids, stride, cin, cout):
    import torch

    import sparse_convolution_gb300 as fvx
    from sparse_convolution_gb300 import synth

    gin, gout, km, okm = _maps(grids, stride)
    x = torch.from_numpy(synth.features(7, gin.n_active, cin, "uniform")).cuda()
    W = torch.from_numpy(synth.weights(8, cin, cout)).cuda()
    y = fvx.sparse_conv(gin, gout, km, x, W)
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y), yo, ao, G.F32_TOL)


# cin a multiple of 16 takes the TMA-fed kernel (16/32/64-channel chunks:
# 48 -> 3 x 16, 96 -> 3 x 32, 80 -> 5 x 16); other multiples of 8 the
# cp.async kernel (8, 24, 40).
@pytest.mark.parametrize("cin,cout", [(8, 16), (16, 32), (32, 64), (64, 64), (128, 128), (128, 256), (24, 48),
                                      (256, 16), (48, 32), (96, 64), (80, 16), (40, 32), (512, 32), (16, 256),
                                      (16, 8), (64, 24), (8, 8), (24, 40), (128, 136)])
@pytest.mark.parametrize("stride", [1, 2])
def test_conv_bf16_matches_oracle(cuda_device, grids, stride, cin, cout):
    import sparse_convolution_gb300 as fvx

    gin, gout, km, okm = _maps(grids, stride)
    x, W = G.bf16_inputs(11, gin.n_active, cin, cout)
    y = fvx.sparse_conv(gin, gout, km, x, W)
    fvx.device_status()
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL)


@pytest.fixture(scope="module")
def many_tiles():
    """About 66k voxels in two batches: several hundred 128-row output tiles,
    so every block of the persistent conv runs several tiles and cycles both
    of its row-table buffers and its stage ring more than once."""
    import sparse_convolution_gb300 as fvx

    c, offs = _random(8, 40000, -30, 60, 2)
    g = G.gpu_grid(c, offs)
    og = oracle.Grid.build(c, offs)
    assert g.n_active > 4 * 128 * 152 // 2
    return g, og, fvx.KernelMap(g, g, 1), oracle.KernelMap(og, og, 1)


@pytest.mark.parametrize("cin,cout", [(8, 16), (24, 16), (16, 16), (32, 32), (48, 16), (64, 64)])
def test_conv_bf16_many_tiles(cuda_device, many_tiles, cin, cout):
    import sparse_convolution_gb300 as fvx

    g, og, km, okm = many_tiles
    x, W = G.bf16_inputs(23, g.n_active, cin, cout)
    y = fvx.sparse_conv(g, g, km, x, W)
    fvx.device_status()
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL)


@pytest.mark.parametrize("cin,cout", [(8, 16), (64, 64), (128, 256), (16, 8), (32, 24)])
@pytest.mark.parametrize("stride", [1, 2])
def test_conv_bf16_out_bf16_matches_oracle(cuda_device, grids, stride, cin, cout):
    """bf16-rounded output: the stated bound plus one bf16 rounding of y."""
    import torch

    import sparse_convolution_gb300 as fvx

    gin, gout, km, okm = _maps(grids, stride)
    x, W = G.bf16_inputs(19, gin.n_active, cin, cout)
    y = fvx.sparse_conv(gin, gout, km, x, W, out_dtype=torch.bfloat16)
    assert y.dtype == torch.bfloat16
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL, rel_y=G.BF16_OUT_REL)
    # and it is the fp32-output result rounded to nearest bf16
    y32 = fvx.sparse_conv(gin, gout, km, x, W)
    assert torch.equal(y, y32.bfloat16())


@pytest.mark.parametrize("c", [16, 32, 48, 64, 96])
def test_conv_bf16_identity_is_exact(cuda_device, grids, c):
    """W[13] = I, other offsets 0: out == feats bit for bit (every channel
    lands where the operand layout says, for each gather width)."""
    import torch

    import sparse_convolution_gb300 as fvx

    g = grids["g"]
    km = fvx.KernelMap(g, g, 1)
    x, _ = G.bf16_inputs(13, g.n_active, c, c)
    W = torch.zeros((27, c, c), dtype=torch.bfloat16, device="cuda")
    W[13] = torch.eye(c, dtype=torch.bfloat16, device="cuda")
    y = fvx.sparse_conv(g, g, km, x, W)
    assert torch.equal(y, x.float())
    assert torch.equal(fvx.sparse_conv(g, g, km, x, W, out_dtype=torch.bfloat16), x)


def test_conv_bf16_repeatable(cuda_device, grids):
    import torch

    import sparse_convolution_gb300 as fvx

    gin, gout, km, _ = _maps(grids, 1)
    x, W = G.bf16_inputs(17, gin.n_active, 64, 128)
    y1 = fvx.sparse_conv(gin, gout, km, x, W)
    y2 = fvx.sparse_conv(gin, gout, km, x, W)
    assert torch.equal(y1, y2)


def test_conv_rejects_bad_shapes(cuda_device, grids):
    import torch

    import sparse_convolution_gb300 as fvx

    gin, gout, km, _ = _maps(grids, 1)
    x = torch.zeros((gin.n_active, 12), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((27, 12, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fvx.FvxError, match="FVX_ERR_INVALID_ARG"):
        fvx.sparse_conv(gin, gout, km, x, W)
    x2 = torch.zeros((gin.n_active, 16), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((27, 16, 16), dtype=torch.bfloat16, device="cuda")
    km2 = fvx.KernelMap(grids["g"], grids["gc"], 2)
    with pytest.raises(fvx.FvxError, match="other grids"):
        fvx.sparse_conv(gin, gout, km2, x2, W2)


_EXACT_PATH_CHILD = r"""
import numpy as np, oracle
from tests import gpu_common as G
from tests.test_gpu_kmap_conv import _random
import sparse_convolution_gb300 as fvx
c, offs = _random(5, 4000, -20, 40, 2)
g, og = G.gpu_grid(c, offs), oracle.Grid.build(c, offs)
for stride in (1, 2):
    gout, ogout = (g, og) if stride == 1 else (g.coarsen(2), og.coarsen(2))
    km, okm = fvx.KernelMap(g, gout, stride), oracle.KernelMap(og, ogout, stride)
    G.assert_kmap_equal(km, okm)
    x, W = G.bf16_inputs(7, g.n_active, 16, 32)
    y = fvx.sparse_conv(g, gout, km, x, W)
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL)
print("exact path ok")
"""


def test_kmap_exact_size_path(cuda_device):
    """With the capacity limit at 0 the map reads its pair count back and sizes
    its lists exactly (the path of maps past the limit): same map, same conv.
    A child process, since the limit is read once per process."""
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, FVX_KMAP_CAP_BYTES="0")
    r = subprocess.run([sys.executable, "-c", _EXACT_PATH_CHILD], env=env, cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "exact path ok" in r.stdout


@pytest.mark.parametrize("stride", [1, 2])
@pytest.mark.parametrize("transposed", [False, True])
def test_kmap_int32_edges(cuda_device, stride, transposed):
    """Voxels at both ends of the int32 range in one batch: a neighbour past an
    end is no voxel, so the two ends never pair (no wrap-around)."""
    import sparse_convolution_gb300 as fvx

    M = 2 ** 31 - 1
    c = np.array([[M, 0, 0], [-M - 1, 0, 0], [M - 1, 0, 0], [M, M, M], [-M - 1, -M - 1, -M - 1],
                  [-M - 1, M, 0], [M, -M - 1, 5], [M - 8, 3, 3], [-M + 7, 3, 3]], np.int32)
    g, og = G.gpu_grid(c, [0, len(c)]), oracle.Grid.build(c, [0, len(c)])
    gc, ogc = (g, og) if stride == 1 else (g.coarsen(2), og.coarsen(2))
    if transposed:
        km, okm = fvx.KernelMap(gc, g, stride, transposed=True), oracle.KernelMap(ogc, og, stride, transposed=True)
    else:
        km, okm = fvx.KernelMap(g, gc, stride), oracle.KernelMap(og, ogc, stride)
    G.assert_kmap_equal(km, okm)

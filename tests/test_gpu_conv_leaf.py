"""The leaf-densified bf16 convolution (fVDB reading notes, "Sparse-convolution
operators": the leaf backend densifies each 8^3 leaf plus a one-voxel halo in
shared memory and runs the stencil as dense tensor-core GEMMs).

Forced through fvx_set_conv_algo and compared with the CPU oracle within the
bf16 bound (2e-3 * sum|w*x| per output element), on sparse and dense grids,
two batches, unrelated input/output grids and the exact special cases; the
automatic choice and the refusals are checked too."""
import numpy as np
import pytest

import oracle
from sparse_convolution_gb300 import synth
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_algo():
    yield
    import sparse_convolution_gb300 as fvx

    fvx.set_conv_algo(fvx.FVX_CONV_AUTO)


def _random(seed, n, lo, span, B, dup=0.1):
    rng = np.random.default_rng(seed)
    rows, offs = [], [0]
    for _ in range(B):
        c = rng.integers(lo, lo + span, size=(n, 3)).astype(np.int32)
        c = np.concatenate([c, c[rng.integers(0, n, size=int(dup * n))]])
        rows.append(c[rng.permutation(len(c))])
        offs.append(offs[-1] + len(c))
    return np.concatenate(rows), np.array(offs, np.int64)


def _dense(seed):
    """Leaf-dense geometry (solid ellipsoids plus a solid 20^3 cube, about 30%
    mean leaf occupancy with full leaves among them), shifted to straddle zero
    so that negative leaves occur, in two batches (the second shifted by a
    vector that is not a multiple of the leaf size)."""
    w = synth.leaf_dense(seed=seed, scale=0.25)
    g = np.stack(np.meshgrid(*[np.arange(20, 40)] * 3, indexing="ij"), -1).reshape(-1, 3).astype(np.int32)
    c = np.unique(np.concatenate([w["coords"], g]), axis=0) - 30
    c = c[np.random.default_rng(seed).permutation(len(c))]
    c1 = c + np.array([3, -5, 7], np.int32)
    return np.concatenate([c, c1]), np.array([0, len(c), 2 * len(c)], np.int64)


def _case(coords, offs):
    import sparse_convolution_gb300 as fvx

    g = G.gpu_grid(coords, offs)
    og = oracle.Grid.build(coords, offs)
    return g, og, fvx.KernelMap(g, g, 1), oracle.KernelMap(og, og, 1)


@pytest.fixture(scope="module")
def sparse_case():
    return _case(*_random(3, 9000, -25, 50, 2))


@pytest.fixture(scope="module")
def dense_case():
    return _case(*_dense(12))


def _check(case, cin, cout, seed=31, out_bf16=False):
    import torch

    import sparse_convolution_gb300 as fvx

    g, og, km, okm = case
    x, W = G.bf16_inputs(seed, g.n_active, cin, cout)
    fvx.set_conv_algo(fvx.FVX_CONV_LEAF)
    y = fvx.sparse_conv(g, g, km, x, W, out_dtype=torch.bfloat16 if out_bf16 else None)
    fvx.device_status()
    assert fvx.last_conv_algo() == fvx.FVX_CONV_LEAF
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL, rel_y=G.BF16_OUT_REL if out_bf16 else 0.0)
    return y, x, W


@pytest.mark.parametrize("cin,cout", [(8, 16), (16, 16), (8, 64), (16, 64), (16, 32), (8, 48)])
def test_leaf_matches_oracle_dense(cuda_device, dense_case, cin, cout):
    g = dense_case[0]
    assert g.n_active >= 0.2 * 512 * g.n_leaf  # the geometry the backend is for
    _check(dense_case, cin, cout)


@pytest.mark.parametrize("cin,cout", [(8, 16), (16, 32)])
def test_leaf_matches_oracle_sparse(cuda_device, sparse_case, cin, cout):
    _check(sparse_case, cin, cout)


def test_leaf_bf16_output_is_rounded_fp32(cuda_device, dense_case):
    import torch

    import sparse_convolution_gb300 as fvx

    yb, x, W = _check(dense_case, 8, 16, out_bf16=True)
    g, _, km, _ = dense_case
    fvx.set_conv_algo(fvx.FVX_CONV_LEAF)
    y32 = fvx.sparse_conv(g, g, km, x, W)
    assert torch.equal(yb, y32.bfloat16())


def test_leaf_agrees_with_gather(cuda_device, dense_case):
    """Same inputs through both kernel families: each within the bound of the
    oracle (above); here the two differ by at most the sum of both bounds."""
    import sparse_convolution_gb300 as fvx

    g, og, km, okm = dense_case
    x, W = G.bf16_inputs(41, g.n_active, 16, 32)
    fvx.set_conv_algo(fvx.FVX_CONV_LEAF)
    yl = G.np_(fvx.sparse_conv(g, g, km, x, W))
    fvx.set_conv_algo(fvx.FVX_CONV_GATHER)
    yg = G.np_(fvx.sparse_conv(g, g, km, x, W))
    assert fvx.last_conv_algo() == fvx.FVX_CONV_GATHER
    _, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    assert np.all(np.abs(yl - yg) <= 2 * G.BF16_TOL * ao)


@pytest.mark.parametrize("c", [8, 16])
def test_leaf_identity_is_exact(cuda_device, dense_case, c):
    """W[13] = I, other offsets 0: out == feats bit for bit."""
    import torch

    import sparse_convolution_gb300 as fvx

    g, _, km, _ = dense_case
    x, _ = G.bf16_inputs(13, g.n_active, c, 16)
    W = torch.zeros((27, c, 16), dtype=torch.bfloat16, device="cuda")
    W[13, :, :c] = torch.eye(c, dtype=torch.bfloat16, device="cuda")
    fvx.set_conv_algo(fvx.FVX_CONV_LEAF)
    y = fvx.sparse_conv(g, g, km, x, W)
    ref = torch.zeros((g.n_active, 16), device="cuda")
    ref[:, :c] = x.float()
    assert torch.equal(y, ref)


def test_leaf_single_offset_shift_is_exact(cuda_device, dense_case):
    """W[s] = I for one off-centre slot s: out[q] = feats[p] for the pair (p, q)
    of list s and 0 where q has none, bit for bit."""
    import torch

    import sparse_convolution_gb300 as fvx

    g, _, km, okm = dense_case
    x, _ = G.bf16_inputs(14, g.n_active, 8, 16)
    for s in (0, 5, 22, 26):
        W = torch.zeros((27, 8, 16), dtype=torch.bfloat16, device="cuda")
        W[s, :, :8] = torch.eye(8, dtype=torch.bfloat16, device="cuda")
        fvx.set_conv_algo(fvx.FVX_CONV_LEAF)
        y = G.np_(fvx.sparse_conv(g, g, km, x, W))
        ref = np.zeros((g.n_active, 16), np.float32)
        lo, hi = okm.offsets[s], okm.offsets[s + 1]
        ref[okm.out_idx[lo:hi], :8] = G.np_(x.float())[okm.in_idx[lo:hi]]
        assert np.array_equal(y, ref), s


def test_leaf_between_unrelated_grids(cuda_device):
    import sparse_convolution_gb300 as fvx

    a, oa = _dense(21)
    b, ob = _dense(22)
    b = b + np.array([4, 0, -3], np.int32)
    ga, gb = G.gpu_grid(a, oa), G.gpu_grid(b, ob)
    oga, ogb = oracle.Grid.build(a, oa), oracle.Grid.build(b, ob)
    km = fvx.KernelMap(ga, gb, 1)
    okm = oracle.KernelMap(oga, ogb, 1)
    x, W = G.bf16_inputs(5, ga.n_active, 16, 32)
    fvx.set_conv_algo(fvx.FVX_CONV_LEAF)
    y = fvx.sparse_conv(ga, gb, km, x, W)
    assert fvx.last_conv_algo() == fvx.FVX_CONV_LEAF
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL)


def test_auto_choice(cuda_device, dense_case, sparse_case):
    import torch

    import sparse_convolution_gb300 as fvx

    for case, want in ((dense_case, fvx.FVX_CONV_LEAF), (sparse_case, fvx.FVX_CONV_GATHER)):
        g, _, km, _ = case
        x, W = G.bf16_inputs(3, g.n_active, 8, 16)
        fvx.sparse_conv(g, g, km, x, W)
        assert fvx.last_conv_algo() == want
    g, _, km, _ = dense_case
    x, W = G.bf16_inputs(3, g.n_active, 32, 32)  # too many channels for the leaf kernel: the halo-staged one
    fvx.sparse_conv(g, g, km, x, W)
    assert fvx.last_conv_algo() == fvx.FVX_CONV_HALO
    x, W = G.bf16_inputs(3, g.n_active, 64, 32)  # fp32 output: two halo-staged passes of 32 channels
    fvx.sparse_conv(g, g, km, x, W)
    assert fvx.last_conv_algo() == fvx.FVX_CONV_HALO
    fvx.sparse_conv(g, g, km, x, W, out_dtype=torch.bfloat16)  # bf16 output: pair lists
    assert fvx.last_conv_algo() == fvx.FVX_CONV_GATHER


def test_leaf_refusals(cuda_device, dense_case):
    import sparse_convolution_gb300 as fvx

    g, _, km, _ = dense_case
    fvx.set_conv_algo(fvx.FVX_CONV_LEAF)
    x, W = G.bf16_inputs(3, g.n_active, 32, 16)
    with pytest.raises(fvx.FvxError, match="leaf-densified"):
        fvx.sparse_conv(g, g, km, x, W)
    x, W = G.bf16_inputs(3, g.n_active, 8, 128)
    with pytest.raises(fvx.FvxError, match="leaf-densified"):
        fvx.sparse_conv(g, g, km, x, W)
    x, W = G.bf16_inputs(3, g.n_active, 8, 8)  # N = 8 is padded to 16 by the pair-list kernels only
    with pytest.raises(fvx.FvxError, match="leaf-densified"):
        fvx.sparse_conv(g, g, km, x, W)
    gc = g.coarsen(2)
    km2 = fvx.KernelMap(g, gc, 2)
    x, W = G.bf16_inputs(3, g.n_active, 8, 16)
    with pytest.raises(fvx.FvxError, match="leaf-densified"):
        fvx.sparse_conv(g, gc, km2, x, W)
    with pytest.raises(fvx.FvxError):
        fvx.set_conv_algo(7)

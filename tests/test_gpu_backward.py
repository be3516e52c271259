"""GPU transposed kernel map, refined grid, transposed convolution and the
backward pass (input and weight gradients) vs the CPU oracle.

Topology and kernel maps: bit-exact ("fVDB" ONNX operator list, §1.2
RefinedGrid / ConvTransposeGrid).  Transposed convolution and input gradient
run the forward convolution kernels, so they meet the same bounds: 2e-3 *
sum|w*x| (bf16) and 1e-5 * sum|w*x| (fp32) per element.  The weight gradient:
fp32 inputs run exact fp32 FFMA, 1e-5 * sum|x*dy| per element; bf16 inputs
(the oracle is fed the same bf16-rounded values) run the tensor cores with
fp32 accumulation when both channel counts are multiples of 64 (otherwise
fp32 FFMA), and meet the bf16 bound 2e-3 * sum|x*dy|.  Training computes its gradients through the pair-list
backend ("fVDB" reading notes, Limitations and future work)."""
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
    """Fine grid (two batches, odd and negative coordinates), its stride-2
    coarse grid and the coarse grid's refinement."""
    c, offs = _random(5, 9000, -25, 50, 2)
    g = G.gpu_grid(c, offs)
    og = oracle.Grid.build(c, offs)
    gc, ogc = g.coarsen(2), og.coarsen(2)
    return dict(g=g, og=og, gc=gc, ogc=ogc, gr=gc.refine(2), ogr=ogc.refine(2))


# ---------------------------------------------------------------- refined grid

@pytest.mark.parametrize("factor", [1, 2, 3])
def test_refine_matches_oracle(cuda_device, grids, factor):
    G.assert_topology_equal(grids["gc"].refine(factor), grids["ogc"].refine(factor))


def test_refine_of_coarsened_covers_fine(cuda_device, grids):
    """Every fine voxel is a child of its coarse parent, so refine(coarsen(g))
    contains g, with 8 children per coarse voxel."""
    import torch

    g, gr = grids["g"], grids["gr"]
    assert gr.n_active == 8 * grids["gc"].n_active
    b = np.repeat(np.arange(g.batch_size), np.diff(g.batch_offsets())).astype(np.int32)
    idx = gr.lookup(g.ijk(), torch.from_numpy(b).cuda())
    assert int((idx < 0).sum()) == 0


def test_refine_empty(cuda_device):
    g = G.gpu_grid(np.zeros((0, 3), np.int32), [0, 0])
    r = g.refine(2)
    assert r.n_active == 0 and r.batch_size == 1


def test_refine_coordinate_overflow_is_reported(cuda_device):
    """A child beyond int32 is an error, not a wrapped coordinate."""
    import sparse_convolution_gb300 as fvx

    g = G.gpu_grid(np.array([[2 ** 30 + 5, 0, 0]], np.int32), [0, 1])
    with pytest.raises(fvx.FvxError):
        g.refine(2)
    fvx.device_status()  # the status word was cleared by the failing call


# ---------------------------------------------------------------- transposed map

def _tmaps(grids, stride):
    """(gin, gout, map, oracle map) of the transposed conv for stride 1 (fine
    to fine) and stride 2 (coarse to refined and coarse to the original fine)."""
    import sparse_convolution_gb300 as fvx

    if stride == 1:
        gi, go, ogi, ogo = grids["g"], grids["g"], grids["og"], grids["og"]
    elif stride == 2:
        gi, go, ogi, ogo = grids["gc"], grids["gr"], grids["ogc"], grids["ogr"]
    else:  # stride 2 onto the original fine grid
        gi, go, ogi, ogo = grids["gc"], grids["g"], grids["ogc"], grids["og"]
        stride = 2
    return gi, go, fvx.KernelMap(gi, go, stride, transposed=True), oracle.KernelMap(ogi, ogo, stride,
                                                                                    transposed=True)


@pytest.mark.parametrize("case", [1, 2, "2fine"])
def test_transposed_kmap_matches_oracle(cuda_device, grids, case):
    _, _, km, okm = _tmaps(grids, case)
    G.assert_kmap_equal(km, okm)


def test_transposed_map_pairs_forward_pairs(cuda_device, grids):
    """The transposed map of (coarse, fine) holds exactly the pairs of the
    forward map of (fine, coarse), roles swapped, slot for slot."""
    import sparse_convolution_gb300 as fvx

    kt = fvx.KernelMap(grids["gc"], grids["g"], 2, transposed=True)
    kf = fvx.KernelMap(grids["g"], grids["gc"], 2)
    ti, to, _ = (G.np_(t) for t in kt.pairs())
    fi, fo, _ = (G.np_(t) for t in kf.pairs())
    assert np.array_equal(kt.offsets, kf.offsets)
    for s in range(27):
        a, b = kt.offsets[s], kt.offsets[s + 1]
        t = sorted(zip(ti[a:b].tolist(), to[a:b].tolist()))
        f = sorted(zip(fo[a:b].tolist(), fi[a:b].tolist()))
        assert t == f, s


def test_transposed_map_empty(cuda_device, grids):
    import sparse_convolution_gb300 as fvx

    e = G.gpu_grid(np.zeros((0, 3), np.int32), [0, 0, 0])
    km = fvx.KernelMap(e, grids["g"], 2, transposed=True)
    assert km.n_pairs == 0 and km.n_out == grids["g"].n_active
    km2 = fvx.KernelMap(grids["gc"], e, 2, transposed=True)
    assert km2.n_pairs == 0 and km2.n_out == 0


# ---------------------------------------------------------------- transposed conv

@pytest.mark.parametrize("cin,cout", [(16, 16), (32, 64), (8, 32), (64, 16)])
@pytest.mark.parametrize("case", [1, 2, "2fine"])
def test_transposed_conv_bf16(cuda_device, grids, case, cin, cout):
    """Runs the pair-list kernels; the leaf-densified kernels never take a
    transposed map."""
    import sparse_convolution_gb300 as fvx

    gi, go, km, okm = _tmaps(grids, case)
    x, W = G.bf16_inputs(13, gi.n_active, cin, cout)
    y = fvx.sparse_conv(gi, go, km, x, W)
    fvx.device_status()
    assert fvx.last_conv_algo() == fvx.FVX_CONV_GATHER
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL)


@pytest.mark.parametrize("cin,cout", [(5, 7), (16, 16)])
@pytest.mark.parametrize("case", [1, 2])
def test_transposed_conv_f32(cuda_device, grids, case, cin, cout):
    import torch

    import sparse_convolution_gb300 as fvx
    from sparse_convolution_gb300 import synth

    gi, go, km, okm = _tmaps(grids, case)
    x = torch.from_numpy(synth.features(17, gi.n_active, cin, "uniform")).cuda()
    W = torch.from_numpy(synth.weights(18, cin, cout)).cuda()
    y = fvx.sparse_conv(gi, go, km, x, W)
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y), yo, ao, G.F32_TOL)


def test_leaf_conv_refuses_transposed_map(cuda_device, grids):
    import sparse_convolution_gb300 as fvx

    gi, go, km, _ = _tmaps(grids, 1)
    x, W = G.bf16_inputs(3, gi.n_active, 16, 16)
    fvx.set_conv_algo(fvx.FVX_CONV_LEAF)
    try:
        with pytest.raises(fvx.FvxError):
            fvx.sparse_conv(gi, go, km, x, W)
    finally:
        fvx.set_conv_algo(fvx.FVX_CONV_AUTO)


# ---------------------------------------------------------------- input gradient

def _fwd(grids, stride):
    """(gin, gout, oracle gin, oracle gout) of a forward conv."""
    if stride == 1:
        return grids["g"], grids["g"], grids["og"], grids["og"]
    return grids["g"], grids["gc"], grids["og"], grids["ogc"]


@pytest.mark.parametrize("cin,cout", [(16, 16), (32, 64), (64, 32), (16, 8), (128, 128), (8, 16), (24, 8), (40, 64)])
@pytest.mark.parametrize("stride", [1, 2])
def test_dgrad_bf16(cuda_device, grids, stride, cin, cout):
    """dx = conv of dy over the transposed map with per-offset W^T."""
    import sparse_convolution_gb300 as fvx

    gi, go, ogi, ogo = _fwd(grids, stride)
    kt = fvx.KernelMap(go, gi, stride, transposed=True)
    okt = oracle.KernelMap(ogo, ogi, stride, transposed=True)
    import torch

    from sparse_convolution_gb300 import synth

    dy = torch.from_numpy(synth.features(29, go.n_active, cout)).cuda().bfloat16()
    W = torch.from_numpy(synth.weights(30, cin, cout)).cuda().bfloat16()
    dx = fvx.sparse_conv_dgrad(gi, go, kt, dy, W)
    fvx.device_status()
    assert tuple(dx.shape) == (gi.n_active, cin)
    ref, a = oracle.conv(okt, G.as_f64(dy), np.ascontiguousarray(G.as_f64(W).transpose(0, 2, 1)))
    G.assert_conv_close(G.np_(dx.float()), ref, a, G.BF16_TOL)


@pytest.mark.parametrize("cin,cout", [(3, 5), (16, 16), (33, 8)])
@pytest.mark.parametrize("stride", [1, 2])
def test_dgrad_f32(cuda_device, grids, stride, cin, cout):
    import torch

    import sparse_convolution_gb300 as fvx
    from sparse_convolution_gb300 import synth

    gi, go, ogi, ogo = _fwd(grids, stride)
    kt = fvx.KernelMap(go, gi, stride, transposed=True)
    okt = oracle.KernelMap(ogo, ogi, stride, transposed=True)
    dy = torch.from_numpy(synth.features(31, go.n_active, cout, "uniform")).cuda()
    W = torch.from_numpy(synth.weights(32, cin, cout)).cuda()
    dx = fvx.sparse_conv_dgrad(gi, go, kt, dy, W)
    ref, a = oracle.conv(okt, G.as_f64(dy), np.ascontiguousarray(G.as_f64(W).transpose(0, 2, 1)))
    G.assert_conv_close(G.np_(dx), ref, a, G.F32_TOL)


def test_dgrad_adjoint_identity(cuda_device, grids):
    """<conv(x, W), dy> == <x, dgrad(dy, W)> (fp32 path, stride 2)."""
    import torch

    import sparse_convolution_gb300 as fvx
    from sparse_convolution_gb300 import synth

    gi, go = grids["g"], grids["gc"]
    km = fvx.KernelMap(gi, go, 2)
    kt = fvx.KernelMap(go, gi, 2, transposed=True)
    x = torch.from_numpy(synth.features(41, gi.n_active, 8)).cuda()
    dy = torch.from_numpy(synth.features(42, go.n_active, 12)).cuda()
    W = torch.from_numpy(synth.weights(43, 8, 12)).cuda()
    lhs = float((fvx.sparse_conv(gi, go, km, x, W).double() * dy.double()).sum())
    rhs = float((x.double() * fvx.sparse_conv_dgrad(gi, go, kt, dy, W).double()).sum())
    assert abs(lhs - rhs) <= 1e-4 * max(1.0, abs(lhs))


def test_dgrad_rejects_forward_map(cuda_device, grids):
    import sparse_convolution_gb300 as fvx

    gi, go = grids["g"], grids["gc"]
    km = fvx.KernelMap(gi, go, 2)
    dy, W = G.bf16_inputs(3, go.n_active, 16, 16)
    with pytest.raises(fvx.FvxError):
        fvx.sparse_conv_dgrad(gi, go, km, dy, W)


# ---------------------------------------------------------------- weight gradient

@pytest.mark.parametrize("cin,cout", [(16, 16), (8, 64), (64, 32), (3, 5), (40, 72), (64, 64), (128, 64), (64, 256),
                                      (192, 128), (128, 320)])
@pytest.mark.parametrize("stride", [1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_wgrad_matches_oracle(cuda_device, grids, stride, cin, cout, dtype):
    import torch

    import sparse_convolution_gb300 as fvx
    from sparse_convolution_gb300 import synth

    gi, go, ogi, ogo = _fwd(grids, stride)
    km = fvx.KernelMap(gi, go, stride)
    okm = oracle.KernelMap(ogi, ogo, stride)
    x = torch.from_numpy(synth.features(51, gi.n_active, cin)).cuda()
    dy = torch.from_numpy(synth.features(52, go.n_active, cout)).cuda()
    if dtype == "bf16":
        x, dy = x.bfloat16(), dy.bfloat16()
    dW = fvx.sparse_conv_wgrad(gi, go, km, x, dy)
    assert dW.dtype == torch.float32 and tuple(dW.shape) == (27, cin, cout)
    x64, dy64 = G.as_f64(x), G.as_f64(dy)
    ref = oracle.conv_wgrad(okm, x64, dy64)
    a = oracle.conv_wgrad(okm, np.abs(x64), np.abs(dy64))
    G.assert_conv_close(G.np_(dW), ref, a, G.BF16_TOL if dtype == "bf16" else G.F32_TOL)


def test_wgrad_many_pairs(cuda_device):
    """Tens of thousands of pairs per list: several 32768-pair chunks, so
    each list's sums cross block boundaries."""
    import torch

    import sparse_convolution_gb300 as fvx
    from sparse_convolution_gb300 import synth

    c, offs = _random(61, 60000, -25, 50, 1, dup=0.0)
    g = G.gpu_grid(c, offs)
    og = oracle.Grid.build(c, offs)
    km = fvx.KernelMap(g, g, 1)
    okm = oracle.KernelMap(og, og, 1)
    assert km.offsets[14] - km.offsets[13] > 32768 and km.n_pairs > 8 * 32768  # the centre list spans 2 chunks
    for cin, cout in ((16, 32), (64, 64)):  # fp32 FFMA; tensor cores
        x = torch.from_numpy(synth.features(62, g.n_active, cin)).cuda().bfloat16()
        dy = torch.from_numpy(synth.features(63, g.n_active, cout)).cuda().bfloat16()
        dW = fvx.sparse_conv_wgrad(g, g, km, x, dy)
        fvx.device_status()
        x64, dy64 = G.as_f64(x), G.as_f64(dy)
        ref = oracle.conv_wgrad(okm, x64, dy64)
        a = oracle.conv_wgrad(okm, np.abs(x64), np.abs(dy64))
        G.assert_conv_close(G.np_(dW), ref, a, G.BF16_TOL)


def test_wgrad_empty_input(cuda_device, grids):
    """No input voxels: no pairs, dW all zero (overwritten, not left as is)."""
    import torch

    import sparse_convolution_gb300 as fvx

    e = G.gpu_grid(np.zeros((0, 3), np.int32), [0, 0, 0])
    km = fvx.KernelMap(e, grids["gc"], 2)
    x = torch.zeros((0, 16), device="cuda", dtype=torch.bfloat16)
    dy = torch.ones((grids["gc"].n_active, 16), device="cuda", dtype=torch.bfloat16)
    out = torch.full((27, 16, 16), 7.0, device="cuda")
    fvx.sparse_conv_wgrad(e, grids["gc"], km, x, dy, out=out)
    assert int((out != 0).sum()) == 0


@pytest.fixture(scope="module")
def dense_grid():
    """A solid ball (radius 13, two batches, one shifted to negative
    coordinates): leaves well above 20% occupied."""
    r = np.arange(-14, 15)
    c = np.stack(np.meshgrid(r, r, r, indexing="ij"), -1).reshape(-1, 3)
    ball = c[(c ** 2).sum(1) <= 13 ** 2].astype(np.int32)
    coords = np.concatenate([ball + 40, ball - 21])
    offs = np.array([0, len(ball), 2 * len(ball)], np.int64)
    rng = np.random.default_rng(3)
    perm = np.concatenate([rng.permutation(len(ball)), len(ball) + rng.permutation(len(ball))])
    coords = coords[perm]
    g = G.gpu_grid(coords, offs)
    og = oracle.Grid.build(coords, offs)
    assert g.n_active >= 0.2 * 512 * g.n_leaf
    return g, og


@pytest.mark.parametrize("cin,cout", [(8, 16), (16, 16), (32, 8), (64, 16), (24, 8)])
@pytest.mark.parametrize("algo", ["auto", "leaf", "gather"])
def test_dgrad_leaf_densified(cuda_device, dense_grid, cin, cout, algo):
    """Stride-1 input gradient on dense leaves: the leaf-densified kernel with
    slot-mirrored weights (automatic choice or forced) and the pair-list
    kernels give the oracle's result within the bf16 bound."""
    import torch

    import sparse_convolution_gb300 as fvx
    from sparse_convolution_gb300 import synth

    g, og = dense_grid
    kt = fvx.KernelMap(g, g, 1, transposed=True)
    okt = oracle.KernelMap(og, og, 1, transposed=True)
    dy = torch.from_numpy(synth.features(71, g.n_active, cout)).cuda().bfloat16()
    W = torch.from_numpy(synth.weights(72, cin, cout)).cuda().bfloat16()
    fvx.set_conv_algo({"auto": fvx.FVX_CONV_AUTO, "leaf": fvx.FVX_CONV_LEAF, "gather": fvx.FVX_CONV_GATHER}[algo])
    try:
        dx = fvx.sparse_conv_dgrad(g, g, kt, dy, W)
        fvx.device_status()
        ran = fvx.last_conv_algo()
    finally:
        fvx.set_conv_algo(fvx.FVX_CONV_AUTO)
    assert ran == (fvx.FVX_CONV_GATHER if algo == "gather" else fvx.FVX_CONV_LEAF)
    ref, a = oracle.conv(okt, G.as_f64(dy), np.ascontiguousarray(G.as_f64(W).transpose(0, 2, 1)))
    G.assert_conv_close(G.np_(dx.float()), ref, a, G.BF16_TOL)


def test_forward_conv_refuses_leaf_on_transposed_map(cuda_device, dense_grid):
    """A transposed map's leaf table serves the input gradient only: the
    forward conv over a transposed map takes the pair-list kernels."""
    import sparse_convolution_gb300 as fvx

    g, og = dense_grid
    kt = fvx.KernelMap(g, g, 1, transposed=True)
    x, W = G.bf16_inputs(5, g.n_active, 16, 16)
    y = fvx.sparse_conv(g, g, kt, x, W)
    assert fvx.last_conv_algo() == fvx.FVX_CONV_GATHER
    yo, ao = oracle.conv(oracle.KernelMap(og, og, 1, transposed=True), G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL)

"""Voxels along rays on the GPU (hierarchical DDA, "fVDB" reading notes,
HDDA) against the CPU oracle's per-voxel DDA: offsets, voxel indices and the
entry/exit times bit-exact (both follow one fp32 definition, so floating
point decides the same cells on both sides).

Small random grids with rays of every kind (outside and inside, zero
direction components, batches, negative coordinates across root tiles),
exact-tie rays, segment clips, empty inputs, errors; the narrow-band scene at
full size with camera rays, compared on every ray of a 4096-ray subset.
"""
import numpy as np
import pytest

import oracle
from sparse_convolution_gb300 import synth
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


def _gpu_hits(g, o, d, batch=None, tmin=0.0, tmax=float("inf")):
    import torch

    import sparse_convolution_gb300 as fvx

    ot = torch.from_numpy(np.ascontiguousarray(o, np.float32)).cuda()
    dt = torch.from_numpy(np.ascontiguousarray(d, np.float32)).cuda()
    bt = None if batch is None else torch.from_numpy(np.ascontiguousarray(batch, np.int32)).cuda()
    h = fvx.Hits(g, ot, dt, bt, tmin, tmax)
    offs, vox, t = (G.np_(x) for x in h.arrays())
    h.destroy()
    return offs, vox, t


def _assert_same(got, exp):
    go, gv, gt = got
    eo, ev, et = exp
    assert np.array_equal(go, eo), f"offsets differ at ray {np.flatnonzero(go != eo)[:5]}"
    assert np.array_equal(gv, ev)
    assert np.array_equal(gt.view(np.uint32), et.view(np.uint32)), "times differ (bitwise)"


def _both(coords, offs, o, d, batch=None, tmin=0.0, tmax=float("inf")):
    g = G.gpu_grid(coords, offs)
    og = oracle.Grid.build(np.ascontiguousarray(coords, np.int32), np.asarray(offs, np.int64))
    got = _gpu_hits(g, o, d, batch, tmin, tmax)
    exp = oracle.voxels_along_rays(og, o, d, batch, tmin, tmax)
    return got, exp


@pytest.mark.parametrize("seed", [0, 1])
def test_random_grids_and_rays(cuda_device, seed):
    rng = np.random.default_rng(seed)
    # two batch elements, negative coordinates, a gap of empty leaves and nodes
    a = rng.integers(-14, 14, size=(12000, 3))
    b = np.concatenate([rng.integers(-4110, -4085, size=(8000, 3)), rng.integers(120, 140, size=(5000, 3))])
    coords = np.concatenate([a, b]).astype(np.int32)
    offs = np.array([0, len(a), len(coords)], np.int64)
    n = 3000
    o = rng.uniform(-4200, 300, size=(n, 3)).astype(np.float32)
    o[: n // 4] = rng.uniform(-10, 10, size=(n // 4, 3))  # starting inside
    batch = rng.integers(0, 2, size=n).astype(np.int32)
    # aim at the batch element's clusters (element 1 straddles a root tile boundary at -4096)
    tgt = np.where(batch[:, None] == 0, rng.uniform(-14, 14, size=(n, 3)),
                   np.where(rng.random((n, 1)) < 0.5, rng.uniform(-4110, -4085, size=(n, 3)),
                            rng.uniform(120, 140, size=(n, 3))))
    d = (tgt - o).astype(np.float32)
    d[::5, 1] = 0.0
    d[::7, 2] = 0.0
    d[::13] = 0.0  # no direction: no hits
    got, exp = _both(coords, offs, o, d, batch, 0.0, 1e6)
    _assert_same(got, exp)
    assert exp[1].shape[0] > 15000


def test_ties_axis_rays_and_segments(cuda_device):
    coords = []
    for k in range(12):
        coords += [(k, k, k), (k + 1, k, k), (k, k + 1, k), (k, k, k + 1), (k, 5, 3)]
    coords = np.array(coords, np.int32)
    offs = [0, len(coords)]
    o = np.array([[0, 0, 0], [-3.5, 5.5, 3.5], [20.5, 5.5, 3.5], [0.5, 0.5, 0.5], [2.25, 2.75, 2.5],
                  [11.9999, 0.0001, 5.5]], np.float32)
    d = np.array([[1, 1, 1], [1, 0, 0], [-1, 0, 0], [0, 0, 0], [1, 1, 0], [-1, 1, 0]], np.float32)
    for tmin, tmax in [(0.0, float("inf")), (2.0, 7.25), (5.0, 5.0), (6.0, 1.0), (-100.0, 3.0)]:
        got, exp = _both(coords, offs, o, d, None, tmin, tmax)
        _assert_same(got, exp)
    got, exp = _both(coords, offs, o, d)
    assert list(exp[1][exp[0][0]:exp[0][1]].shape) == [12]  # the diagonal: 12 cells (k,k,k)


def test_empty_inputs(cuda_device):
    import torch

    import sparse_convolution_gb300 as fvx

    g = G.gpu_grid(np.zeros((0, 3), np.int32), [0, 0])
    offs, vox, t = _gpu_hits(g, np.zeros((5, 3), np.float32), np.ones((5, 3), np.float32))
    assert list(offs) == [0] * 6 and vox.shape == (0,) and t.shape == (0, 2)
    g2 = G.gpu_grid(np.array([[1, 2, 3]], np.int32), [0, 1])
    h = fvx.Hits(g2, torch.zeros((0, 3), device="cuda"), torch.zeros((0, 3), device="cuda"))
    assert h.n_rays == 0 and h.n_hits == 0 and list(G.np_(h.arrays()[0])) == [0]


def test_errors_and_recovery(cuda_device):
    import torch

    import sparse_convolution_gb300 as fvx

    coords = np.array([[i, 0, 0] for i in range(20)], np.int32)
    g = G.gpu_grid(coords, [0, len(coords)])
    o = torch.tensor([[-1.0, 0.5, 0.5]] * 3, device="cuda")
    d = torch.tensor([[1.0, 0.0, 0.0]] * 3, device="cuda")
    with pytest.raises(fvx.FvxError) as e:
        fvx.Hits(g, o, d, torch.tensor([0, 1, 0], device="cuda"))
    assert e.value.status == "FVX_ERR_CHECK" and "batch index" in str(e.value)
    with pytest.raises(fvx.FvxError) as e:
        fvx.Hits(g, o, d, tmin=float("nan"))
    assert e.value.status == "FVX_ERR_INVALID_ARG"
    far = G.gpu_grid(np.array([[1 << 24, 0, 0], [0, 0, 0]], np.int32), [0, 2])
    with pytest.raises(fvx.FvxError) as e:
        fvx.Hits(far, o, d)
    assert e.value.status == "FVX_ERR_CHECK"
    fvx.device_status()
    h = fvx.Hits(g, o, d)  # the library keeps working
    assert h.n_hits == 60


def test_narrow_band_scene_camera_rays(cuda_device):
    """The ray benchmark's input: the 1024^3 narrow-band scene and a
    1024 x 1024 camera.  Every ray: offsets consistent, times ordered, each
    hit's cell holds the midpoint of its interval.  A 2048-ray sample: equal
    to the oracle, bit for bit."""
    w = synth.ray_scene(1024)
    o, d = synth.camera_rays(1024, 1024)
    g = G.gpu_grid(w["coords"], w["batch_offsets"])
    offs, vox, t = _gpu_hits(g, o, d)
    n = np.diff(offs)
    assert offs[0] == 0 and offs[-1] == vox.shape[0] and np.all(n >= 0)
    assert (n > 0).mean() > 0.3
    assert np.all(t[:, 0] < t[:, 1])
    ray = np.repeat(np.arange(o.shape[0]), n)
    same = ray[1:] == ray[:-1]
    assert np.all(t[1:, 0][same] >= t[:-1, 1][same])  # in order, no overlap
    ijk = G.np_(g.ijk()).astype(np.float64)[vox]
    mid = o[ray].astype(np.float64) + d[ray].astype(np.float64) * t.astype(np.float64).mean(axis=1, keepdims=True)
    assert np.all((mid >= ijk - 1e-3) & (mid <= ijk + 1 + 1e-3))
    og = oracle.Grid.build(w["coords"], w["batch_offsets"])
    rows = np.sort(np.random.default_rng(5).choice(o.shape[0], size=2048, replace=False))
    eo, ev, et = oracle.voxels_along_rays(og, o[rows], d[rows])
    sel = np.concatenate([np.arange(offs[r], offs[r + 1]) for r in rows])
    assert np.array_equal(n[rows], np.diff(eo))
    assert np.array_equal(vox[sel], ev)
    assert np.array_equal(t[sel].view(np.uint32), et.view(np.uint32))

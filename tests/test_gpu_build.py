"""GPU IndexGrid build, lookup and coarsen vs the CPU oracle (bit-exact).

Build: "fVDB: A Deep-Learning Framework for Sparse, Large Scale, and High
Performance Spatial Intelligence" notes, "GPU-accelerated IndexGrid build" and
"IndexGrid"."""
import numpy as np
import pytest

import oracle
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


def _random(seed, n, lo, span, B, dup=0.2):
    rng = np.random.default_rng(seed)
    rows, offs = [], [0]
    for _ in range(B):
        c = rng.integers(lo, lo + span, size=(n, 3)).astype(np.int32)
        c = np.concatenate([c, c[rng.integers(0, n, size=int(dup * n))]])
        rows.append(c[rng.permutation(len(c))])
        offs.append(offs[-1] + len(c))
    return np.concatenate(rows), np.array(offs, np.int64)


CASES = {
    "small_one_tile": (0, 5000, 0, 64, 1),
    "negative": (1, 4097, -70, 100, 1),
    "three_batches": (2, 3001, -30, 60, 3),
    "tile_straddle": (3, 20000, -5000, 10000, 2),
    "ragged_2049": (4, 2049, 100, 40, 1),
    "dense_block": (5, 40000, 0, 32, 1),
    "many_batches": (6, 300, -10, 25, 40),
    # one batch in one root tile: a key space of <= 2^28 takes the presence
    # bitmap instead of the sort; the full 4096^3 tile (36 varying bits) sorts
    "one_tile_bitmap": (7, 30000, 1024, 512, 1),
    "one_tile_full_width": (8, 30000, 0, 4096, 1),
    "one_tile_bitmap_27_bits": (9, 20000, 0, 512, 1),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_build_matches_oracle(cuda_device, name):
    seed, n, lo, span, B = CASES[name]
    c, offs = _random(seed, n, lo, span, B)
    g = G.gpu_grid(c, offs)
    og = oracle.Grid.build(c, offs)
    G.assert_topology_equal(g, og)
    assert np.array_equal(g.batch_offsets(), og.voxels()["voxel_batch_offsets"])


@pytest.mark.parametrize("coords,offs", [
    (np.array([[5, -3, 7]], np.int32), [0, 1]),
    (np.array([[-1, -1, -1], [0, 0, 0], [-4096, 0, 0], [4095, 0, 0], [-1, 0, 0]], np.int32), [0, 5]),
    (np.array([[1, 2, 3], [1, 2, 3], [9, 9, 9]], np.int32), [0, 2, 2, 3]),
    (np.repeat(np.array([[7, 7, 7]], np.int32), 5000, axis=0), [0, 5000]),
    ((np.stack(np.meshgrid(*[np.arange(8)] * 3, indexing="ij"), -1).reshape(-1, 3) + 16)[::-1].astype(np.int32),
     [0, 512]),
    (np.array([[2 ** 31 - 1, -2 ** 31, 0], [-2 ** 31, 2 ** 31 - 1, 5], [0, 0, 0]], np.int32), [0, 3]),
])
def test_build_special_cases(cuda_device, coords, offs):
    g = G.gpu_grid(coords, offs)
    og = oracle.Grid.build(coords, offs)
    G.assert_topology_equal(g, og)


def test_build_empty(cuda_device):
    g = G.gpu_grid(np.zeros((0, 3), np.int32), [0, 0, 0])
    assert g.counts() == dict(n_upper=0, n_lower=0, n_leaf=0, n_active=0)
    assert g.batch_offsets().tolist() == [0, 0, 0]


def test_build_range_error(cuda_device):
    """17 batches over the full int32 tile range need a 65-bit first key."""
    import sparse_convolution_gb300 as fvx

    c = np.array([[2 ** 31 - 1, 2 ** 31 - 1, 2 ** 31 - 1], [-2 ** 31, -2 ** 31, -2 ** 31]] * 17, np.int32)
    offs = np.arange(0, 35, 2)
    with pytest.raises(fvx.FvxError, match="FVX_ERR_RANGE"):
        G.gpu_grid(c, offs)
    g = G.gpu_grid(c[:32], offs[:17])  # 16 batches fit exactly
    G.assert_topology_equal(g, oracle.Grid.build(c[:32], offs[:17]))


def test_lookup_matches_oracle(cuda_device):
    import torch

    c, offs = _random(11, 6000, -40, 80, 2)
    g = G.gpu_grid(c, offs)
    og = oracle.Grid.build(c, offs)
    rng = np.random.default_rng(12)
    q = rng.integers(-50, 50, size=(50000, 3)).astype(np.int32)
    qb = rng.integers(0, 3, size=50000).astype(np.int32)  # batch 2 does not exist -> -1
    got = G.np_(g.lookup(torch.from_numpy(q).cuda(), torch.from_numpy(qb).cuda()))
    assert np.array_equal(got, og.lookup(q, qb))
    v = og.voxels()
    got = G.np_(g.lookup(torch.from_numpy(v["ijk"]).cuda(), torch.from_numpy(v["batch"]).cuda()))
    assert np.array_equal(got, np.arange(og.n_active))


@pytest.mark.parametrize("stride", [2, 3, 4])
def test_coarsen_matches_oracle(cuda_device, stride):
    c, offs = _random(21 + stride, 8000, -60, 120, 2)
    g = G.gpu_grid(c, offs)
    gc = g.coarsen(stride)
    og = oracle.Grid.build(c, offs)
    G.assert_topology_equal(gc, og.coarsen(stride))


def test_build_is_deterministic(cuda_device):
    c, offs = _random(31, 30000, -100, 200, 2)
    t1 = {k: G.np_(v) for k, v in G.gpu_grid(c, offs).topology().items()}
    t2 = {k: G.np_(v) for k, v in G.gpu_grid(c, offs).topology().items()}
    assert all(np.array_equal(t1[k], t2[k]) for k in t1)

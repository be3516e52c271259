"""Pins of the oracle's voxels-along-rays ("fVDB" reading notes, HDDA: the
voxels each ray passes through, found level by level).

The oracle walks every cell with a per-voxel DDA in fp32 plane-crossing times.
It is checked here against things that do not share that walk:
* closed forms: rays along a grid axis through a row of voxels (hits are the
  active voxels of the row, entry and exit at the cell faces), and the main
  diagonal through a corner (crossings tie on all three axes: only the
  diagonal cells are occupied for a positive time);
* a brute force in exact rational arithmetic on small random grids: every
  active voxel's cell is intersected with the ray (slab method with
  fractions.Fraction on the exact values of the fp32 inputs); the cells with
  an intersection of positive length, in order of entry, are the hits.  Cells
  within 1e-4 of a grazing or tied decision, where fp32 rounding may decide
  either way, are left out of the comparison;
* batches: a ray of batch element b sees only that element's voxels.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _grid(coords, B=1, offs=None):
    coords = np.ascontiguousarray(coords, np.int32).reshape(-1, 3)
    if offs is None:
        offs = [0, len(coords)]
    return oracle.Grid.build(coords, np.asarray(offs, np.int64))


def _index_of(g):
    v = g.voxels()
    return {(int(b), *map(int, c)): n for n, (b, c) in enumerate(zip(v["batch"], v["ijk"]))}


@pytest.mark.parametrize("sign", [1, -1])
def test_axis_aligned_ray_through_a_row(sign):
    row = [0, 1, 2, 5, 6, 9, 13]
    coords = [(i, 3, 5) for i in row] + [(4, 4, 5), (7, 3, 6)]  # off-row voxels are not hit
    g = _grid(coords)
    idx = _index_of(g)
    o = np.array([[-2.5 if sign > 0 else 20.5, 3.5, 5.25]], np.float32)
    d = np.array([[float(sign), 0.0, 0.0]], np.float32)
    offs, vox, t = oracle.voxels_along_rays(g, o, d)
    order = row if sign > 0 else row[::-1]
    assert list(vox) == [idx[(0, i, 3, 5)] for i in order]
    ox = float(o[0, 0])
    exp = [((i - ox), (i + 1 - ox)) if sign > 0 else ((ox - (i + 1)), (ox - i)) for i in order]
    assert np.array_equal(t, np.array(exp, np.float32))
    assert list(offs) == [0, len(row)]


def test_diagonal_through_corners_ties():
    """o = (0,0,0), d = (1,1,1): every crossing happens on all three axes at
    once (t = 1, 2, ...), so only cells (k,k,k) are occupied for a positive
    time; their face neighbours are touched at single points only."""
    coords = []
    for k in range(6):
        coords += [(k, k, k), (k + 1, k, k), (k, k + 1, k), (k, k, k + 1)]
    g = _grid(coords)
    idx = _index_of(g)
    offs, vox, t = oracle.voxels_along_rays(g, np.zeros((1, 3), np.float32), np.ones((1, 3), np.float32))
    assert list(vox) == [idx[(0, k, k, k)] for k in range(6)]
    assert np.array_equal(t, np.array([(k, k + 1) for k in range(6)], np.float32))


def test_segment_clip_and_degenerate_rays():
    g = _grid([(i, 0, 0) for i in range(10)])
    o = np.array([[0.5, 0.5, 0.5]] * 4, np.float32)
    d = np.array([[1, 0, 0], [0, 0, 0], [0, 1, 0], [1, 0, 0]], np.float32)
    offs, vox, t = oracle.voxels_along_rays(g, o, d, tmin=2.0, tmax=4.25)
    # ray 0: cells 2 (from t = 2.0, mid-cell), 3, 4 (until 4.25); ray 1: d = 0; ray 2: leaves the
    # row's box at y = 1 (cell 0 only, from the clipped start); ray 3 as ray 0
    assert list(np.diff(offs)) == [3, 0, 0, 3]
    assert np.array_equal(t[:3], np.array([(2.0, 2.5), (2.5, 3.5), (3.5, 4.25)], np.float32))
    offs2, vox2, _ = oracle.voxels_along_rays(g, o[2:3], d[2:3], tmin=0.0, tmax=10.0)
    assert list(vox2) == [0]


def test_batches_are_separate():
    c = np.array([(i, 2, 2) for i in range(8)], np.int32)
    g = _grid(np.concatenate([c, c[::2]]), offs=[0, 8, 12])
    o = np.array([[-1.5, 2.5, 2.5]] * 2, np.float32)
    d = np.array([[1, 0, 0]] * 2, np.float32)
    offs, vox, _ = oracle.voxels_along_rays(g, o, d, batch=np.array([0, 1], np.int32))
    assert list(vox[:8]) == list(range(8))
    assert list(vox[8:]) == [8, 9, 10, 11]


def _exact_hits(ijk, o32, d32, tmin, tmax):
    """Exact (Fraction) positive-length intersections of the ray with every
    active cell, clipped to [tmin, tmax] and to the box of the voxels.
    Returns [(enter, exit, voxel index)] sorted by enter."""
    o = [Fraction(float(v)) for v in o32]
    d = [Fraction(float(v)) for v in d32]
    lo, hi = ijk.min(0), ijk.max(0) + 1

    def slab(a, b):  # the ray's t interval inside [a, b) per axis, intersected
        t0, t1 = Fraction(tmin), Fraction(tmax) if np.isfinite(tmax) else None
        for ax in range(3):
            if d[ax] == 0:
                if not (a[ax] <= o[ax] < b[ax]):
                    return None
                continue
            ta, tb = (a[ax] - o[ax]) / d[ax], (b[ax] - o[ax]) / d[ax]
            if ta > tb:
                ta, tb = tb, ta
            t0 = max(t0, ta)
            t1 = tb if t1 is None else min(t1, tb)
        return (t0, t1) if t1 is not None and t0 < t1 else None

    box = slab([int(v) for v in lo], [int(v) for v in hi])
    if box is None:
        return []
    out = []
    for n, c in enumerate(ijk):
        iv = slab([int(v) for v in c], [int(v) + 1 for v in c])
        if iv is None:
            continue
        e, x = max(iv[0], box[0]), min(iv[1], box[1])
        if e < x:
            out.append((e, x, n))
    return sorted(out)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_exact_brute_force(seed):
    rng = np.random.default_rng(seed)
    ijk = np.unique(rng.integers(-6, 7, size=(1500, 3)), axis=0).astype(np.int32)
    g = _grid(ijk)
    ijk = g.voxels()["ijk"]  # index order
    n = 200
    # origins inside and outside the box, directions of all signs and some zero components
    o = rng.uniform(-12, 12, size=(n, 3)).astype(np.float32)
    d = (rng.uniform(-6, 7, size=(n, 3)) - o).astype(np.float32)  # towards a point of the box
    d[::7, 0] = 0.0
    d[::11, 2] = 0.0
    tmin, tmax = 0.0, 60.0
    offs, vox, t = oracle.voxels_along_rays(g, o, d, tmin=tmin, tmax=tmax)
    eps = Fraction(1, 10000)
    compared = 0
    for r in range(n):
        got = list(zip(t[offs[r]:offs[r + 1], 0], t[offs[r]:offs[r + 1], 1], vox[offs[r]:offs[r + 1]]))
        exact = _exact_hits(ijk, o[r], d[r], tmin, tmax)
        sure = {v for e, x, v in exact if x - e > eps}
        maybe = {v for e, x, v in exact if x - e <= eps}
        got_set = [v for _, _, v in got]
        assert len(set(got_set)) == len(got_set), "a cell visited twice"
        assert sure <= set(got_set), (r, sorted(sure - set(got_set)))
        assert set(got_set) <= sure | maybe, (r, sorted(set(got_set) - sure - maybe))
        # order and times of the sure hits
        ex = {v: (e, x) for e, x, v in exact}
        seq = [v for v in got_set if v in sure]
        assert seq == [v for e, x, v in exact if v in sure]
        for te, tx, v in got:
            if v in sure:
                assert abs(float(ex[v][0]) - float(te)) < 1e-4 and abs(float(ex[v][1]) - float(tx)) < 1e-4
            assert te < tx
        assert all(got[i][0] <= got[i + 1][0] for i in range(len(got) - 1))
        compared += len(sure)
    assert compared > 1000  # the rays do cross the grid

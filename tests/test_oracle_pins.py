"""Pins for the CPU oracle, checked against things other than the oracle:
numbers the pages print, library routines (torch conv3d, numpy unique),
brute force on tiny inputs, invariants and special cases.

Pages: "fVDB: A Deep-Learning Framework for Sparse, Large Scale, and High
Performance Spatial Intelligence" (reading notes: Core method; IndexGrid;
GPU-accelerated IndexGrid build) and "DriveRT" (Shared neighbour maps).
"""
import os

import numpy as np
import pytest

import oracle
from tests import helpers as H

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "vdb_tree_config.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = int(v)
    return out


def _random_grid(seed, n=3000, span=40, lo=-20, B=1, dup=0.2):
    rng = np.random.default_rng(seed)
    rows, offs = [], [0]
    for b in range(B):
        c = rng.integers(lo, lo + span, size=(n, 3)).astype(np.int32)
        c = np.concatenate([c, c[rng.integers(0, n, size=int(dup * n))]])
        c = c[rng.permutation(len(c))]
        rows.append(c)
        offs.append(offs[-1] + len(c))
    return np.concatenate(rows), np.array(offs, np.int64)


def _check_topology(g, coords, offs):
    v = g.voxels()
    uniq = H.unique_voxels(coords, offs)
    # |unique coords| == number of active voxels (numpy unique vs std::map)
    assert g.n_active == uniq.shape[0]
    # ijk_of_index is a permutation of the unique set
    got = np.unique(np.concatenate([v["batch"][:, None], v["ijk"]], axis=1).astype(np.int64), axis=0)
    assert np.array_equal(got, uniq)
    # indices follow the canonical order (strictly increasing)
    assert H.strictly_increasing_rows(H.canonical_tuples(v["batch"], v["ijk"]))
    # every input row maps to the index of its own coordinate
    b_rows = np.repeat(np.arange(len(offs) - 1), np.diff(offs))
    r2i = v["row_to_index"]
    assert np.array_equal(v["ijk"][r2i], coords)
    assert np.array_equal(v["batch"][r2i], b_rows)
    # lookup(ijk_of_index[t]) == t
    assert np.array_equal(g.lookup(v["ijk"], v["batch"]), np.arange(g.n_active))
    # batch CSR over voxels
    vbo = v["voxel_batch_offsets"]
    assert np.array_equal(np.diff(vbo), np.bincount(v["batch"], minlength=len(offs) - 1))
    # tree walk with the exported masks / prefix counts reproduces the map
    up, lo, lf = g.upper(), g.lower(), g.leaves()
    assert np.array_equal(H.tree_lookup(up, lo, lf, v["batch"], v["ijk"]), np.arange(g.n_active))
    # leaf popcounts sum to U; first index = exclusive prefix of popcounts
    pc = H.popcount64(lf["mask"]).sum(axis=1)
    assert pc.sum() == g.n_active
    assert np.array_equal(lf["first"].astype(np.int64), np.concatenate([[0], np.cumsum(pc)[:-1]]))
    # node origins are multiples of the node extents (fanouts 32/16/8)
    gold = _golden()
    assert np.all(np.mod(lf["origin"], gold["leaf_extent"]) == 0)
    assert np.all(np.mod(lo["origin"], gold["lower_extent"]) == 0)
    assert np.all(np.mod(up["origin"], gold["upper_extent"]) == 0)
    # each voxel's leaf/lower/upper origin is its coordinate rounded down
    leaf_of_vox = np.repeat(np.arange(g.n_leaf), pc)
    assert np.array_equal(lf["origin"][leaf_of_vox], v["ijk"] - np.mod(v["ijk"], 8))
    assert np.array_equal(lf["batch"][leaf_of_vox], v["batch"])
    lpc = H.popcount64(lo["mask"]).sum(axis=1)
    assert lpc.sum() == g.n_leaf
    lower_of_leaf = np.repeat(np.arange(g.n_lower), lpc)
    assert np.array_equal(lo["origin"][lower_of_leaf], lf["origin"] - np.mod(lf["origin"], 128))
    upc = H.popcount64(up["mask"]).sum(axis=1)
    assert upc.sum() == g.n_lower
    upper_of_lower = np.repeat(np.arange(g.n_upper), upc)
    assert np.array_equal(up["origin"][upper_of_lower], lo["origin"] - np.mod(lo["origin"], 4096))
    return v


def test_golden_tree_numbers():
    gold = _golden()
    # fanout^3 children; extents multiply down the tree
    assert gold["leaf_extent"] == gold["leaf_fanout"]
    assert gold["lower_extent"] == gold["lower_fanout"] * gold["leaf_extent"]
    assert gold["upper_extent"] == gold["upper_fanout"] * gold["lower_extent"]
    assert 2 ** gold["key1_shift"] == gold["upper_extent"]
    # the oracle's leaf record is the 80-byte record of the pages, > 50x
    # smaller than a 4 KB one-uint64-per-voxel leaf
    assert oracle.leaf_record_bytes() == gold["leaf_record_bytes"]
    assert gold["naive_leaf_bytes_min"] / gold["leaf_record_bytes"] > gold["compression_min"]
    assert 8 ** 3 * 8 == gold["naive_leaf_bytes_min"]


@pytest.mark.parametrize("seed,lo,B", [(0, -20, 1), (1, 4080, 1), (2, -5000, 2), (3, 0, 3)])
def test_build_invariants(seed, lo, B):
    coords, offs = _random_grid(seed, n=2500, span=48, lo=lo, B=B)
    g = oracle.Grid.build(coords, offs)
    _check_topology(g, coords, offs)
    # absent coordinates map to -1 (map and tree walk agree)
    rng = np.random.default_rng(seed + 100)
    q = rng.integers(lo - 10, lo + 60, size=(4000, 3)).astype(np.int32)
    qb = rng.integers(0, B, size=4000).astype(np.int32)
    m = g.lookup(q, qb)
    assert np.array_equal(m, H.tree_lookup(g.upper(), g.lower(), g.leaves(), qb, q))
    present = set(map(tuple, H.unique_voxels(coords, offs).tolist()))
    expect = np.array([(int(b), *map(int, c)) in present for b, c in zip(qb, q)])
    assert np.array_equal(m >= 0, expect)


def test_single_voxel():
    g = oracle.Grid.build(np.array([[5, -3, 7]], np.int32), [0, 1])
    assert g.counts() == dict(n_upper=1, n_lower=1, n_leaf=1, n_active=1)
    lf = g.leaves()
    n = (5 % 8 * 8 + (-3) % 8) * 8 + 7 % 8
    assert lf["mask"][0, n // 64] == np.uint64(1) << np.uint64(n % 64)
    assert lf["first"][0] == 0 and np.array_equal(lf["origin"][0], [0, -8, 0])


def test_full_leaf():
    ii = np.stack(np.meshgrid(np.arange(8), np.arange(8), np.arange(8), indexing="ij"), -1).reshape(-1, 3) + 16
    g = oracle.Grid.build(ii[::-1].astype(np.int32), [0, 512])
    lf = g.leaves()
    assert g.n_leaf == 1 and g.n_active == 512
    assert np.all(lf["mask"] == np.uint64(0xFFFFFFFFFFFFFFFF))
    fields = [(int(lf["prefix9"][0]) >> (9 * (w - 1))) & 511 for w in range(1, 8)]
    assert fields == [64 * w for w in range(1, 8)]
    v = g.voxels()
    # in a full leaf the index is the x-major bit number
    n = ((v["ijk"][:, 0] - 16) * 8 + (v["ijk"][:, 1] - 16)) * 8 + (v["ijk"][:, 2] - 16)
    assert np.array_equal(n, np.arange(512))


def test_negative_tiles_straddle_zero():
    c = np.array([[-1, -1, -1], [0, 0, 0], [-4096, 0, 0], [4095, 0, 0], [-1, 0, 0]], np.int32)
    g = oracle.Grid.build(c, [0, 5])
    v = g.voxels()
    # tiles (-1,-1,-1) < (-1,0,0) < (0,0,0); inside a tile, children in x-major order
    order = [tuple(r) for r in v["ijk"].tolist()]
    assert order == [(-1, -1, -1), (-4096, 0, 0), (-1, 0, 0), (0, 0, 0), (4095, 0, 0)]
    up = g.upper()
    assert up["origin"].tolist() == [[-4096, -4096, -4096], [-4096, 0, 0], [0, 0, 0]]
    _check_topology(g, c, [0, 5])


def test_two_batches_identical_coords():
    rng = np.random.default_rng(7)
    c = rng.integers(0, 30, size=(600, 3)).astype(np.int32)
    coords = np.concatenate([c, c[::-1]])
    g = oracle.Grid.build(coords, [0, 600, 1200])
    v = _check_topology(g, coords, [0, 600, 1200])
    U1 = v["voxel_batch_offsets"][1]
    assert g.n_active == 2 * U1
    assert np.array_equal(v["ijk"][:U1], v["ijk"][U1:])
    assert np.array_equal(v["row_to_index"][600:], v["row_to_index"][:600][::-1] + U1)


def test_empty_batch_element():
    c = np.array([[1, 2, 3], [1, 2, 3], [9, 9, 9]], np.int32)
    g = oracle.Grid.build(c, [0, 2, 2, 3])
    v = _check_topology(g, c, [0, 2, 2, 3])
    assert v["voxel_batch_offsets"].tolist() == [0, 1, 1, 2]


@pytest.mark.parametrize("stride", [1, 2])
@pytest.mark.parametrize("seed", [0, 1])
def test_kmap_brute_force(stride, seed):
    coords, offs = _random_grid(seed + 10, n=700, span=14, lo=-7, B=2, dup=0.1)
    gin = oracle.Grid.build(coords, offs)
    gout = gin if stride == 1 else gin.coarsen(2)
    km = oracle.KernelMap(gin, gout, stride)
    vi, vo = gin.voxels(), gout.voxels()
    bf = H.brute_force_pairs(vi["ijk"], vi["batch"], vo["ijk"], vo["batch"], stride)
    assert H.kmap_triples(km.offsets, km.in_idx, km.out_idx) == bf
    # within each list, outputs ascend
    for s in range(27):
        seg = km.out_idx[km.offsets[s]:km.offsets[s + 1]]
        assert np.all(np.diff(seg) > 0)
    # mask bit s <=> a pair in list s for that output
    m = np.zeros(km.n_out, np.uint32)
    for s, p, q in bf:
        m[q] |= np.uint32(1 << s)
    assert np.array_equal(m, km.mask)
    if stride == 1:
        # symmetry (p,q) in s <=> (q,p) in 26-s; the centre list is the identity
        tr = set(bf)
        assert all((26 - s, q, p) in tr for s, p, q in bf)
        c = km.in_idx[km.offsets[13]:km.offsets[14]]
        assert np.array_equal(c, np.arange(gin.n_active)) and np.array_equal(
            km.out_idx[km.offsets[13]:km.offsets[14]], np.arange(gin.n_active))
    else:
        # every input voxel reaches its own floor(ijk/2) output through d in {0,1}^3
        assert np.all(km.mask != 0)


def test_coarsen_is_unique_floor_half():
    coords, offs = _random_grid(21, n=1500, span=30, lo=-15, B=2)
    g = oracle.Grid.build(coords, offs)
    c = g.coarsen(2)
    v, vc = g.voxels(), c.voxels()
    exp = np.unique(np.concatenate([v["batch"][:, None], np.floor_divide(v["ijk"], 2)], axis=1).astype(np.int64),
                    axis=0)
    got = np.unique(np.concatenate([vc["batch"][:, None], vc["ijk"]], axis=1).astype(np.int64), axis=0)
    assert np.array_equal(exp, got)


@pytest.mark.parametrize("stride,cin,cout", [(1, 5, 7), (2, 4, 6), (1, 16, 16)])
def test_conv_matches_dense_conv3d(stride, cin, cout):
    coords, offs = _random_grid(31 + stride, n=900, span=16, lo=-9, B=1, dup=0.0)
    gin = oracle.Grid.build(coords, offs)
    gout = gin if stride == 1 else gin.coarsen(2)
    km = oracle.KernelMap(gin, gout, stride)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((gin.n_active, cin))
    W = rng.standard_normal((27, cin, cout))
    y, a = oracle.conv(km, x, W)
    ref = H.dense_conv_active(gin.voxels()["ijk"], x, W, gout.voxels()["ijk"], stride)
    assert np.max(np.abs(y - ref)) <= 1e-12 * max(1.0, np.max(a))
    assert np.all(np.abs(y) <= a + 1e-12)
    # the sampled-row variant gives the same rows
    rows = rng.choice(gout.n_active, size=50, replace=False)
    yr, ar = oracle.conv_rows(gin, gout, stride, rows, x, W)
    assert np.allclose(yr, y[rows], rtol=0, atol=1e-12) and np.allclose(ar, a[rows], rtol=0, atol=1e-12)


@pytest.mark.parametrize("stride,transposed", [(1, False), (2, False), (2, True)])
def test_conv_tolerance_scale_is_abs_conv(stride, transposed):
    """The per-element scale a[q, co] = sum over pairs and channels of |x w|,
    which every conv tolerance multiplies, is the convolution of |x| with |W|
    ("fVDB" reading notes, Sparse-convolution operators: the sum that defines
    each output).  Pinned to torch's dense conv3d (conv_transpose3d for the
    transposed map) of the absolute inputs, so an a that is off by any factor
    (counted twice, accumulated into the wrong row, taken from one offset only)
    fails here, not just an a that is too small."""
    coords, offs = _random_grid(33 + stride + 10 * transposed, n=900, span=16, lo=-9, B=1, dup=0.0)
    fine = oracle.Grid.build(coords, offs)
    coarse = fine if stride == 1 else fine.coarsen(2)
    gin, gout = (coarse, fine) if transposed else (fine, coarse)
    km = oracle.KernelMap(gin, gout, stride, transposed=transposed)
    rng = np.random.default_rng(6)
    cin, cout = 5, 3
    x = rng.standard_normal((gin.n_active, cin))
    W = rng.standard_normal((27, cin, cout))
    _, a = oracle.conv(km, x, W)
    dense = H.dense_conv_transpose_active if transposed else H.dense_conv_active
    ref = dense(gin.voxels()["ijk"], np.abs(x), np.abs(W), gout.voxels()["ijk"], stride)
    assert np.max(np.abs(a - ref)) <= 1e-12 * np.max(ref)
    assert np.max(np.abs(2.0 * a - ref)) > 0.1 * np.max(ref)  # the check sees a factor of 2
    if not transposed:
        rows = rng.choice(gout.n_active, size=40, replace=False)
        _, ar = oracle.conv_rows(gin, gout, stride, rows, x, W)
        assert np.max(np.abs(ar - ref[rows])) <= 1e-12 * np.max(ref)


@pytest.mark.parametrize("stride", [1, 2])
def test_wgrad_tolerance_scale_is_abs_wgrad(stride):
    """The weight gradient's tolerance scale, conv_wgrad(|x|, |dy|) = sum over
    pairs of |x[p]|^T |dy[q]|, equals torch autograd's weight gradient of the
    dense conv3d with the absolute inputs."""
    coords, offs = _random_grid(95 + stride, n=700, span=14, lo=-7, B=1, dup=0.0)
    fine = oracle.Grid.build(coords, offs)
    coarse = fine if stride == 1 else fine.coarsen(2)
    km = oracle.KernelMap(fine, coarse, stride)
    rng = np.random.default_rng(9)
    x = rng.standard_normal((fine.n_active, 4))
    dy = rng.standard_normal((coarse.n_active, 6))
    a = oracle.conv_wgrad(km, np.abs(x), np.abs(dy))
    ref = H.dense_conv_wgrad(fine.voxels()["ijk"], np.abs(x), coarse.voxels()["ijk"], np.abs(dy), stride, 4, 6)
    assert np.max(np.abs(a - ref)) <= 1e-12 * np.max(ref)
    assert np.max(np.abs(2.0 * a - ref)) > 0.1 * np.max(ref)


def test_conv_identity_and_ones():
    coords, offs = _random_grid(41, n=800, span=12, lo=0, B=1, dup=0.0)
    g = oracle.Grid.build(coords, offs)
    km = oracle.KernelMap(g, g, 1)
    C = 6
    x = np.random.default_rng(0).standard_normal((g.n_active, C))
    W = np.zeros((27, C, C))
    W[13] = np.eye(C)
    y, _ = oracle.conv(km, x, W)
    assert np.array_equal(y, x)
    y1, _ = oracle.conv(km, np.ones((g.n_active, C)), np.ones((27, C, C)))
    per_out = np.array([bin(int(m)).count("1") for m in km.mask])
    assert np.array_equal(y1, np.repeat((per_out * C)[:, None], C, axis=1).astype(np.float64))


def test_dense_check_detects_flipped_kernel():
    """The dense conv3d pin is sensitive to the offset convention: flipping the
    kernel (true convolution instead of cross-correlation) or swapping the
    channel axes of W must fail it."""
    coords, offs = _random_grid(51, n=600, span=10, lo=-5, B=1, dup=0.0)
    g = oracle.Grid.build(coords, offs)
    km = oracle.KernelMap(g, g, 1)
    rng = np.random.default_rng(1)
    C = 4
    x = rng.standard_normal((g.n_active, C))
    W = rng.standard_normal((27, C, C))
    ref = H.dense_conv_active(g.voxels()["ijk"], x, W, g.voxels()["ijk"], 1)
    y_flip, _ = oracle.conv(km, x, W[::-1].copy())
    y_tr, _ = oracle.conv(km, x, W.transpose(0, 2, 1).copy())
    assert np.max(np.abs(y_flip - ref)) > 1e-3
    assert np.max(np.abs(y_tr - ref)) > 1e-3


def _pairs_python_ints(vin, vout, stride, transposed):
    """Brute-force (slot, in, out) triples in Python integers (no fixed-width
    arithmetic, so no wrap-around at the int32 edges)."""
    index = {(int(b), *map(int, ijk)): n for n, (b, ijk) in enumerate(zip(vin["batch"], vin["ijk"]))}
    out = set()
    for q, (b, ijk) in enumerate(zip(vout["batch"], vout["ijk"])):
        for s in range(27):
            d = (s // 9 - 1, (s // 3) % 3 - 1, s % 3 - 1)
            if transposed:
                c = [int(x) - e for x, e in zip(ijk, d)]
                if any(v % stride for v in c):
                    continue
                c = [v // stride for v in c]
            else:
                c = [stride * int(x) + e for x, e in zip(ijk, d)]
            p = index.get((int(b), *c))
            if p is not None:
                out.add((s, p, q))
    return out


@pytest.mark.parametrize("stride", [1, 2])
@pytest.mark.parametrize("transposed", [False, True])
def test_kmap_int32_edges_do_not_wrap(stride, transposed):
    """Voxels at both ends of the int32 range in one batch: a neighbour
    position past an end is no voxel (IndexGrid coordinates are int32 ijk), so
    2^31 - 1 and -2^31 never pair."""
    M = 2 ** 31 - 1
    c = np.array([[M, 0, 0], [-M - 1, 0, 0], [M - 1, 0, 0], [M, M, M], [-M - 1, -M - 1, -M - 1],
                  [-M - 1, M, 0], [M, -M - 1, 5]], np.int32)
    fine = oracle.Grid.build(c, [0, len(c)])
    coarse = fine if stride == 1 else fine.coarsen(2)
    gi, go = (coarse, fine) if transposed else (fine, coarse)
    km = oracle.KernelMap(gi, go, stride, transposed=transposed)
    exp = _pairs_python_ints(gi.voxels(), go.voxels(), stride, transposed)
    assert H.kmap_triples(km.offsets, km.in_idx, km.out_idx) == sorted(exp)
    if stride == 1:  # only the centre pairs and the one pair along i at the top
        assert len(exp) == len(c) + 2


# ------------------------------------------------------------ transposed conv, backward, refine
@pytest.mark.parametrize("stride", [1, 2])
def test_transposed_map_is_swapped_forward_map(stride):
    """Pairs of the transposed map (output p of the fine grid, input q of the
    coarse one) = pairs of the forward map with input and output swapped, per
    offset list, ordered by p."""
    coords, offs = _random_grid(61 + stride, n=2500, span=30, lo=-15, B=2)
    fine = oracle.Grid.build(coords, offs)
    coarse = fine if stride == 1 else fine.coarsen(2)
    fwd = oracle.KernelMap(fine, coarse, stride)
    tr = oracle.KernelMap(coarse, fine, stride, transposed=True)
    assert tr.n_pairs == fwd.n_pairs
    assert np.array_equal(np.diff(tr.offsets), np.diff(fwd.offsets))
    for s in range(27):
        a, b = fwd.offsets[s], fwd.offsets[s + 1]
        c, d = tr.offsets[s], tr.offsets[s + 1]
        exp = np.stack([fwd.out_idx[a:b], fwd.in_idx[a:b]], 1)  # (in, out) of the transposed map
        exp = exp[np.argsort(exp[:, 1], kind="stable")]
        got = np.stack([tr.in_idx[c:d], tr.out_idx[c:d]], 1)
        assert np.array_equal(exp, got), s
        assert np.all(np.diff(tr.out_idx[c:d]) > 0)
    # mask bit s of output p: p has a pair in list s
    for s in range(27):
        c, d = tr.offsets[s], tr.offsets[s + 1]
        m = np.zeros(fine.n_active, bool)
        m[tr.out_idx[c:d]] = True
        assert np.array_equal(m, (tr.mask >> s) & 1 == 1)


@pytest.mark.parametrize("stride,cin,cout", [(2, 4, 6), (1, 5, 3)])
def test_transposed_conv_matches_dense_conv_transpose3d(stride, cin, cout):
    coords, offs = _random_grid(71 + stride, n=900, span=16, lo=-9, B=1, dup=0.0)
    fine = oracle.Grid.build(coords, offs)
    coarse = fine if stride == 1 else fine.coarsen(2)
    tr = oracle.KernelMap(coarse, fine, stride, transposed=True)
    rng = np.random.default_rng(6)
    x = rng.standard_normal((coarse.n_active, cin))
    W = rng.standard_normal((27, cin, cout))
    y, a = oracle.conv(tr, x, W)
    ref = H.dense_conv_transpose_active(coarse.voxels()["ijk"], x, W, fine.voxels()["ijk"], stride)
    assert np.max(np.abs(y - ref)) <= 1e-12 * max(1.0, np.max(a))


@pytest.mark.parametrize("stride", [1, 2])
def test_adjoint_identity(stride):
    """<conv(u; K, W), v> = <u, conv(v; K^T, W^T)>: the transposed map with the
    per-offset transposed weights is the adjoint (the input gradient)."""
    coords, offs = _random_grid(81 + stride, n=1200, span=18, lo=-9, B=2)
    fine = oracle.Grid.build(coords, offs)
    coarse = fine if stride == 1 else fine.coarsen(2)
    fwd = oracle.KernelMap(fine, coarse, stride)
    tr = oracle.KernelMap(coarse, fine, stride, transposed=True)
    rng = np.random.default_rng(7)
    u = rng.standard_normal((fine.n_active, 5))
    v = rng.standard_normal((coarse.n_active, 3))
    W = rng.standard_normal((27, 5, 3))
    y, _ = oracle.conv(fwd, u, W)
    z, _ = oracle.conv(tr, v, W.transpose(0, 2, 1).copy())
    lhs, rhs = float(np.sum(y * v)), float(np.sum(u * z))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))
    # a transposed map built with the forward (unmirrored) offsets breaks it
    if stride == 1:
        z_bad, _ = oracle.conv(fwd, v, W.transpose(0, 2, 1).copy())
        assert abs(float(np.sum(u * z_bad)) - lhs) > 1e-6


@pytest.mark.parametrize("stride,cin,cout", [(1, 4, 5), (2, 3, 4)])
def test_wgrad_matches_autograd(stride, cin, cout):
    coords, offs = _random_grid(91 + stride, n=800, span=14, lo=-7, B=1, dup=0.0)
    fine = oracle.Grid.build(coords, offs)
    coarse = fine if stride == 1 else fine.coarsen(2)
    km = oracle.KernelMap(fine, coarse, stride)
    rng = np.random.default_rng(8)
    x = rng.standard_normal((fine.n_active, cin))
    dy = rng.standard_normal((coarse.n_active, cout))
    dW = oracle.conv_wgrad(km, x, dy)
    ref = H.dense_conv_wgrad(fine.voxels()["ijk"], x, coarse.voxels()["ijk"], dy, stride, cin, cout)
    assert np.max(np.abs(dW - ref)) <= 1e-10 * max(1.0, np.max(np.abs(ref)))


def test_refine_is_all_children():
    coords, offs = _random_grid(99, n=700, span=20, lo=-10, B=2)
    g = oracle.Grid.build(coords, offs)
    r = g.refine(2)
    v, vr = g.voxels(), r.voxels()
    kids = np.stack(np.meshgrid(*[np.arange(2)] * 3, indexing="ij"), -1).reshape(-1, 3)
    exp = (2 * v["ijk"][:, None, :].astype(np.int64) + kids[None]).reshape(-1, 3)
    eb = np.repeat(v["batch"], 8)
    exp = np.unique(np.concatenate([eb[:, None], exp], 1), axis=0)
    got = np.unique(np.concatenate([vr["batch"][:, None], vr["ijk"]], 1).astype(np.int64), axis=0)
    assert np.array_equal(exp, got)
    assert r.n_active == 8 * g.n_active  # children of distinct voxels are distinct
    assert np.array_equal(r.coarsen(2).voxels()["ijk"], v["ijk"])

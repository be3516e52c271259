"""The full-size checkers against the oracle, on the CPU.

At the sizes the benchmark times, the GPU tests cannot run the oracle; they
check the CUDA path against independent numpy derivations instead
(`tests/gpu_common.py`: the tree derived from the sorted canonical keys, every
output's 27 neighbours by searchsorted, sampled conv rows in fp64).  Here those
checkers are run on the oracle's own results for small grids, wrapped in the
shape the CUDA path's objects have: they must accept the oracle's results and
reject a result with one planted mistake.  This pins the checkers (a checker
that accepts anything would hide a GPU error) and gives the oracle's build and
kernel map one more independent derivation to agree with.
"""
import numpy as np
import pytest

import oracle
from tests import gpu_common as G
from tests import helpers as H


class _Grid:
    """The oracle's grid with the CUDA grid's accessors (CPU tensors)."""

    def __init__(self, og, mutate=None):
        import torch

        v, lf, lo, up = og.voxels(), og.leaves(), og.lower(), og.upper()
        rec = np.concatenate([lf["mask"], lf["first"][:, None], lf["prefix9"][:, None]], axis=1)
        t = dict(ijk=v["ijk"], row_to_index=v["row_to_index"], voxel_batch_offsets=v["voxel_batch_offsets"],
                 leaf_origin=lf["origin"], leaf_batch=lf["batch"], leaf_records=rec.view(np.int64))
        for name, d in (("lower", lo), ("upper", up)):
            t[f"{name}_origin"], t[f"{name}_batch"] = d["origin"], d["batch"]
            t[f"{name}_mask"] = d["mask"].view(np.int64)
            t[f"{name}_prefix"] = d["prefix"].view(np.int32)
            t[f"{name}_first"] = d["first"].view(np.int32)
        if mutate:
            mutate(t)
        self._t = {k: torch.from_numpy(np.ascontiguousarray(a)) for k, a in t.items()}
        self.n_active, self.n_leaf, self.n_lower, self.n_upper = og.n_active, og.n_leaf, og.n_lower, og.n_upper

    def topology(self):
        return self._t


class _KernelMap:
    """The oracle's kernel map with the CUDA map's accessors."""

    def __init__(self, okm, mutate=None):
        import torch

        ii, oo, mm = okm.in_idx.copy(), okm.out_idx.copy(), okm.mask.copy()
        self.offsets = okm.offsets.copy()
        if mutate:
            ii, oo, mm = mutate(ii, oo, mm, self.offsets)
        self._p = tuple(torch.from_numpy(np.ascontiguousarray(a)) for a in (ii, oo, mm.view(np.int32)))
        self.n_pairs = int(self.offsets[27])

    def pairs(self):
        return self._p


def _coords(seed, n=4000, span=40, lo=-20, B=2):
    rng = np.random.default_rng(seed)
    c = rng.integers(lo, lo + span, size=(n, 3)).astype(np.int32)
    c = np.concatenate([c, c[: n // 5]])  # duplicate rows
    cuts = np.sort(rng.choice(np.arange(1, len(c)), size=B - 1, replace=False)) if B > 1 else []
    return c, np.array([0, *cuts, len(c)], np.int64)


def _out_grid(og, stride):
    if stride == 1:
        return og
    return og.coarsen(2)


def _ijk_batch(og):
    v = og.voxels()
    return v["ijk"], np.repeat(np.arange(og.B), np.diff(v["voxel_batch_offsets"]))


@pytest.mark.parametrize("seed,span,lo", [(1, 40, -20), (2, 300, -150), (3, 9000, -4500)])
def test_build_checker_accepts_the_oracle(seed, span, lo):
    """Dense, sparse and multi-root-tile grids (span 9000 crosses several
    4096-voxel root tiles on each axis)."""
    coords, offs = _coords(seed, span=span, lo=lo)
    og = oracle.Grid.build(coords, offs)
    uniq, ijk, vb = G.check_build_full(_Grid(og), coords, offs)
    assert uniq.shape[0] == og.n_active
    assert np.array_equal(H.key64(vb, ijk), uniq)


def _flip_leaf_bit(t):
    rec = t["leaf_records"].copy()
    rec[0, 0] ^= 1 << 5
    t["leaf_records"] = rec


def _bump_lower_prefix(t):
    p = t["lower_prefix"].copy()
    p[0, 5] += 1
    t["lower_prefix"] = p


def _swap_rows(t):
    r = t["row_to_index"].copy()
    i = int(np.flatnonzero(r != r[0])[0])
    r[0], r[i] = r[i], r[0]
    t["row_to_index"] = r


def _shift_leaf_origin(t):
    o = t["leaf_origin"].copy()
    o[-1, 2] += 8
    t["leaf_origin"] = o


@pytest.mark.parametrize("mutate", [_flip_leaf_bit, _bump_lower_prefix, _swap_rows, _shift_leaf_origin])
def test_build_checker_rejects_a_planted_mistake(mutate):
    coords, offs = _coords(4)
    og = oracle.Grid.build(coords, offs)
    with pytest.raises(AssertionError):
        G.check_build_full(_Grid(og, mutate), coords, offs)


@pytest.mark.parametrize("stride", [1, 2])
def test_kmap_checker_accepts_the_oracle(stride):
    coords, offs = _coords(5, span=60, lo=-30)
    og = oracle.Grid.build(coords, offs)
    uniq, _, _ = G.check_build_full(_Grid(og), coords, offs)
    gout = _out_grid(og, stride)
    ijk_out, b_out = _ijk_batch(gout)
    G.check_kmap_full(_KernelMap(oracle.KernelMap(og, gout, stride)), uniq, ijk_out, b_out, stride)


def _drop_pair(ii, oo, mm, offs):
    s = int(np.argmax(np.diff(offs)))  # the longest list
    k = int(offs[s])
    keep = np.ones(ii.shape[0], bool)
    keep[k] = False
    offs[s + 1:] -= 1
    return ii[keep], oo[keep], mm


def _wrong_input(ii, oo, mm, offs):
    ii = ii.copy()
    ii[offs[13]] += 1
    return ii, oo, mm


def _wrong_mask(ii, oo, mm, offs):
    mm = mm.copy()
    mm[0] ^= np.uint32(1 << 13)
    return ii, oo, mm


@pytest.mark.parametrize("mutate", [_drop_pair, _wrong_input, _wrong_mask])
def test_kmap_checker_rejects_a_planted_mistake(mutate):
    coords, offs = _coords(6, span=50, lo=-25)
    og = oracle.Grid.build(coords, offs)
    uniq, ijk, vb = G.check_build_full(_Grid(og), coords, offs)
    with pytest.raises(AssertionError):
        G.check_kmap_full(_KernelMap(oracle.KernelMap(og, og, 1), mutate), uniq, ijk, vb, 1)


@pytest.mark.parametrize("stride", [1, 2])
def test_sampled_conv_rows_match_the_oracle(stride):
    """The neighbours found by searchsorted and the fp64 rows built from them
    equal the oracle's conv on every output row (and its sum|w*x| scale)."""
    coords, offs = _coords(7, span=50, lo=-25)
    og = oracle.Grid.build(coords, offs)
    uniq = np.unique(H.key64(np.repeat(np.arange(len(offs) - 1), np.diff(offs)), coords))
    gout = _out_grid(og, stride)
    ijk_out, b_out = _ijk_batch(gout)
    rng = np.random.default_rng(8)
    x = rng.standard_normal((og.n_active, 8))
    W = rng.standard_normal((27, 8, 5))
    rows = np.arange(gout.n_active)
    nbr = G.neighbours_independent(uniq, ijk_out, b_out, stride, rows)
    y, a = G.conv_rows_independent(nbr, x, W)
    yo, ao = oracle.conv(oracle.KernelMap(og, gout, stride), x, W)
    assert np.allclose(y, yo, rtol=0, atol=1e-12 * max(1.0, float(np.abs(ao).max())))
    assert np.allclose(a, ao, rtol=1e-12, atol=0)

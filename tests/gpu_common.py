"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the oracle (small sizes) or with independent numpy
derivations and properties (full sizes)."""
from __future__ import annotations

import numpy as np

from tests import helpers as H

BF16_TOL = 2e-3   # |y - y_ref| <= 2e-3 * sum|w*x|  (bf16-rounded inputs, fp32 accumulation, fp32 output)
F32_TOL = 1e-5    # |y - y_ref| <= 1e-5 * sum|w*x|  (exact fp32 FFMA)
# A bf16 output adds one rounding of the fp32 result: bf16 keeps 8 significant
# bits, so round-to-nearest moves y by at most 2^-8 |y| (relative to the exact
# y_ref that is 2^-8 (|y_ref| + err) <= 2^-8 |y_ref| (1 + 2e-3)).
BF16_OUT_REL = 2.0 ** -8 * (1 + 2e-3)


def np_(t):
    return t.detach().cpu().numpy()


def gpu_grid(coords, offs):
    import torch

    import sparse_convolution_gb300 as fvx

    return fvx.Grid.build(torch.from_numpy(np.ascontiguousarray(coords, np.int32)).cuda(), np.asarray(offs))


def assert_topology_equal(g, og):
    """Bit-exact comparison of every topology array with the oracle's."""
    assert g.counts() == og.counts(), (g.counts(), og.counts())
    t = {k: np_(v) for k, v in g.topology().items()}
    v = og.voxels()
    assert np.array_equal(t["ijk"], v["ijk"])
    assert np.array_equal(t["row_to_index"], v["row_to_index"])
    assert np.array_equal(t["voxel_batch_offsets"], v["voxel_batch_offsets"])
    lf = og.leaves()
    assert np.array_equal(t["leaf_origin"], lf["origin"])
    assert np.array_equal(t["leaf_batch"], lf["batch"])
    rec = t["leaf_records"].astype(np.uint64)
    assert np.array_equal(rec[:, :8], lf["mask"])
    assert np.array_equal(rec[:, 8], lf["first"])
    assert np.array_equal(rec[:, 9], lf["prefix9"])
    for lvl, od in (("lower", og.lower()), ("upper", og.upper())):
        assert np.array_equal(t[f"{lvl}_origin"], od["origin"]), lvl
        assert np.array_equal(t[f"{lvl}_batch"], od["batch"]), lvl
        assert np.array_equal(t[f"{lvl}_mask"].astype(np.uint64), od["mask"]), lvl
        assert np.array_equal(t[f"{lvl}_prefix"].astype(np.uint32), od["prefix"]), lvl
        assert np.array_equal(t[f"{lvl}_first"].astype(np.uint32), od["first"]), lvl


def assert_kmap_equal(km, okm):
    ii, oo, mm = km.pairs()
    assert np.array_equal(km.offsets, okm.offsets)
    assert np.array_equal(np_(ii), okm.in_idx)
    assert np.array_equal(np_(oo), okm.out_idx)
    assert np.array_equal(np_(mm).astype(np.uint32), okm.mask)


def assert_conv_close(y, y_ref, a_ref, tol, rel_y=0.0):
    y = np.asarray(y, np.float64)
    err = np.abs(y - y_ref)
    bound = tol * a_ref + rel_y * np.abs(y_ref)
    bad = err > bound
    if bad.any():
        i = np.argmax(err - bound)
        raise AssertionError(f"{int(bad.sum())} elements out of tolerance; worst flat index {i}: "
                             f"got {y.flat[i]}, ref {y_ref.flat[i]}, scale {a_ref.flat[i]}")


def bf16_inputs(seed, n, cin, cout, kind="normal"):
    import torch

    from sparse_convolution_gb300 import synth

    x = torch.from_numpy(synth.features(seed, n, cin, kind)).cuda().bfloat16()
    W = torch.from_numpy(synth.weights(seed + 1, cin, cout)).cuda().bfloat16()
    return x, W


def as_f64(t):
    return np_(t.float()).astype(np.float64)


# ---------------------------------------------------------------- full-size checks (no oracle)

def derive_topology(uniq):
    """Independent numpy derivation of the tree from the sorted canonical keys
    (``helpers.key64``): leaves are runs of key >> 9, lower nodes runs of
    key >> 21, upper nodes runs of key >> 36."""
    out = {}
    U = uniq.shape[0]
    leafkey = uniq >> 9
    lstart = np.flatnonzero(np.concatenate([[True], leafkey[1:] != leafkey[:-1]]))
    L = lstart.shape[0]
    leaf_of = np.repeat(np.arange(L), np.diff(np.concatenate([lstart, [U]])))
    n = (uniq & 511).astype(np.int64)
    word = leaf_of * 8 + (n >> 6)
    bits = np.left_shift(np.uint64(1), (n & 63).astype(np.uint64))
    gstart = np.flatnonzero(np.concatenate([[True], word[1:] != word[:-1]]))
    mask = np.zeros(L * 8, np.uint64)
    mask[word[gstart]] = np.bitwise_or.reduceat(bits, gstart)
    mask = mask.reshape(L, 8)
    pc = H.popcount64(mask)
    cum = np.cumsum(pc, axis=1)
    prefix9 = np.zeros(L, np.uint64)
    for w in range(1, 8):
        prefix9 |= cum[:, w - 1].astype(np.uint64) << np.uint64(9 * (w - 1))
    out["leaf_mask"], out["leaf_first"], out["leaf_prefix9"] = mask, lstart.astype(np.uint64), prefix9
    out["n_leaf"] = L

    def level(child_key, shift_bits, words):
        parent = child_key >> shift_bits
        pstart = np.flatnonzero(np.concatenate([[True], parent[1:] != parent[:-1]]))
        NP = pstart.shape[0]
        par_of = np.repeat(np.arange(NP), np.diff(np.concatenate([pstart, [child_key.shape[0]]])))
        nb = (child_key & ((1 << shift_bits) - 1)).astype(np.int64)
        wd = par_of * words + (nb >> 6)
        bt = np.left_shift(np.uint64(1), (nb & 63).astype(np.uint64))
        gs = np.flatnonzero(np.concatenate([[True], wd[1:] != wd[:-1]]))
        m = np.zeros(NP * words, np.uint64)
        m[wd[gs]] = np.bitwise_or.reduceat(bt, gs)
        m = m.reshape(NP, words)
        p = H.popcount64(m)
        pre = (np.cumsum(p, axis=1) - p).astype(np.uint32)
        return parent[pstart], m, pre, pstart.astype(np.uint32)

    leaf_keys = leafkey[lstart]
    lower_keys, out["lower_mask"], out["lower_prefix"], out["lower_first"] = level(leaf_keys, 12, 64)
    _, out["upper_mask"], out["upper_prefix"], out["upper_first"] = level(lower_keys, 15, 512)
    out["n_lower"] = lower_keys.shape[0]
    out["n_upper"] = out["upper_first"].shape[0]
    return out


def check_build_full(g, coords, offs):
    """Full-size bit-exact build check against numpy derivations."""
    b_rows = np.repeat(np.arange(len(offs) - 1), np.diff(offs))
    keys_rows = H.key64(b_rows, coords)
    uniq = np.unique(keys_rows)
    assert g.n_active == uniq.shape[0]
    t = {k: np_(v) for k, v in g.topology().items()}
    vbo = t["voxel_batch_offsets"]
    vb = np.repeat(np.arange(len(offs) - 1), np.diff(vbo))
    assert np.array_equal(H.key64(vb, t["ijk"]), uniq), "ijk_of_index is not the sorted unique set"
    assert np.array_equal(uniq[t["row_to_index"]], keys_rows), "row_to_index"
    d = derive_topology(uniq)
    assert (g.n_leaf, g.n_lower, g.n_upper) == (d["n_leaf"], d["n_lower"], d["n_upper"])
    rec = t["leaf_records"].astype(np.uint64)
    assert np.array_equal(rec[:, :8], d["leaf_mask"])
    assert np.array_equal(rec[:, 8], d["leaf_first"])
    assert np.array_equal(rec[:, 9], d["leaf_prefix9"])
    assert np.array_equal(t["leaf_origin"], t["ijk"][d["leaf_first"].astype(np.int64)] & ~7)
    for lvl in ("lower", "upper"):
        assert np.array_equal(t[f"{lvl}_mask"].astype(np.uint64), d[f"{lvl}_mask"]), lvl
        assert np.array_equal(t[f"{lvl}_prefix"].astype(np.uint32), d[f"{lvl}_prefix"]), lvl
        assert np.array_equal(t[f"{lvl}_first"].astype(np.uint32), d[f"{lvl}_first"]), lvl
    return uniq, t["ijk"], vb


def neighbours_independent(uniq_in, ijk_out, b_out, stride, rows):
    """For output rows `rows`: the 27 input indices (or -1), by searchsorted in
    the sorted canonical keys of the input grid."""
    res = np.full((rows.shape[0], 27), -1, np.int64)
    for s in range(27):
        d = np.array([s // 9 - 1, (s // 3) % 3 - 1, s % 3 - 1])
        c = stride * ijk_out[rows].astype(np.int64) + d
        k = H.key64(b_out[rows], c)
        pos = np.searchsorted(uniq_in, k)
        pos = np.minimum(pos, uniq_in.shape[0] - 1)
        hit = uniq_in[pos] == k
        res[hit, s] = pos[hit]
    return res


def check_kmap_full(km, uniq_in, ijk_out, b_out, stride):
    """Every output's 27 neighbours, list by list: list s must hold exactly
    the outputs whose position stride*ijk + d_s is an input voxel, in
    ascending order, each with that voxel's index (searchsorted in the sorted
    canonical keys of the input grid); the masks must agree."""
    ii, oo, mm = (np_(t) for t in km.pairs())
    offs = km.offsets
    assert offs[0] == 0 and np.all(np.diff(offs) >= 0) and offs[27] == km.n_pairs
    n_out = ijk_out.shape[0]
    mask = np.zeros(n_out, np.uint32)
    base = stride * ijk_out.astype(np.int64)
    last = uniq_in.shape[0] - 1
    for s in range(27):
        d = np.array([s // 9 - 1, (s // 3) % 3 - 1, s % 3 - 1], np.int64)
        k = H.key64(b_out, base + d)
        pos = np.searchsorted(uniq_in, k)
        np.minimum(pos, last, out=pos)
        hit = uniq_in[pos] == k
        seg_o = oo[offs[s]:offs[s + 1]]
        seg_i = ii[offs[s]:offs[s + 1]]
        assert np.array_equal(seg_o, np.flatnonzero(hit)), f"list {s}: outputs"
        assert np.array_equal(seg_i, pos[hit]), f"list {s}: inputs"
        mask[hit] |= np.uint32(1 << s)
    assert np.array_equal(mm.astype(np.uint32), mask)


def conv_rows_independent(nbr, x64, W64):
    """y, a for sampled rows from their 27 neighbour indices (numpy fp64)."""
    cout = W64.shape[2]
    y = np.zeros((nbr.shape[0], cout))
    a = np.zeros((nbr.shape[0], cout))
    for s in range(27):
        sel = nbr[:, s] >= 0
        if not sel.any():
            continue
        xs = x64[nbr[sel, s]]
        y[sel] += xs @ W64[s]
        a[sel] += np.abs(xs) @ np.abs(W64[s])
    return y, a

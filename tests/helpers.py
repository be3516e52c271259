"""Independent checkers used by the tests (numpy / torch CPU only).

Nothing here is shared with the CUDA path or with the oracle's C++: the tree
walk, the canonical-order check, the brute-force neighbour search and the
dense-conv check are written from the definitions, so that they can pin both.
"""
from __future__ import annotations

import numpy as np

UPPER, LOWER, LEAF = 4096, 128, 8  # node extents; fanouts 32, 16, 8


def popcount64(x):
    x = np.asarray(x, dtype=np.uint64)
    if hasattr(np, "bitwise_count"):
        return np.bitwise_count(x).astype(np.int64)
    c = np.zeros(x.shape, np.int64)
    y = x.copy()
    for _ in range(64):
        c += (y & np.uint64(1)).astype(np.int64)
        y >>= np.uint64(1)
    return c


def canonical_tuples(batch, ijk):
    """13 order fields per voxel: batch, tile ijk, upper-child ijk, lower-child
    ijk, voxel-in-leaf ijk (tile = floor(c/4096), child = digits of c mod 4096)."""
    ijk = np.asarray(ijk, dtype=np.int64)
    tile = np.floor_divide(ijk, UPPER)
    o = np.mod(ijk, UPPER)
    cols = [np.asarray(batch, dtype=np.int64)]
    cols += [tile[:, a] for a in range(3)]
    cols += [o[:, a] // LOWER for a in range(3)]
    cols += [(o[:, a] % LOWER) // LEAF for a in range(3)]
    cols += [o[:, a] % LEAF for a in range(3)]
    return np.stack(cols, axis=1)


def strictly_increasing_rows(t):
    """True iff consecutive rows of the int matrix t are strictly increasing in
    lexicographic order."""
    if t.shape[0] < 2:
        return True
    a, b = t[:-1], t[1:]
    diff = a != b
    first = np.argmax(diff, axis=1)
    anydiff = diff.any(axis=1)
    rows = np.arange(a.shape[0])
    return bool(np.all(anydiff & (a[rows, first] < b[rows, first])))


def unique_voxels(coords, batch_offsets):
    """Unique (batch, i, j, k) rows of a CSR-batched coordinate array."""
    coords = np.asarray(coords, dtype=np.int64).reshape(-1, 3)
    offs = np.asarray(batch_offsets, dtype=np.int64)
    b = np.repeat(np.arange(len(offs) - 1), np.diff(offs))
    return np.unique(np.concatenate([b[:, None], coords], axis=1), axis=0)


def tree_lookup(upper, lower, leaves, batch, ijk):
    """Coordinate -> index by walking root -> upper -> lower -> leaf with the
    exported masks and prefix counts; -1 where a node or bit is absent."""
    ijk = np.asarray(ijk, dtype=np.int64).reshape(-1, 3)
    batch = np.asarray(batch, dtype=np.int64).reshape(-1)
    n = ijk.shape[0]
    out = np.full(n, -1, np.int64)
    # root: sorted (batch, origin) keys of the upper nodes, searched per query
    ukeys = np.concatenate([np.asarray(upper["batch"], np.int64)[:, None],
                            np.asarray(upper["origin"], np.int64)], axis=1)
    qkeys = np.concatenate([batch[:, None], ijk - np.mod(ijk, UPPER)], axis=1)
    uidx = np.full(n, -1, np.int64)
    if 0 < ukeys.shape[0] <= 64:
        for u in range(ukeys.shape[0]):
            uidx[np.all(qkeys == ukeys[u], axis=1)] = u
    elif ukeys.shape[0] > 64:
        allk = np.concatenate([ukeys, qkeys], axis=0)
        _, inv = np.unique(allk, axis=0, return_inverse=True)
        inv = inv.reshape(-1)
        pos = np.full(inv.max() + 1, -1, np.int64)
        pos[inv[:ukeys.shape[0]]] = np.arange(ukeys.shape[0])
        uidx = pos[inv[ukeys.shape[0]:]]
    ok = uidx >= 0

    def child(mask, prefix, first, node, nbit, words):
        w = nbit // 64
        bit = (nbit % 64).astype(np.uint64)
        m = mask.reshape(-1, words)[node, w]
        has = ((m >> bit) & np.uint64(1)) == np.uint64(1)
        below = m & ((np.uint64(1) << bit) - np.uint64(1))
        idx = first[node].astype(np.int64) + prefix.reshape(-1, words)[node, w].astype(np.int64) + popcount64(below)
        return has, idx

    o = np.mod(ijk, UPPER)
    nu = ((o[:, 0] // LOWER) * 32 + o[:, 1] // LOWER) * 32 + o[:, 2] // LOWER
    has, lidx = child(upper["mask"], upper["prefix"], upper["first"], np.where(ok, uidx, 0), nu, 512)
    ok &= has
    o = np.mod(ijk, LOWER)
    nl = ((o[:, 0] // LEAF) * 16 + o[:, 1] // LEAF) * 16 + o[:, 2] // LEAF
    has, fidx = child(lower["mask"], lower["prefix"], lower["first"], np.where(ok, lidx, 0), nl, 64)
    ok &= has
    o = np.mod(ijk, LEAF)
    nv = (o[:, 0] * 8 + o[:, 1]) * 8 + o[:, 2]
    f = np.where(ok, fidx, 0)
    w = nv // 64
    bit = (nv % 64).astype(np.uint64)
    m = leaves["mask"][f, w]
    has = ((m >> bit) & np.uint64(1)) == np.uint64(1)
    packed = leaves["prefix9"][f]
    shift = (np.maximum(w - 1, 0) * 9).astype(np.uint64)
    pre = np.where(w > 0, ((packed >> shift) & np.uint64(511)).astype(np.int64), 0)
    idx = leaves["first"][f].astype(np.int64) + pre + popcount64(m & ((np.uint64(1) << bit) - np.uint64(1)))
    ok &= has
    out[ok] = idx[ok]
    return out


def brute_force_pairs(ijk_in, b_in, ijk_out, b_out, stride):
    """All (s, p, q) with ijk_in[p] - stride*ijk_out[q] = d_s, same batch,
    by an O(U_in * U_out) scan; s = (di+1)*9 + (dj+1)*3 + (dk+1)."""
    ijk_in = np.asarray(ijk_in, dtype=np.int64)
    ijk_out = np.asarray(ijk_out, dtype=np.int64)
    res = []
    for q in range(ijk_out.shape[0]):
        d = ijk_in - stride * ijk_out[q]
        sel = np.nonzero(np.all(np.abs(d) <= 1, axis=1) & (np.asarray(b_in) == b_out[q]))[0]
        for p in sel:
            s = (d[p, 0] + 1) * 9 + (d[p, 1] + 1) * 3 + (d[p, 2] + 1)
            res.append((int(s), int(p), int(q)))
    return sorted(res)


def kmap_triples(offsets, in_idx, out_idx):
    res = []
    for s in range(27):
        for e in range(int(offsets[s]), int(offsets[s + 1])):
            res.append((s, int(in_idx[e]), int(out_idx[e])))
    return sorted(res)


def dense_conv_active(ijk_in, x, W, ijk_out, stride):
    """Dense conv3d (torch, float64, cross-correlation, padding 1) over a
    zero-filled box holding the input grid, read back at the active outputs.
    For stride 2 the box origin is even so that dense output o sits at input
    2*o - 1 .. 2*o + 1."""
    import torch

    ijk_in = np.asarray(ijk_in, dtype=np.int64)
    ijk_out = np.asarray(ijk_out, dtype=np.int64)
    lo = np.minimum(ijk_in.min(0), stride * ijk_out.min(0)) - 2
    lo = lo - np.mod(lo, 2)  # even origin
    hi = np.maximum(ijk_in.max(0), stride * ijk_out.max(0)) + 3
    size = hi - lo
    cin, cout = W.shape[1], W.shape[2]
    dense = torch.zeros((1, cin) + tuple(int(v) for v in size), dtype=torch.float64)
    rel = ijk_in - lo
    dense[0, :, rel[:, 0], rel[:, 1], rel[:, 2]] = torch.from_numpy(np.asarray(x, np.float64)).T
    # torch weight [cout, cin, kd, kh, kw]; slot s = kd*9 + kh*3 + kw
    wt = torch.from_numpy(np.asarray(W, np.float64)).reshape(3, 3, 3, cin, cout).permute(4, 3, 0, 1, 2).contiguous()
    y = torch.nn.functional.conv3d(dense, wt, stride=stride, padding=1)
    # dense output index o corresponds to coordinate lo/stride + o
    orel = ijk_out - lo // stride
    return y[0, :, orel[:, 0], orel[:, 1], orel[:, 2]].T.numpy()


def key64(batch, ijk):
    """Order-preserving int64 packing of the canonical tuple for data whose
    batch < 16 and root tiles lie in [-8, 8): batch | 3 tiles | 36 offset bits."""
    ijk = np.asarray(ijk, dtype=np.int64).reshape(-1, 3)
    b = np.asarray(batch, dtype=np.int64).reshape(-1)
    tile = np.floor_divide(ijk, UPPER)
    assert b.size == 0 or (b.min() >= 0 and b.max() < 16 and tile.min() >= -8 and tile.max() < 8)
    o = np.mod(ijk, UPPER)
    u, l, v = o // LOWER, (o % LOWER) // LEAF, o % LEAF
    off = ((u[:, 0] * 32 + u[:, 1]) * 32 + u[:, 2])
    off = (off * 16 + l[:, 0]) * 16 + l[:, 1]
    off = (off * 16 + l[:, 2]) * 8 + v[:, 0]
    off = (off * 8 + v[:, 1]) * 8 + v[:, 2]
    t = ((b * 16 + tile[:, 0] + 8) * 16 + tile[:, 1] + 8) * 16 + tile[:, 2] + 8
    return (t << 36) | off


def dense_conv_transpose_active(ijk_in, x, W, ijk_out, stride):
    """Dense conv_transpose3d (torch, float64, padding 1; output_padding 1 for
    stride 2) over a zero-filled box holding the input grid, read back at the
    active outputs: out[stride*i + d] += x[i] W[d] for d in {-1,0,1}^3."""
    import torch

    ijk_in = np.asarray(ijk_in, dtype=np.int64)
    ijk_out = np.asarray(ijk_out, dtype=np.int64)
    lo = np.minimum(ijk_in.min(0), np.floor_divide(ijk_out.min(0), stride)) - 2
    hi = np.maximum(ijk_in.max(0), np.floor_divide(ijk_out.max(0), stride)) + 3
    size = hi - lo
    cin, cout = W.shape[1], W.shape[2]
    dense = torch.zeros((1, cin) + tuple(int(v) for v in size), dtype=torch.float64)
    rel = ijk_in - lo
    dense[0, :, rel[:, 0], rel[:, 1], rel[:, 2]] = torch.from_numpy(np.asarray(x, np.float64)).T
    # transposed-conv weight [cin, cout, kd, kh, kw]; slot s = kd*9 + kh*3 + kw
    wt = torch.from_numpy(np.asarray(W, np.float64)).reshape(3, 3, 3, cin, cout).permute(3, 4, 0, 1, 2).contiguous()
    y = torch.nn.functional.conv_transpose3d(dense, wt, stride=stride, padding=1, output_padding=stride - 1)
    # dense output index o is coordinate stride*lo + o
    orel = ijk_out - stride * lo
    return y[0, :, orel[:, 0], orel[:, 1], orel[:, 2]].T.numpy()


def dense_conv_wgrad(ijk_in, x, ijk_out, dy, stride, cin, cout):
    """Gradient with respect to W of sum(conv(x, W)[active outputs] * dy), by
    torch autograd on the dense conv3d (float64) of dense_conv_active."""
    import torch

    ijk_in = np.asarray(ijk_in, dtype=np.int64)
    ijk_out = np.asarray(ijk_out, dtype=np.int64)
    lo = np.minimum(ijk_in.min(0), stride * ijk_out.min(0)) - 2
    lo = lo - np.mod(lo, 2)
    hi = np.maximum(ijk_in.max(0), stride * ijk_out.max(0)) + 3
    size = hi - lo
    dense = torch.zeros((1, cin) + tuple(int(v) for v in size), dtype=torch.float64)
    rel = ijk_in - lo
    dense[0, :, rel[:, 0], rel[:, 1], rel[:, 2]] = torch.from_numpy(np.asarray(x, np.float64)).T
    w = torch.zeros((cout, cin, 3, 3, 3), dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.conv3d(dense, w, stride=stride, padding=1)
    orel = ijk_out - lo // stride
    ya = y[0, :, orel[:, 0], orel[:, 1], orel[:, 2]].T
    (ya * torch.from_numpy(np.asarray(dy, np.float64))).sum().backward()
    # w.grad [cout, cin, kd, kh, kw] -> dW [27, cin, cout]
    return w.grad.permute(2, 3, 4, 1, 0).reshape(27, cin, cout).numpy()

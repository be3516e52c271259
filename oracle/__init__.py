"""Python access to the plain CPU oracle (``oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may use this module; the product library never
does.  The oracle shares no code with the CUDA path.

The C++ source states every convention it follows and cites the pages:
"fVDB: A Deep-Learning Framework for Sparse, Large Scale, and High Performance
Spatial Intelligence" (reading notes: Core method, IndexGrid, GPU-accelerated
IndexGrid build, Sparse-convolution operators) and "DriveRT" (Shared neighbour
maps, Kernels selected per GPU).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with the host C++ compiler (portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I32 = ctypes.c_int32
    sigs = {
        "oracle_leaf_record_bytes": ([], I32),
        "oracle_build": ([P, I64, P, I32], P),
        "oracle_grid_free": ([P], None),
        "oracle_grid_counts": ([P, P], None),
        "oracle_grid_rows": ([P], I64),
        "oracle_grid_voxels": ([P, P, P, P, P], None),
        "oracle_grid_leaves": ([P, P, P, P], None),
        "oracle_grid_lower": ([P, P, P, P, P, P], None),
        "oracle_grid_upper": ([P, P, P, P, P, P], None),
        "oracle_lookup": ([P, P, P, I64, P], None),
        "oracle_coarsen": ([P, I32], P),
        "oracle_kernel_map": ([P, P, I32], P),
        "oracle_kernel_map_transposed": ([P, P, I32], P),
        "oracle_refine": ([P, I32], P),
        "oracle_conv_wgrad": ([P, P, I64, P, I64, P], None),
        "oracle_kmap_free": ([P], None),
        "oracle_kmap_pairs": ([P], I64),
        "oracle_kmap_export": ([P, P, P, P, P], None),
        "oracle_conv": ([P, P, I64, P, I64, P, P], None),
        "oracle_conv_rows": ([P, P, I32, P, I64, P, I64, P, I64, P, P], None),
        "oracle_voxels_along_rays": ([P, P, P, P, I64, ctypes.c_float, ctypes.c_float], P),
        "oracle_rays_hits": ([P], I64),
        "oracle_rays_export": ([P, P, P, P], None),
        "oracle_rays_free": ([P], None),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def leaf_record_bytes() -> int:
    return int(_load().oracle_leaf_record_bytes())


class Grid:
    """IndexGrid built by ``std::map`` in canonical order."""

    def __init__(self, handle, B: int):
        self._h = handle
        self.B = B
        lib = _load()
        c = np.zeros(4, np.int64)
        lib.oracle_grid_counts(self._h, _ptr(c))
        self.n_upper, self.n_lower, self.n_leaf, self.n_active = (int(v) for v in c)
        self.n_rows = int(lib.oracle_grid_rows(self._h))

    @classmethod
    def build(cls, coords: np.ndarray, batch_offsets) -> "Grid":
        coords = np.ascontiguousarray(coords, dtype=np.int32).reshape(-1, 3)
        offs = np.ascontiguousarray(batch_offsets, dtype=np.int64)
        h = _load().oracle_build(_ptr(coords), coords.shape[0], _ptr(offs), len(offs) - 1)
        if not h:
            raise ValueError("oracle_build: malformed batch offsets")
        return cls(h, len(offs) - 1)

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.oracle_grid_free(self._h)
            self._h = None

    def counts(self):
        return dict(n_upper=self.n_upper, n_lower=self.n_lower, n_leaf=self.n_leaf, n_active=self.n_active)

    def voxels(self):
        U = self.n_active
        ijk = np.zeros((U, 3), np.int32)
        batch = np.zeros(U, np.int32)
        r2i = np.zeros(self.n_rows, np.int32)
        vbo = np.zeros(self.B + 1, np.int64)
        _load().oracle_grid_voxels(self._h, _ptr(ijk), _ptr(batch), _ptr(r2i), _ptr(vbo))
        return dict(ijk=ijk, batch=batch, row_to_index=r2i, voxel_batch_offsets=vbo)

    def leaves(self):
        L = self.n_leaf
        origin = np.zeros((L, 3), np.int32)
        batch = np.zeros(L, np.int32)
        rec = np.zeros((L, 10), np.uint64)
        _load().oracle_grid_leaves(self._h, _ptr(origin), _ptr(batch), _ptr(rec))
        return dict(origin=origin, batch=batch, mask=rec[:, :8].copy(), first=rec[:, 8].copy(),
                    prefix9=rec[:, 9].copy())

    def lower(self):
        n = self.n_lower
        origin = np.zeros((n, 3), np.int32)
        batch = np.zeros(n, np.int32)
        mask = np.zeros((n, 64), np.uint64)
        prefix = np.zeros((n, 64), np.uint32)
        first = np.zeros(n, np.uint32)
        _load().oracle_grid_lower(self._h, _ptr(origin), _ptr(batch), _ptr(mask), _ptr(prefix), _ptr(first))
        return dict(origin=origin, batch=batch, mask=mask, prefix=prefix, first=first)

    def upper(self):
        n = self.n_upper
        origin = np.zeros((n, 3), np.int32)
        batch = np.zeros(n, np.int32)
        mask = np.zeros((n, 512), np.uint64)
        prefix = np.zeros((n, 512), np.uint32)
        first = np.zeros(n, np.uint32)
        _load().oracle_grid_upper(self._h, _ptr(origin), _ptr(batch), _ptr(mask), _ptr(prefix), _ptr(first))
        return dict(origin=origin, batch=batch, mask=mask, prefix=prefix, first=first)

    def lookup(self, coords: np.ndarray, batch=None) -> np.ndarray:
        coords = np.ascontiguousarray(coords, dtype=np.int32).reshape(-1, 3)
        n = coords.shape[0]
        b = np.zeros(n, np.int32) if batch is None else np.ascontiguousarray(batch, dtype=np.int32)
        out = np.zeros(n, np.int32)
        _load().oracle_lookup(self._h, _ptr(coords), _ptr(b), n, _ptr(out))
        return out

    def coarsen(self, stride: int = 2) -> "Grid":
        h = _load().oracle_coarsen(self._h, int(stride))
        if not h:
            raise ValueError("oracle_coarsen: bad stride")
        return Grid(h, self.B)

    def refine(self, factor: int = 2) -> "Grid":
        """All factor^3 children of every voxel (the refined grid)."""
        h = _load().oracle_refine(self._h, int(factor))
        if not h:
            raise ValueError("oracle_refine: bad factor")
        return Grid(h, self.B)


class KernelMap:
    """Per-offset (in, out) pair lists of a 3x3x3 kernel, ordered by output."""

    def __init__(self, gin: Grid, gout: Grid, stride: int, transposed: bool = False):
        """transposed: the map of the transposed convolution (output voxel p of
        gout, input voxel q of gin with stride * ijk(q) + d_s = ijk(p))."""
        f = _load().oracle_kernel_map_transposed if transposed else _load().oracle_kernel_map
        self._h = f(gin._h, gout._h, int(stride))
        if not self._h:
            raise ValueError("oracle_kernel_map: bad stride")
        self.transposed = bool(transposed)
        self.stride = int(stride)
        self.n_out = gout.n_active
        P = int(_lib.oracle_kmap_pairs(self._h))
        self.offsets = np.zeros(28, np.int64)
        self.in_idx = np.zeros(P, np.int32)
        self.out_idx = np.zeros(P, np.int32)
        self.mask = np.zeros(self.n_out, np.uint32)
        _lib.oracle_kmap_export(self._h, _ptr(self.offsets), _ptr(self.in_idx), _ptr(self.out_idx), _ptr(self.mask))
        self.n_pairs = P

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.oracle_kmap_free(self._h)
            self._h = None


def conv(kmap: KernelMap, x: np.ndarray, W: np.ndarray):
    """Returns (y, a): fp64 output and the sum of |x*w| per output element."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.float64)
    cin, cout = W.shape[1], W.shape[2]
    assert W.shape[0] == 27 and x.shape[1] == cin
    y = np.zeros((kmap.n_out, cout), np.float64)
    a = np.zeros((kmap.n_out, cout), np.float64)
    _load().oracle_conv(kmap._h, _ptr(x), cin, _ptr(W), cout, _ptr(y), _ptr(a))
    return y, a


def conv_wgrad(kmap: KernelMap, x: np.ndarray, dy: np.ndarray):
    """dW [27, cin, cout] (fp64): per list s, the sum over its pairs (p, q) of
    the outer product x[p] (x) dy[q]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    dy = np.ascontiguousarray(dy, dtype=np.float64)
    cin, cout = x.shape[1], dy.shape[1]
    dW = np.zeros((27, cin, cout), np.float64)
    _load().oracle_conv_wgrad(kmap._h, _ptr(x), cin, _ptr(dy), cout, _ptr(dW))
    return dW


def conv_rows(gin: Grid, gout: Grid, stride: int, rows: np.ndarray, x: np.ndarray, W: np.ndarray):
    """The conv sum for selected output rows only (no kernel map needed)."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    x = np.ascontiguousarray(x, dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.float64)
    cin, cout = W.shape[1], W.shape[2]
    y = np.zeros((rows.shape[0], cout), np.float64)
    a = np.zeros((rows.shape[0], cout), np.float64)
    _load().oracle_conv_rows(gin._h, gout._h, int(stride), _ptr(rows), rows.shape[0], _ptr(x), cin, _ptr(W), cout,
                             _ptr(y), _ptr(a))
    return y, a


def voxels_along_rays(grid: Grid, origins: np.ndarray, dirs: np.ndarray, batch=None, tmin=0.0, tmax=float("inf")):
    """Active voxels each ray passes through, in order ("fVDB" reading notes,
    HDDA; the exact definition is in oracle.cpp).  Returns (offsets int64
    [n+1], voxel index int32 [hits], t float32 [hits, 2] = entry, exit)."""
    lib = _load()
    o = np.ascontiguousarray(origins, np.float32).reshape(-1, 3)
    d = np.ascontiguousarray(dirs, np.float32).reshape(-1, 3)
    n = o.shape[0]
    b = None if batch is None else np.ascontiguousarray(batch, np.int32).reshape(-1)
    h = lib.oracle_voxels_along_rays(grid._h, _ptr(o), _ptr(d), None if b is None else _ptr(b), n,
                                     ctypes.c_float(tmin), ctypes.c_float(tmax))
    if not h:
        raise ValueError("ray batch index out of range")
    try:
        nh = int(lib.oracle_rays_hits(h))
        offs = np.zeros(n + 1, np.int64)
        vox = np.zeros(nh, np.int32)
        t = np.zeros((nh, 2), np.float32)
        lib.oracle_rays_export(h, _ptr(offs), _ptr(vox), _ptr(t))
    finally:
        lib.oracle_rays_free(h)
    return offs, vox, t

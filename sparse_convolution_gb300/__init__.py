"""fvx: sparse-voxel IndexGrid build, 3x3x3 kernel map and sparse convolution
on GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/fvx.h`` (argument
marshalling only; every step runs in the CUDA library ``libfvx.so``).  Torch
tensors supply device memory and the current CUDA stream.  There is no CPU
fallback: if the library is missing or no GPU is visible, calls raise.

Pages: "fVDB: A Deep-Learning Framework for Sparse, Large Scale, and High
Performance Spatial Intelligence" (reading notes: IndexGrid, GPU-accelerated
IndexGrid build, Sparse-convolution operators) and "DriveRT" (Shared neighbour
maps, Kernels selected per GPU).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfvx.so")

_lib = None

FVX_F32, FVX_BF16, FVX_BF16_OUT_BF16 = 0, 1, 2
FVX_CONV_AUTO, FVX_CONV_GATHER, FVX_CONV_LEAF, FVX_CONV_DIRECT, FVX_CONV_UNION, FVX_CONV_HALO = 0, 1, 2, 3, 4, 5


class FvxError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{status}: {message}")
        self.status = status


class GridView(ctypes.Structure):
    _fields_ = [("batch_size", ctypes.c_int32)] + [
        (n, ctypes.c_int64) for n in ("n_rows", "n_upper", "n_lower", "n_leaf", "n_active")
    ] + [(n, ctypes.c_void_p) for n in (
        "ijk", "row_to_index", "voxel_batch_offsets", "leaf_origin", "leaf_batch", "leaf_records",
        "lower_origin", "lower_batch", "lower_mask", "lower_prefix", "lower_first",
        "upper_origin", "upper_batch", "upper_mask", "upper_prefix", "upper_first")]


def load():
    """Loads ``libfvx.so`` (must have been built by ``__graft_entry__.build()``
    or ``build_lib.build()``).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise FvxError("FVX_NOT_BUILT", f"{LIB_PATH} is missing; build the CUDA library first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
    PP = ctypes.POINTER(ctypes.c_void_p)
    sigs = {
        "fvx_set_allocator": ([P, P, P], I32),
        "fvx_build_grid": ([P, I64, P, I32, P, PP], I32),
        "fvx_grid_counts": ([P, P, P, P, P], I32),
        "fvx_grid_view": ([P, ctypes.POINTER(GridView)], I32),
        "fvx_grid_batch_offsets": ([P, P], I32),
        "fvx_lookup": ([P, P, P, I64, P, P], I32),
        "fvx_coarsen": ([P, I32, P, PP], I32),
        "fvx_kernel_map": ([P, P, I32, I32, P, PP], I32),
        "fvx_kernel_map_transposed": ([P, P, I32, I32, P, PP], I32),
        "fvx_refine": ([P, I32, P, PP], I32),
        "fvx_kmap_view": ([P, PP, PP, PP, PP, P, P], I32),
        "fvx_sparse_conv": ([P, P, P, I32, P, I64, P, I64, P, P], I32),
        "fvx_sparse_conv_noalloc": ([P, P, P, I32, P, I64, P, I64, P, P], I32),
        "fvx_noalloc_status": ([P], I32),
        "fvx_testing_bounded_wait": ([I32, U64, P], I32),
        "fvx_sparse_conv_dgrad": ([P, P, P, I32, P, I64, P, I64, P, P], I32),
        "fvx_sparse_conv_wgrad": ([P, P, P, I32, P, I64, P, I64, P, P], I32),
        "fvx_voxels_along_rays": ([P, P, P, P, I64, ctypes.c_float, ctypes.c_float, P, PP], I32),
        "fvx_hits_view": ([P, PP, PP, PP, P, P], I32),
        "fvx_hits_destroy": ([P], I32),
        "fvx_grid_destroy": ([P], I32),
        "fvx_kmap_destroy": ([P], I32),
        "fvx_status_string": ([I32], ctypes.c_char_p),
        "fvx_last_error": ([], ctypes.c_char_p),
        "fvx_device_status": ([P], I32),
        "fvx_launch_count": ([], U64),
        "fvx_profile_enable": ([ctypes.c_char_p], I32),
        "fvx_profile_read": ([P, P], I32),
        "fvx_profile_read_each": ([P, ctypes.c_int64, P], I32),
        "fvx_set_conv_algo": ([I32], I32),
        "fvx_last_conv_algo": ([], I32),
        "fvx_last_conv_kernel": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _check(st):
    if st != 0:
        lib = load()
        raise FvxError(lib.fvx_status_string(st).decode(), lib.fvx_last_error().decode())


def _stream(stream=None):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


class _DevArray:
    """Zero-copy handle on library-owned device memory for torch.as_tensor."""

    def __init__(self, ptr, shape, typestr, owner):
        self.__cuda_array_interface__ = dict(shape=tuple(int(s) for s in shape), typestr=typestr,
                                             data=(int(ptr or 0), False), version=3, strides=None)
        self._owner = owner


_TYPESTR = {"i4": "<i4", "i8": "<i8", "u4": "<u4", "u8": "<u8", "f4": "<f4"}


def _view(ptr, shape, code, owner):
    import torch

    if any(int(s) == 0 for s in shape) or not ptr:
        dt = {"i4": torch.int32, "i8": torch.int64, "u4": torch.uint32, "u8": torch.uint64,
              "f4": torch.float32}[code]
        return torch.zeros(tuple(int(s) for s in shape), dtype=dt, device="cuda")
    t = torch.as_tensor(_DevArray(ptr, shape, _TYPESTR[code], owner), device="cuda")
    return t.clone()


class Grid:
    """A batch of IndexGrids built on the GPU (library-owned topology)."""

    def __init__(self, handle, stream=None):
        self._h = handle
        lib = load()
        c = (ctypes.c_int64 * 4)()
        _check(lib.fvx_grid_counts(self._h, ctypes.byref(c, 0), ctypes.byref(c, 8), ctypes.byref(c, 16),
                                   ctypes.byref(c, 24)))
        self.n_upper, self.n_lower, self.n_leaf, self.n_active = (int(v) for v in c)
        v = GridView()
        _check(lib.fvx_grid_view(self._h, ctypes.byref(v)))
        self.batch_size = int(v.batch_size)
        self.n_rows = int(v.n_rows)
        self._v = v

    @classmethod
    def build(cls, coords, batch_offsets=None, stream=None) -> "Grid":
        """coords: int32 CUDA tensor [N, 3]; batch_offsets: CSR int64 [B+1]
        (host sequence / numpy / CPU tensor), default one batch."""
        import torch

        assert coords.is_cuda and coords.dtype == torch.int32 and coords.dim() == 2 and coords.shape[1] == 3
        coords = coords.contiguous()
        n = coords.shape[0]
        if batch_offsets is None:
            batch_offsets = [0, n]
        offs = np.ascontiguousarray(np.asarray(batch_offsets, dtype=np.int64))
        h = ctypes.c_void_p()
        _check(load().fvx_build_grid(_ptr(coords), n, offs.ctypes.data_as(ctypes.c_void_p), len(offs) - 1,
                                     _stream(stream), ctypes.byref(h)))
        return cls(h)

    def destroy(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.fvx_grid_destroy(self._h)
            self._h = None

    __del__ = destroy

    def counts(self):
        return dict(n_upper=self.n_upper, n_lower=self.n_lower, n_leaf=self.n_leaf, n_active=self.n_active)

    def batch_offsets(self):
        out = np.zeros(self.batch_size + 1, np.int64)
        _check(load().fvx_grid_batch_offsets(self._h, out.ctypes.data_as(ctypes.c_void_p)))
        return out

    def topology(self):
        """Copies of every topology array as CUDA tensors."""
        v = self._v
        U, L, NL, NU = self.n_active, self.n_leaf, self.n_lower, self.n_upper
        return dict(
            ijk=_view(v.ijk, (U, 3), "i4", self), row_to_index=_view(v.row_to_index, (self.n_rows,), "i4", self),
            voxel_batch_offsets=_view(v.voxel_batch_offsets, (self.batch_size + 1,), "i8", self),
            leaf_origin=_view(v.leaf_origin, (L, 3), "i4", self), leaf_batch=_view(v.leaf_batch, (L,), "i4", self),
            leaf_records=_view(v.leaf_records, (L, 10), "u8", self),
            lower_origin=_view(v.lower_origin, (NL, 3), "i4", self),
            lower_batch=_view(v.lower_batch, (NL,), "i4", self), lower_mask=_view(v.lower_mask, (NL, 64), "u8", self),
            lower_prefix=_view(v.lower_prefix, (NL, 64), "u4", self),
            lower_first=_view(v.lower_first, (NL,), "u4", self),
            upper_origin=_view(v.upper_origin, (NU, 3), "i4", self),
            upper_batch=_view(v.upper_batch, (NU,), "i4", self),
            upper_mask=_view(v.upper_mask, (NU, 512), "u8", self),
            upper_prefix=_view(v.upper_prefix, (NU, 512), "u4", self),
            upper_first=_view(v.upper_first, (NU,), "u4", self))

    def ijk(self):
        return _view(self._v.ijk, (self.n_active, 3), "i4", self)

    def lookup(self, coords, batch=None, stream=None):
        import torch

        coords = coords.contiguous()
        out = torch.empty(coords.shape[0], dtype=torch.int32, device=coords.device)
        b = batch.contiguous() if batch is not None else None
        _check(load().fvx_lookup(self._h, _ptr(coords), _ptr(b), coords.shape[0], _ptr(out), _stream(stream)))
        return out

    def coarsen(self, stride=2, stream=None) -> "Grid":
        h = ctypes.c_void_p()
        _check(load().fvx_coarsen(self._h, int(stride), _stream(stream), ctypes.byref(h)))
        return Grid(h)

    def refine(self, factor=2, stream=None) -> "Grid":
        """Every voxel's factor^3 children (the refined grid)."""
        h = ctypes.c_void_p()
        _check(load().fvx_refine(self._h, int(factor), _stream(stream), ctypes.byref(h)))
        return Grid(h)


class KernelMap:
    """Per-offset (in, out) pair lists of a 3x3x3 kernel (library-owned)."""

    def __init__(self, gin: Grid, gout: Grid, stride=1, ksize=3, stream=None, transposed=False):
        """transposed: the map of the transposed convolution (output voxel q
        paired with the input p where stride * ijk(p) + d == ijk(q))."""
        h = ctypes.c_void_p()
        f = load().fvx_kernel_map_transposed if transposed else load().fvx_kernel_map
        _check(f(gin._h, gout._h, int(ksize), int(stride), _stream(stream), ctypes.byref(h)))
        self._h = h
        self.gin, self.gout, self.stride, self.transposed = gin, gout, int(stride), bool(transposed)
        ii, oo, mm = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        nout = ctypes.c_int64()
        _check(_lib.fvx_kmap_view(h, None, ctypes.byref(ii), ctypes.byref(oo), ctypes.byref(mm), None,
                                  ctypes.byref(nout)))
        self.n_out = int(nout.value)
        self._ptrs = (ii.value, oo.value, mm.value)
        self._totals = None

    def _read_totals(self):
        # the list offsets stay on the device until first asked for (that read
        # synchronises the map's stream)
        if self._totals is None:
            offs, npairs = ctypes.c_void_p(), ctypes.c_int64()
            _check(_lib.fvx_kmap_view(self._h, ctypes.byref(offs), None, None, None, ctypes.byref(npairs), None))
            self._totals = (np.ctypeslib.as_array((ctypes.c_int64 * 28).from_address(offs.value)).copy(),
                            int(npairs.value))
        return self._totals

    @property
    def offsets(self):
        """HOST int64 [28]: list s is pairs [offsets[s], offsets[s+1])."""
        return self._read_totals()[0]

    @property
    def n_pairs(self):
        return self._read_totals()[1]

    def destroy(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.fvx_kmap_destroy(self._h)
            self._h = None

    __del__ = destroy

    def pairs(self):
        ii, oo, mm = self._ptrs
        return (_view(ii, (self.n_pairs,), "i4", self), _view(oo, (self.n_pairs,), "i4", self),
                _view(mm, (self.n_out,), "u4", self))


class Hits:
    """Active voxels along rays (library-owned CSR result of
    fvx_voxels_along_rays)."""

    def __init__(self, grid: Grid, origins, dirs, batch=None, tmin=0.0, tmax=float("inf"), stream=None):
        import torch

        assert origins.dtype == torch.float32 and dirs.dtype == torch.float32 and origins.is_cuda and dirs.is_cuda
        origins = origins.contiguous()
        dirs = dirs.contiguous()
        n = origins.shape[0]
        assert tuple(origins.shape) == (n, 3) and tuple(dirs.shape) == (n, 3)
        if batch is not None:
            batch = batch.to(torch.int32).contiguous()
        h = ctypes.c_void_p()
        _check(load().fvx_voxels_along_rays(grid._h, _ptr(origins), _ptr(dirs), _ptr(batch), n,
                                            ctypes.c_float(tmin), ctypes.c_float(tmax), _stream(stream),
                                            ctypes.byref(h)))
        self._h = h
        off, vox, t = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        nh, nr = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.fvx_hits_view(h, ctypes.byref(off), ctypes.byref(vox), ctypes.byref(t), ctypes.byref(nh),
                                  ctypes.byref(nr)))
        self.n_hits, self.n_rays = int(nh.value), int(nr.value)
        self._ptrs = (off.value, vox.value, t.value)

    def arrays(self):
        """(offsets int64 [n_rays + 1], voxel int32 [n_hits], t float32 [n_hits, 2]), device copies."""
        off, vox, t = self._ptrs
        return (_view(off, (self.n_rays + 1,), "i8", self), _view(vox, (self.n_hits,), "i4", self),
                _view(t, (self.n_hits, 2), "f4", self))

    def destroy(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.fvx_hits_destroy(self._h)
            self._h = None

    __del__ = destroy


def sparse_conv(gin: Grid, gout: Grid, kmap: KernelMap, feats, W, out=None, out_dtype=None, stream=None):
    """out[q] = sum over pairs (p, q) of list s of feats[p] @ W[s].

    feats [gin.n_active, cin] and W [27, cin, cout]: both float32 (exact fp32
    FFMA, float32 out) or both bfloat16 (tensor cores, fp32 accumulation;
    out_dtype float32 by default, or bfloat16 for a rounded bf16 output)."""
    import torch

    assert feats.dtype == W.dtype and feats.is_cuda and W.is_cuda
    if feats.dtype == torch.float32:
        dt, odt = FVX_F32, torch.float32
    else:
        assert feats.dtype == torch.bfloat16
        odt = out_dtype or (out.dtype if out is not None else torch.float32)
        dt = {torch.float32: FVX_BF16, torch.bfloat16: FVX_BF16_OUT_BF16}[odt]
    feats = feats.contiguous()
    W = W.contiguous()
    cin, cout = W.shape[1], W.shape[2]
    assert W.shape[0] == 27 and feats.shape[1] == cin
    if out is None:
        out = torch.empty((gout.n_active, cout), dtype=odt, device=feats.device)
    assert out.dtype == odt and out.is_contiguous() and tuple(out.shape) == (gout.n_active, cout)
    _check(load().fvx_sparse_conv(gin._h, gout._h, kmap._h, dt, _ptr(feats), cin, _ptr(W), cout, _ptr(out),
                                  _stream(stream)))
    return out


def sparse_conv_dgrad(gin: Grid, gout: Grid, kmap_t: KernelMap, dout, W, out=None, out_dtype=None, stream=None):
    """Input gradient of sparse_conv(gin, gout, ...): dx [gin.n_active, cin].

    kmap_t: KernelMap(gout, gin, stride, transposed=True).  dout [gout.n_active,
    cout] and W [27, cin, cout] both float32 or both bfloat16 (float32 dx by
    default, bfloat16 with out_dtype=torch.bfloat16)."""
    import torch

    assert dout.dtype == W.dtype and dout.is_cuda and W.is_cuda
    if dout.dtype == torch.float32:
        dt, odt = FVX_F32, torch.float32
    else:
        assert dout.dtype == torch.bfloat16
        odt = out_dtype or (out.dtype if out is not None else torch.float32)
        dt = {torch.float32: FVX_BF16, torch.bfloat16: FVX_BF16_OUT_BF16}[odt]
    dout = dout.contiguous()
    W = W.contiguous()
    cin, cout = W.shape[1], W.shape[2]
    assert W.shape[0] == 27 and dout.shape[1] == cout
    if out is None:
        out = torch.empty((gin.n_active, cin), dtype=odt, device=dout.device)
    assert out.dtype == odt and out.is_contiguous() and tuple(out.shape) == (gin.n_active, cin)
    _check(load().fvx_sparse_conv_dgrad(gin._h, gout._h, kmap_t._h, dt, _ptr(dout), cout, _ptr(W), cin, _ptr(out),
                                        _stream(stream)))
    return out


def sparse_conv_wgrad(gin: Grid, gout: Grid, kmap: KernelMap, feats, dout, out=None, stream=None):
    """Weight gradient of sparse_conv(gin, gout, kmap, feats, W): float32
    [27, cin, cout].  feats and dout both float32 or both bfloat16."""
    import torch

    assert feats.dtype == dout.dtype and feats.is_cuda and dout.is_cuda
    dt = FVX_F32 if feats.dtype == torch.float32 else FVX_BF16
    assert dt == FVX_F32 or feats.dtype == torch.bfloat16
    feats = feats.contiguous()
    dout = dout.contiguous()
    cin, cout = feats.shape[1], dout.shape[1]
    if out is None:
        out = torch.empty((27, cin, cout), dtype=torch.float32, device=feats.device)
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (27, cin, cout)
    _check(load().fvx_sparse_conv_wgrad(gin._h, gout._h, kmap._h, dt, _ptr(feats), cin, _ptr(dout), cout, _ptr(out),
                                        _stream(stream)))
    return out


def device_status(stream=None):
    _check(load().fvx_device_status(_stream(stream)))


def noalloc_status(stream=None):
    """Status of the last fvx_sparse_conv_noalloc call (raises FvxError on a
    recorded timeout or check failure)."""
    _check(load().fvx_noalloc_status(_stream(stream)))


def set_conv_algo(algo: int) -> None:
    """FVX_CONV_AUTO (default), FVX_CONV_GATHER, FVX_CONV_DIRECT,
    FVX_CONV_UNION, FVX_CONV_HALO or FVX_CONV_LEAF: which bf16 convolution
    kernel sparse_conv runs (process-wide)."""
    _check(load().fvx_set_conv_algo(int(algo)))


def last_conv_algo() -> int:
    """FVX_CONV_GATHER, FVX_CONV_LEAF or FVX_CONV_HALO: what the last bf16
    convolution on this thread ran (FVX_CONV_AUTO before any)."""
    return int(load().fvx_last_conv_algo())


def last_conv_kernel() -> str:
    """Name of the kernel the last convolution on this thread launched."""
    return load().fvx_last_conv_kernel().decode()


def launch_count() -> int:
    return int(load().fvx_launch_count())


def profile_enable(kernel_name):
    _check(load().fvx_profile_enable(kernel_name.encode() if kernel_name else None))


def profile_read():
    ms, n = ctypes.c_double(), ctypes.c_int64()
    _check(load().fvx_profile_read(ctypes.byref(ms), ctypes.byref(n)))
    return float(ms.value), int(n.value)


def profile_read_each(cap=4096):
    """Durations (ms) of the timed launches, in launch order."""
    buf = (ctypes.c_double * cap)()
    n = ctypes.c_int64()
    _check(load().fvx_profile_read_each(buf, cap, ctypes.byref(n)))
    return [float(buf[i]) for i in range(min(cap, n.value))]

"""Failure reporting on the GPU, in forms that fault, trap or hang nothing.

* A bounded device-side wait that runs out ("DriveRT", Inspection and
  debugging: a failure is reported, naming what failed): a test hook runs one
  wait of each form the kernels use (mbarrier phase wait, look-back flag poll)
  on something nothing completes, with a short limit.  The status word
  reports FVX_ERR_DEVICE_TIMEOUT once, is cleared, and the library keeps
  working.
* A device allocation that fails: an allocator that returns NULL on its k-th
  call, for every k over the allocations of build, kernel map and conv.  Each
  call returns FVX_ERR_ALLOC with a message naming the entry point, frees what
  it had taken (nothing leaks), and the same calls succeed afterwards.
"""
import ctypes

import numpy as np
import pytest

import oracle
from tests import gpu_common as G

pytestmark = pytest.mark.gpu

ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p)
FREE_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)


def _small_grid(seed=3):
    rng = np.random.default_rng(seed)
    c = rng.integers(-25, 25, size=(9000, 3)).astype(np.int32)
    c = np.concatenate([c, c[:900]])
    return c, np.array([0, 5000, len(c)], np.int64)


def _pipeline_ok(coords, offs):
    """Build, kernel map and bf16 conv through the library, checked against
    the oracle."""
    import sparse_convolution_gb300 as fvx

    g = G.gpu_grid(coords, offs)
    og = oracle.Grid.build(coords, offs)
    assert g.counts() == og.counts()
    km = fvx.KernelMap(g, g, 1)
    okm = oracle.KernelMap(og, og, 1)
    G.assert_kmap_equal(km, okm)
    x, W = G.bf16_inputs(11, g.n_active, 16, 32)
    y = fvx.sparse_conv(g, g, km, x, W)
    fvx.device_status()
    yo, ao = oracle.conv(okm, G.as_f64(x), G.as_f64(W))
    G.assert_conv_close(G.np_(y.float()), yo, ao, G.BF16_TOL)
    km.destroy()
    g.destroy()


@pytest.mark.parametrize("kind", [0, 1])
def test_bounded_wait_runs_out_and_is_reported(cuda_device, kind):
    import torch

    import sparse_convolution_gb300 as fvx

    lib = fvx.load()
    fvx.device_status()  # start from a clear status word
    limit_ns = 3_000_000
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    assert lib.fvx_testing_bounded_wait(kind, limit_ns, ctypes.c_void_p(stream.cuda_stream)) == 0, \
        lib.fvx_last_error()
    e1.record(stream)
    with pytest.raises(fvx.FvxError) as ei:
        fvx.device_status()
    assert ei.value.status == "FVX_ERR_DEVICE_TIMEOUT"
    assert "gave up" in str(ei.value)
    # the wait lasted at least its limit and ended on its own
    ms = e0.elapsed_time(e1)
    assert limit_ns / 1e6 <= ms < 2000.0, ms
    fvx.device_status()  # read once: cleared
    _pipeline_ok(*_small_grid())  # the context is still usable


class CountingAllocator:
    """fvx_set_allocator callbacks over torch's caching allocator that fail
    (return NULL) on call number fail_at and record what is outstanding."""

    def __init__(self, fail_at=None):
        import torch

        self.torch = torch
        self.fail_at = fail_at
        self.calls = 0
        self.live = {}
        self.failed = False
        self.alloc = ALLOC_FN(self._alloc)
        self.free = FREE_FN(self._free)

    def _alloc(self, nbytes, stream, ctx):
        self.calls += 1
        if self.fail_at is not None and self.calls == self.fail_at:
            self.failed = True
            return None
        dev = self.torch.cuda.current_device()
        p = self.torch.cuda.caching_allocator_alloc(int(nbytes), dev, stream or 0)
        self.live[p] = int(nbytes)
        return p

    def _free(self, ptr, stream, ctx):
        assert ptr in self.live, "free of a pointer this allocator did not hand out"
        del self.live[ptr]
        self.torch.cuda.caching_allocator_delete(ptr)

    def __enter__(self):
        import sparse_convolution_gb300 as fvx

        lib = fvx.load()
        assert lib.fvx_set_allocator(ctypes.cast(self.alloc, ctypes.c_void_p),
                                     ctypes.cast(self.free, ctypes.c_void_p), None) == 0
        return self

    def __exit__(self, *a):
        import sparse_convolution_gb300 as fvx

        self.torch.cuda.synchronize()
        fvx.load().fvx_set_allocator(None, None, None)
        return False


def _attempt(coords, offs):
    """Build -> kernel map -> conv; returns (entry point that failed or None,
    its status name, message).  Handles it created are destroyed."""
    import torch

    import sparse_convolution_gb300 as fvx

    handles = []
    try:
        g = fvx.Grid.build(torch.from_numpy(coords).cuda(), offs)
        handles.append(g)
        km = fvx.KernelMap(g, g, 1)
        handles.append(km)
        x, W = G.bf16_inputs(11, g.n_active, 16, 32)
        fvx.sparse_conv(g, g, km, x, W)
        fvx.device_status()
        return None, None, None
    except fvx.FvxError as e:
        return e, e.status, str(e)
    finally:
        for h in reversed(handles):
            h.destroy()
        torch.cuda.synchronize()


def test_allocation_failure_at_every_allocation(cuda_device):
    import sparse_convolution_gb300 as fvx

    coords, offs = _small_grid(5)
    with CountingAllocator() as probe:  # how many allocations one pass makes
        err, _, _ = _attempt(coords, offs)
        assert err is None
    n_alloc = probe.calls
    assert n_alloc >= 3 and not probe.live, (n_alloc, probe.live)
    for k in range(1, n_alloc + 1):
        with CountingAllocator(fail_at=k) as ca:
            err, name, msg = _attempt(coords, offs)
            assert ca.failed
            assert err is not None and name == "FVX_ERR_ALLOC", (k, name, msg)
            assert "device allocation" in msg and any(
                ep in msg for ep in ("fvx_build_grid", "fvx_kernel_map", "fvx_sparse_conv")), msg
        assert not ca.live, f"allocation {k} failing leaked {len(ca.live)} buffers"
        fvx.device_status()
    _pipeline_ok(coords, offs)  # default allocator again, same results

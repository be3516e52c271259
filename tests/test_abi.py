"""The C-ABI library builds for sm_103a, loads, exports every entry point that
include/fvx.h declares, and validates arguments on the host (no GPU needed:
every call below returns before any CUDA work)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_convolution_gb300 import build_lib

    build_lib.build()
    import sparse_convolution_gb300 as fvx

    return fvx.load()


def _declared(header="fvx.h"):
    txt = open(os.path.join(ROOT, "include", header)).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(fvx_[a-z_0-9]+)\s*\(", txt)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("fvx_build_grid", "fvx_kernel_map", "fvx_sparse_conv", "fvx_lookup", "fvx_coarsen",
              "fvx_grid_view", "fvx_kmap_view", "fvx_grid_destroy", "fvx_kmap_destroy", "fvx_set_allocator",
              "fvx_status_string", "fvx_last_error", "fvx_refine", "fvx_kernel_map_transposed",
              "fvx_sparse_conv_dgrad", "fvx_sparse_conv_wgrad", "fvx_sparse_conv_noalloc", "fvx_noalloc_status",
              "fvx_set_conv_algo", "fvx_last_conv_algo", "fvx_device_status", "fvx_grid_counts",
              "fvx_grid_batch_offsets", "fvx_launch_count", "fvx_profile_enable", "fvx_profile_read",
              "fvx_profile_read_each"):
        assert n in names, n
    assert _declared("fvx_testing.h") == ["fvx_testing_bounded_wait"]


def test_header_is_plain_c(tmp_path):
    """The boundary compiles as ISO C (no C++ or CUDA types), with and without
    extern "C" handling."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    src.write_text('#include "fvx.h"\n#include "fvx_testing.h"\n'
                   'int main(void) { fvx_grid g = 0; (void)g; return (int)FVX_OK; }\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        "-fsyntax-only", str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() + _declared("fvx_testing.h") if not hasattr(lib, n)]
    assert not missing, missing


def test_testing_hook_validates_on_host(lib):
    """The bounded-wait test hook refuses a kind or limit outside its range
    before any device work."""
    assert lib.fvx_testing_bounded_wait(2, 10_000, None) == 1
    assert lib.fvx_testing_bounded_wait(0, 10, None) == 1
    assert lib.fvx_testing_bounded_wait(1, 3_000_000_000, None) == 1
    assert b"fvx_testing_bounded_wait" in lib.fvx_last_error()


def test_status_strings(lib):
    assert lib.fvx_status_string(0) == b"FVX_OK"
    assert lib.fvx_status_string(2) == b"FVX_ERR_RANGE"
    assert lib.fvx_status_string(6) == b"FVX_ERR_DEVICE_TIMEOUT"


def _build(lib, coords_ptr, n, offs, B):
    out = ctypes.c_void_p()
    o = np.asarray(offs, np.int64)
    st = lib.fvx_build_grid(coords_ptr, n, o.ctypes.data_as(ctypes.c_void_p), B, None, ctypes.byref(out))
    return st, lib.fvx_last_error().decode()


def test_build_validates_on_host(lib):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    st, msg = _build(lib, fake, 10, [0, 10], 0)
    assert st == 1 and "B >= 1" in msg
    st, msg = _build(lib, fake, 10, [0, 4, 3, 10], 3)
    assert st == 1 and "monotone" in msg
    st, msg = _build(lib, fake, 10, [0, 9], 1)
    assert st == 1 and "end at n_rows" in msg
    st, msg = _build(lib, fake, -1, [0, -1], 1)
    assert st == 1
    st, msg = _build(lib, None, 10, [0, 10], 1)
    assert st == 1 and "NULL" in msg


def test_kmap_and_conv_validate_on_host(lib):
    out = ctypes.c_void_p()
    assert lib.fvx_kernel_map(None, None, 3, 1, None, ctypes.byref(out)) == 1
    assert lib.fvx_sparse_conv(None, None, None, 1, None, 8, None, 16, None, None) == 1
    assert lib.fvx_coarsen(None, 2, None, ctypes.byref(out)) == 1
    assert lib.fvx_set_allocator(ctypes.c_void_p(1), None, None) == 1
    assert lib.fvx_set_allocator(None, None, None) == 0


def test_launch_counter_and_profiler_idle(lib):
    import sparse_convolution_gb300 as fvx

    n0 = fvx.launch_count()
    fvx.profile_enable("conv_bf16_tc")
    assert fvx.profile_read() == (0.0, 0)
    fvx.profile_enable(None)
    assert fvx.launch_count() == n0


def test_package_fails_loudly_without_library(tmp_path, monkeypatch):
    import sparse_convolution_gb300 as fvx

    monkeypatch.setattr(fvx, "_lib", None)
    monkeypatch.setattr(fvx, "LIB_PATH", str(tmp_path / "libfvx.so"))
    with pytest.raises(fvx.FvxError, match="missing"):
        fvx.load()


def test_backward_entry_points_validate_on_host(lib):
    """The transposed map, refined grid and gradient entry points reject NULL
    handles and bad arguments before any device work."""
    out = ctypes.c_void_p()
    assert lib.fvx_kernel_map_transposed(None, None, 3, 2, None, ctypes.byref(out)) == 1
    assert lib.fvx_refine(None, 2, None, ctypes.byref(out)) == 1
    assert lib.fvx_sparse_conv_dgrad(None, None, None, 1, None, 16, None, 8, None, None) == 1
    assert lib.fvx_sparse_conv_wgrad(None, None, None, 1, None, 8, None, 16, None, None) == 1
    assert b"NULL" in lib.fvx_last_error() or b"bad argument" in lib.fvx_last_error()


def test_reference_arm_line_on_cpu():
    """bench.py --impl reference: the oracle's line on the host (tiny
    workload), with the keys the driver reads."""
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    class A:
        warmup = 0
        steps = 1
        workload = "tiny_shell"
        scale = 1.0

    out = bench.bench_reference(A, 1, 0)
    assert out["impl"] == "reference" and out["value"] > 0 and out["unit"] == bench.UNIT
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["cores"] == 1
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["value"] == out["value"]


def test_c_program_links_and_calls_the_library(lib, tmp_path):
    """A plain C program links libfvx.so and gets status codes and messages
    from it (host paths only)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    pkg = os.path.join(ROOT, "sparse_convolution_gb300")
    src = tmp_path / "use.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "fvx.h"
int main(void) {
  fvx_grid g = 0;
  if (fvx_refine(NULL, 2, NULL, &g) != FVX_ERR_INVALID_ARG) return 1;
  if (strstr(fvx_last_error(), "fvx_refine") == NULL) return 2;
  if (strcmp(fvx_status_string(FVX_ERR_RANGE), "FVX_ERR_RANGE") != 0) return 3;
  puts("ok");
  return 0;
}
""")
    exe = tmp_path / "use"
    r = subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-L", pkg, "-lfvx",
                        "-Wl,-rpath," + pkg, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)


def test_bench_roofline_arithmetic(tmp_path, monkeypatch):
    """The bench line's roofline: tensor above the measured ridge, HBM below,
    FFMA for fp32; achieved = algorithmic flops or bytes over the time; and
    a kernel's DRAM traffic read from an ncu summary only while the source
    hash the summary records matches the kernel's file."""
    import hashlib
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    peaks = {"hbm_gbs": 6785.2, "bf16_tflops": 1917.5, "sm_max_mhz": 2070.0}
    ridge = 1917.5e12 / 6785.2e9  # flop per byte
    r = bench.conv_roofline(flops=1e12, alg_bytes=1e12 / (2 * ridge), sec=1e-3, fp32=False, peaks=peaks,
                            peak_kind="measured", sm_count=152)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["achieved"] == 1000.0
    assert r["frac"] == round(1000.0 / 1917.5, 4)
    r = bench.conv_roofline(flops=1e12, alg_bytes=2e12 / ridge, sec=1e-3, fp32=False, peaks=peaks,
                            peak_kind="measured", sm_count=152)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 2e12 / ridge / 1e-3 / 1e9) < 0.1
    r = bench.conv_roofline(flops=8.05e13, alg_bytes=1e9, sec=1.0, fp32=True, peaks=peaks, peak_kind="measured",
                            sm_count=152)
    assert r["bound"] == "alu" and abs(r["peak"] - 152 * 128 * 2 * 2070e6 / 1e12) < 0.1
    # a summary in the committed format, over a stand-in source tree
    src = tmp_path / "sparse_convolution_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "conv.cu").write_text("// kernel source\n")
    sha = hashlib.sha256((src / "conv.cu").read_bytes()).hexdigest()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "conv_halo_w.md").write_text(
        f"source_sha256: {sha} (sparse_convolution_gb300/csrc/conv.cu)\n"
        "| dram__bytes_read.sum | 100.0 | MB |\n"
        "full launch: dram__bytes_read.sum 801.1 MB, dram__bytes_write.sum 2907.5 MB\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("conv_halo", "w") == int((801.1 + 2907.5) * 1e6)
    assert bench.profiled_traffic("conv_halo", "other") is None
    (src / "conv.cu").write_text("// kernel source, changed\n")
    assert bench.profiled_traffic("conv_halo", "w") is None

"""Compiles the fvx CUDA library (``libfvx.so``) in-tree for sm_103a.

Translation units are compiled in parallel with nvcc and linked into one
shared library next to this file.  Rebuilds only when a source or header is
newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libfvx.so")
BUILD_DIR = os.path.join(ROOT, "_build")

SOURCES = ["api.cu", "primitives.cu", "build.cu", "kmap.cu", "conv.cu", "rays.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the fvx CUDA library cannot be built")
    return cand


def _deps():
    return glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(ROOT, "include", "*.h")) + [__file__]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and not needs_build():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")] + list(extra_flags)
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0 or (verbose and out):
            (errors if p.returncode != 0 else [None]).append((src, out.decode(errors="replace")))
            if p.returncode == 0:
                print(out.decode(errors="replace"), file=sys.stderr)
    if errors:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in errors if s)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else ()))

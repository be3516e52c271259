"""Benchmark of the sparse-voxel hot path on GB300: IndexGrid build from
unsorted int32 coordinates -> 3x3x3 kernel map -> bf16 sparse convolution.

One step = one pass of the whole path over the workload: fvx_build_grid,
fvx_kernel_map (submanifold, stride 1), fvx_sparse_conv.  The default workload
is the leaf-dense grid (union of 40 solid ellipsoids with radii 8-40 in a 256^3
box, bf16 8 -> 16).

Prints ONE JSON line (rank 0).  `value` is whole-step throughput in active
voxels per second (Mvoxels/s) with inputs resident in HBM; `components` splits
it into the two quantities the metric names (build+kmap Mvoxels/s and conv
active-pair TFLOP/s).  `--impl reference` times the CPU oracle on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse conv3d active-pair TFLOP/s (bf16); IndexGrid build+kmap Mvoxels/s"
UNIT = "Mvoxels/s"
L2_FLUSH_BYTES = 256 << 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="fvx", choices=["fvx", "reference"])
    p.add_argument("--workload", default="leaf_dense")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-kernel", default=None, help="kernel whose launches are timed for the roofline")
    return p.parse_args()


# ---------------------------------------------------------------- distributed plumbing
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "fvx" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(smax) if smax else None,
                    reasons=sorted(reasons), samples=len(sm))


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch (read + write) of `kernel` from the committed ncu
    summary under profiles/, if that capture was taken on the current source of
    the kernel (sha256 of its .cu file recorded in the summary); else None."""
    import hashlib
    import re

    src = {"conv_bf16_tc": "conv.cu", "kmap1_write": "kmap.cu"}.get(kernel)
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if src is None or not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_rd = re.search(r"dram__bytes_read\.sum[^0-9]*([0-9.]+)\s*MB", text)
    m_wr = re.search(r"dram__bytes_write\.sum[^0-9]*([0-9.]+)\s*MB", text)
    if not (m_sha and m_rd and m_wr):
        return None
    cur = hashlib.sha256(open(os.path.join(ROOT, "sparse_convolution_gb300", "csrc", src), "rb").read()).hexdigest()
    if cur != m_sha.group(1):
        return None
    return int((float(m_rd.group(1)) + float(m_wr.group(1))) * 1e6)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0), "fallback"


# ---------------------------------------------------------------- workload
def make_workload(name):
    from sparse_convolution_gb300 import synth

    w = synth.WORKLOADS[name]()
    return w


def oracle_sample(w, target_rows=250_000):
    """A spatially contiguous crop of the workload (first batch, lowest i)
    with about target_rows rows: same density and structure, bounded CPU work."""
    coords, offs = w["coords"], w["batch_offsets"]
    c = coords[offs[0]:offs[1]]
    if c.shape[0] <= target_rows:
        return c, np.array([0, c.shape[0]], np.int64), "whole first batch element"
    cut = np.partition(c[:, 0], target_rows)[target_rows]
    sel = c[c[:, 0] < cut]
    return sel, np.array([0, sel.shape[0]], np.int64), f"crop i < {int(cut)} of batch 0 ({sel.shape[0]} rows)"


def run_oracle_step(coords, offs, cv, seed):
    import oracle
    from sparse_convolution_gb300 import synth

    g = oracle.Grid.build(coords, offs)
    km = oracle.KernelMap(g, g, 1)
    x = synth.features(seed, g.n_active, cv["cin"])
    W = synth.weights(seed + 1, cv["cin"], cv["cout"])
    oracle.conv(km, x.astype(np.float64), W.astype(np.float64))
    return g.n_active


def cpu_baseline(w, budget_s=20.0):
    coords, offs, desc = oracle_sample(w)
    cv = w["convs"][0]
    t0 = time.perf_counter()
    n = run_oracle_step(coords, offs, cv, 1)
    dt = time.perf_counter() - t0
    return dict(value=n / dt / 1e6, unit=UNIT, cores=1, kind="oracle",
                sample=f"{desc}: build+kmap+conv of {n} voxels, single-threaded, {dt:.1f} s",
                host_cores=os.cpu_count())


# ---------------------------------------------------------------- GPU arm
def bench_fvx(args, world, rank, local):
    import torch

    from sparse_convolution_gb300 import build_lib
    import sparse_convolution_gb300 as fvx

    torch.cuda.set_device(local)
    build_lib.build()
    fvx.load()
    w = make_workload(args.workload)
    cv = w["convs"][0]
    assert cv["stride"] == 1 and w["dtype"] == "bf16"
    coords_h = torch.from_numpy(w["coords"]).pin_memory()
    offs = w["batch_offsets"]
    U = int(np.sum(w["n_unique"])) if w["n_unique"] is not None else None
    from sparse_convolution_gb300 import synth

    dev = torch.device("cuda", local)
    coords = coords_h.to(dev)
    # feature rows follow the active-voxel index order; values are i.i.d. so any order is a valid input
    g0 = fvx.Grid.build(coords, offs)
    U = g0.n_active
    g0.destroy()
    x_h = torch.from_numpy(synth.features(w["seed"] + 10, U, cv["cin"])).bfloat16().pin_memory()
    W_h = torch.from_numpy(synth.weights(w["seed"] + 20, cv["cin"], cv["cout"])).bfloat16().pin_memory()
    x = x_h.to(dev)
    W = W_h.to(dev)
    # bf16 operands, fp32 accumulation and fp32 output (the mode whose error
    # meets 2e-3 * sum|w*x|; a bf16 output would add a 2^-8 |y| rounding)
    y = torch.empty((U, cv["cout"]), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        g = fvx.Grid.build(coords, offs)
        if ev:
            ev[1].record(stream)
        km = fvx.KernelMap(g, g, 1)
        if ev:
            ev[2].record(stream)
        fvx.sparse_conv(g, g, km, x, W, out=y)
        if ev:
            ev[3].record(stream)
        return g, km

    for _ in range(args.warmup):
        g, km = step()
        npairs = km.n_pairs
        km.destroy()
        g.destroy()
    torch.cuda.synchronize()
    fvx.device_status()

    prof_kernel = args.profile_kernel or "conv_bf16_tc"
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    fvx.profile_enable(prof_kernel)
    l0 = fvx.launch_count()
    for k in range(args.steps):
        flush.fill_(float(k))  # evict L2 between steps (outside the step's events)
        g, km = step(evs[k])
        km.destroy()
        g.destroy()
    torch.cuda.synchronize()
    launches = fvx.launch_count() - l0
    prof_ms, prof_n = fvx.profile_read()
    fvx.profile_enable(None)
    barrier(world)
    clk = clocks.stop()
    fvx.device_status()
    t_build = sum(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    t_kmap = sum(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    t_conv = sum(e[2].elapsed_time(e[3]) for e in evs) / 1e3
    t_total = max_over_ranks(t_build + t_kmap + t_conv, world)
    K = args.steps
    value = U * K * world / t_total / 1e6
    flops = 2.0 * cv["cin"] * cv["cout"] * npairs

    # roofline of the profiled kernel
    peaks, peak_kind = measured_peaks()
    if prof_kernel == "conv_bf16_tc":
        # feats read once, fp32 output written once, weights once, and the
        # kernel map's (in, out) int32 pair read once
        alg_bytes = U * cv["cin"] * 2 + U * cv["cout"] * 4 + 27 * cv["cin"] * cv["cout"] * 2 + 8 * npairs
    else:
        alg_bytes = None
    avg_ms = prof_ms / max(prof_n, 1)
    roofline = None
    if alg_bytes is not None and prof_n:
        ach = alg_bytes / (avg_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roofline = dict(bound="hbm", kernel=prof_kernel, achieved=round(ach, 1), peak=peak, unit="GB/s",
                        frac=round(ach / peak, 4), traffic=profiled_traffic(prof_kernel, w["name"]),
                        algorithmic_bytes=int(alg_bytes),
                        avg_launch_ms=round(avg_ms, 5), peak_source=f"{peak_kind} (hbm_gbs)")

    # end to end through the public API with host buffers
    e2e_evs = []
    y_h = torch.empty((U, cv["cout"]), dtype=torch.float32).pin_memory()
    for k in range(max(2, min(K, 10))):
        flush.fill_(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cd = coords_h.to(dev, non_blocking=True)
        xd = x_h.to(dev, non_blocking=True)
        Wd = W_h.to(dev, non_blocking=True)
        g = fvx.Grid.build(cd, offs)
        km = fvx.KernelMap(g, g, 1)
        yd = fvx.sparse_conv(g, g, km, xd, Wd)
        y_h.copy_(yd, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_evs.append(e0.elapsed_time(e1) / 1e3)
        km.destroy()
        g.destroy()
    t_e2e = max_over_ranks(sum(e2e_evs), world)
    e2e = dict(value=round(U * len(e2e_evs) * world / t_e2e / 1e6, 2), unit=UNIT,
               h2d_bytes_per_step=int(coords_h.numel() * 4 + x_h.numel() * 2 + W_h.numel() * 2),
               d2h_bytes_per_step=int(y_h.numel() * 4))

    out = dict(metric=METRIC, value=round(value, 2), unit=UNIT, n_gpus=world, steps=K, warmup=args.warmup,
               ms_per_step=round(t_total / K * 1e3, 4), higher_is_better=True, scaling="weak",
               vs_baseline=None, dtype="bf16", data="synthetic",
               config=dict(workload=w["name"], rows=int(w["coords"].shape[0]), active_voxels=U, pairs=int(npairs),
                           cin=cv["cin"], cout=cv["cout"], stride=1, batch=int(len(offs) - 1),
                           l2="flushed between steps (256 MB write outside the step events)",
                           parallelism=f"replicas x{world}"),
               components=dict(build_kmap_mvoxels_s=round(U * K / (t_build + t_kmap) / 1e6, 2),
                               conv_active_pair_tflops=round(flops * K / t_conv / 1e12, 4),
                               build_ms=round(t_build / K * 1e3, 4), kmap_ms=round(t_kmap / K * 1e3, 4),
                               conv_ms=round(t_conv / K * 1e3, 4)),
               roofline=roofline, e2e=e2e, gpu_launches=int(launches), clocks=clk)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w)
    return out


# ---------------------------------------------------------------- reference arm (the oracle)
def bench_reference(args, world, rank):
    if rank != 0:
        return None
    import oracle

    oracle.build()
    w = make_workload(args.workload)
    coords, offs, desc = oracle_sample(w, target_rows=120_000)
    cv = w["convs"][0]
    for _ in range(args.warmup):
        run_oracle_step(coords, offs, cv, 1)
    times, n = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        n = run_oracle_step(coords, offs, cv, 1)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = n * args.steps / tot / 1e6
    cb = dict(value=round(value, 4), unit=UNIT, cores=1, kind="oracle",
              sample=f"{desc}: build+kmap+conv of {n} voxels per step, single-threaded", host_cores=os.cpu_count())
    return dict(impl="reference", metric=METRIC, value=round(value, 4), unit=UNIT, n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(tot / args.steps * 1e3, 2), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                config=dict(workload=w["name"], sample=desc, cin=cv["cin"], cout=cv["cout"], stride=1),
                cpu_baseline=cb, e2e=dict(value=round(value, 4), unit=UNIT, h2d_bytes_per_step=0,
                                          d2h_bytes_per_step=0))


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        out = bench_reference(args, world, rank)
    else:
        out = bench_fvx(args, world, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

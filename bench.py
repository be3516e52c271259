"""Benchmark of the sparse-voxel hot path on GB300: IndexGrid build from
unsorted int32 coordinates -> 3x3x3 kernel map -> bf16 sparse convolution.

One step = one pass of the whole path over the workload: fvx_build_grid,
fvx_kernel_map, fvx_sparse_conv (and, for a stride-2 layer, fvx_coarsen and
its map and conv).  The default workload is the largest: a batch of 8
narrow-band grids in 1024^3 boxes (12.0M voxels from 17.1M unsorted rows with
30% duplicates, bf16 32 -> 64).  The four other workloads (tiny shell, leaf
dense, narrow band, LiDAR) are timed the same way after it and reported under
components.per_workload (skip with --no-all-workloads).

Prints ONE JSON line (rank 0).  `value` is whole-step throughput in active
voxels per second (Mvoxels/s) with inputs resident in HBM; `components` splits
it into the two quantities the metric names (build+kmap Mvoxels/s and conv
active-pair TFLOP/s).  `--impl reference` times the CPU oracle on a bounded
crop of the same workload instead (the crop the line's cpu_baseline times).
`--pass backward` times the training backward of the workload's convs
instead (transposed kernel map, input and weight gradients; its own metric,
in TFLOP/s).
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
    p.add_argument("--workload", default="batched_narrow_band")
    p.add_argument("--no-all-workloads", dest="all_workloads", action="store_false",
                   help="time only --workload (no per-workload entries for the other four)")
    p.add_argument("--scale", type=float, default=1.0,
                   help="smaller instance of the same workload generator (< 1), e.g. for profiler captures")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--profile-kernel", default=None, help="kernel whose launches are timed for the roofline")
    p.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward"],
                   help="forward: build -> kernel map -> conv (the default step); backward: the training "
                        "backward of the workload's convs (transposed kernel map, input and weight gradients)")
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

    src = {"conv_bf16_tc": "conv.cu", "conv_bf16_tma": "conv.cu", "conv_leaf": "conv.cu", "conv_halo": "conv.cu",
           "conv_wgrad_tc": "conv.cu", "kmap1_write": "kmap.cu"}.get(kernel)
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
def make_workload(name, scale=1.0):
    from sparse_convolution_gb300 import synth

    f = synth.WORKLOADS[name]
    return f(scale=scale) if scale != 1.0 else f()


def oracle_sample(w, target_rows=30_000):
    """A spatially contiguous crop of the workload (first batch element, lowest
    i) with about target_rows rows (fewer for wide convs, whose fp64 oracle
    cost grows with cin*cout): same density and structure, bounded CPU work.
    The CPU baseline and the reference arm time the same crop."""
    coords, offs = w["coords"], w["batch_offsets"]
    width = sum(c["cin"] * c["cout"] for c in w["convs"])
    target_rows = max(2000, int(target_rows * min(1.0, 2048.0 / width)))
    c = coords[offs[0]:offs[1]]
    if c.shape[0] <= target_rows:
        return c, np.array([0, c.shape[0]], np.int64), f"whole first batch element ({c.shape[0]} rows)"
    cut = np.partition(c[:, 0], target_rows)[target_rows]
    sel = c[c[:, 0] < cut]
    return sel, np.array([0, sel.shape[0]], np.int64), f"crop i < {int(cut)} of batch 0 ({sel.shape[0]} rows)"


def run_oracle_step(coords, offs, convs, seed):
    """The oracle's pass over one input: build, then per conv of the workload
    (coarsen for stride 2) kernel map and conv, each conv reading the last.
    Returns (active voxels, seconds in build + kernel maps, seconds in convs,
    active-pair flops)."""
    import oracle
    from sparse_convolution_gb300 import synth

    t0 = time.perf_counter()
    g = oracle.Grid.build(coords, offs)
    t_bk = time.perf_counter() - t0
    t_cv = 0.0
    flops = 0.0
    x = synth.features(seed, g.n_active, convs[0]["cin"]).astype(np.float64)
    gin = g
    for i, c in enumerate(convs):
        t0 = time.perf_counter()
        gout = gin if c["stride"] == 1 else gin.coarsen(c["stride"])
        km = oracle.KernelMap(gin, gout, c["stride"])
        t_bk += time.perf_counter() - t0
        W = synth.weights(seed + 1 + i, c["cin"], c["cout"]).astype(np.float64)
        t0 = time.perf_counter()
        x, _ = oracle.conv(km, x, W)
        t_cv += time.perf_counter() - t0
        flops += 2.0 * c["cin"] * c["cout"] * km.n_pairs
        gin = gout
    return g.n_active, t_bk, t_cv, flops


def oracle_passes(w, min_s, max_passes):
    """Repeats the oracle's pass over the shared crop until min_s seconds (at
    most max_passes passes); returns the per-pass figures and the crop."""
    coords, offs, desc = oracle_sample(w)
    n, tb, tc, fl, k = 0, 0.0, 0.0, 0.0, 0
    t0 = time.perf_counter()
    while k < max_passes and (k == 0 or time.perf_counter() - t0 < min_s):
        n, b, c, fl = run_oracle_step(coords, offs, w["convs"], 1)
        tb, tc, k = tb + b, tc + c, k + 1
    return dict(n=n, t_bk=tb / k, t_cv=tc / k, flops=fl, passes=k, desc=desc)


def cpu_baseline(w):
    """The oracle as it stands, single-threaded, on the crop the reference
    arm times (10-30 s of CPU work)."""
    r = oracle_passes(w, min_s=10.0, max_passes=8)
    t = r["t_bk"] + r["t_cv"]
    return dict(value=round(r["n"] / t / 1e6, 6), unit=UNIT, cores=1, kind="oracle",
                sample=f"{r['desc']}: oracle build + kernel map + conv of {r['n']} voxels per pass, "
                       f"{r['passes']} passes, single-threaded",
                build_kmap_mvoxels_s=round(r["n"] / r["t_bk"] / 1e6, 6),
                conv_active_pair_gflops=round(r["flops"] / r["t_cv"] / 1e9, 4),
                host_cores=os.cpu_count())


# ---------------------------------------------------------------- GPU arm
def ffma_peak(sm_count, peaks):
    """FP32 FFMA peak: SMs x 128 FP32 lanes x 2 flops x the maximum SM clock."""
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    return sm_count * 128 * 2 * mhz * 1e6 / 1e12, f"derived: {sm_count} SMs x 128 FP32 lanes x 2 x {mhz:.0f} MHz"


def conv_roofline(flops, alg_bytes, sec, fp32, peaks, peak_kind, sm_count):
    """Roofline of one conv kernel: FFMA for fp32, else tensor or HBM by the
    kernel's arithmetic intensity against the measured ridge."""
    if fp32:
        peak, src = ffma_peak(sm_count, peaks)
        r = dict(bound="alu", achieved=round(flops / sec / 1e12, 3), peak=round(peak, 1), unit="TFLOP/s",
                 peak_source=src)
    elif flops / alg_bytes > peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9):
        r = dict(bound="tensor", achieved=round(flops / sec / 1e12, 2), peak=peaks["bf16_tflops"], unit="TFLOP/s",
                 peak_source=f"{peak_kind} (bf16_tflops, burst)")
    else:
        r = dict(bound="hbm", achieved=round(alg_bytes / sec / 1e9, 1), peak=peaks["hbm_gbs"], unit="GB/s",
                 peak_source=f"{peak_kind} (hbm_gbs)")
    r["frac"] = round(r["achieved"] / r["peak"], 4)
    return r


class Workload:
    """One workload resident on the device: pinned host inputs, their device
    copies, output buffers, and the sizes of its grids."""

    def __init__(self, fvx, torch, synth, w, dev):
        self.w, self.dev = w, dev
        self.convs = w["convs"]
        self.fp32 = w["dtype"] == "f32"
        self.offs = w["batch_offsets"]
        self.coords_h = torch.from_numpy(w["coords"]).pin_memory()
        self.coords = self.coords_h.to(dev)
        g0 = fvx.Grid.build(self.coords, self.offs)
        self.U = g0.n_active
        self.n_out, self.leaves_out = [self.U], [g0.n_leaf]
        gin = g0
        for c in self.convs[1:]:  # a later conv reads the previous one's output grid
            gc = gin.coarsen(c["stride"]) if c["stride"] != 1 else gin
            self.n_out.append(gc.n_active)
            self.leaves_out.append(gc.n_leaf)
            if gc is not gin and gin is not g0:
                gin.destroy()
            gin = gc
        if gin is not g0:
            gin.destroy()
        g0.destroy()
        # feature rows follow the active-voxel index order; values are i.i.d.,
        # so any order is a valid input
        fdt = torch.float32 if self.fp32 else torch.bfloat16
        self.x_h = torch.from_numpy(synth.features(w["seed"] + 10, self.U, self.convs[0]["cin"],
                                                   w["feat_kind"])).to(fdt).pin_memory()
        self.W_h = [torch.from_numpy(synth.weights(w["seed"] + 20 + i, c["cin"], c["cout"])).to(fdt).pin_memory()
                    for i, c in enumerate(self.convs)]
        self.x = self.x_h.to(dev)
        self.Ws = [t.to(dev) for t in self.W_h]
        # outputs: fp32 (bf16 operands, fp32 accumulation: the mode whose error
        # meets 2e-3 * sum|w*x|); a conv that feeds the next one writes bf16
        self.ys = []
        for i, c in enumerate(self.convs):
            odt = torch.float32 if (self.fp32 or i == len(self.convs) - 1) else torch.bfloat16
            self.ys.append(torch.empty((self.n_out[i], c["cout"]), dtype=odt, device=dev))


def forward_step(fvx, wl, rec, coords_in, x_in, W_in, ys, stream=None, algos=None, pair_counts=None):
    """One pass of the path: build, then per conv (coarsen for stride 2)
    kernel map and conv.  rec(category) brackets each call with events.
    Returns the handles to release."""
    handles = []
    with rec("build"):
        g = fvx.Grid.build(coords_in, wl.offs, stream=stream)
    handles.append(g)
    src, gin = x_in, g
    for i, c in enumerate(wl.convs):
        if c["stride"] == 1:
            gout = gin
        else:
            with rec("build"):
                gout = gin.coarsen(c["stride"], stream=stream)
            handles.append(gout)
        with rec("kmap"):
            km = fvx.KernelMap(gin, gout, c["stride"], stream=stream)
        handles.append(km)
        if pair_counts is not None and len(pair_counts) < len(wl.convs):  # read once (the read synchronises)
            pair_counts.append(km.n_pairs)
        with rec(f"conv{i}"):
            fvx.sparse_conv(gin, gout, km, src, W_in[i], out=ys[i], stream=stream)
        if algos is not None and len(algos) < len(wl.convs):
            algos.append(fvx.last_conv_kernel())
        src, gin = ys[i], gout
    return handles


def release(handles):
    for hnd in reversed(handles):
        hnd.destroy()


class EventRec:
    """Records (category, start event, end event) around each bracketed call
    on the given stream."""

    def __init__(self, torch, stream):
        self.torch, self.stream, self.marks = torch, stream, []

    def __call__(self, cat):
        self.cat = cat
        return self

    def __enter__(self):
        self.e0 = self.torch.cuda.Event(enable_timing=True)
        self.e0.record(self.stream)
        return self

    def __exit__(self, *a):
        e1 = self.torch.cuda.Event(enable_timing=True)
        e1.record(self.stream)
        self.marks.append((self.cat, self.e0, e1))
        return False


class NoRec:
    def __call__(self, cat):
        return self

    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def time_forward(fvx, torch, wl, K, warmup, flush, peaks, peak_kind, sm_count, world=1, clocks=None):
    """Warm-up, then K timed steps (L2 flushed before each, outside the
    events).  Per call category CUDA-event time; per conv kernel the launch
    durations the library's event timing records.  Returns the workload's
    figures and the raw timing for the caller's line."""
    stream = torch.cuda.current_stream()
    algos, pairs = [], []
    for _ in range(max(1, warmup)):
        release(forward_step(fvx, wl, NoRec(), wl.coords, wl.x, wl.Ws, wl.ys, algos=algos, pair_counts=pairs))
    torch.cuda.synchronize()
    fvx.device_status()
    kernels = list(algos)  # kernel names the library reports for each conv
    flops_i = [2.0 * c["cin"] * c["cout"] * p for c, p in zip(wl.convs, pairs)]
    # the kernel timed in the main loop: the one doing the most arithmetic
    main_k = kernels[max(range(len(wl.convs)), key=lambda i: flops_i[i])]
    recs = EventRec(torch, stream)
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    fvx.profile_enable(main_k)
    l0 = fvx.launch_count()
    for k in range(K):
        flush.fill_(float(k))  # evict L2 between steps (outside the step's events)
        release(forward_step(fvx, wl, recs, wl.coords, wl.x, wl.Ws, wl.ys))
    torch.cuda.synchronize()
    launches = fvx.launch_count() - l0
    each = {main_k: fvx.profile_read_each(cap=64 * K)}
    fvx.profile_enable(None)
    barrier(world)
    clk = clocks.stop() if clocks is not None else None
    fvx.device_status()
    # a conv kernel other than the main one: timed in a second loop of its own
    for kn in sorted(set(kernels) - {main_k}):
        fvx.profile_enable(kn)
        for k in range(K):
            flush.fill_(float(k))
            release(forward_step(fvx, wl, NoRec(), wl.coords, wl.x, wl.Ws, wl.ys))
        torch.cuda.synchronize()
        each[kn] = fvx.profile_read_each(cap=64 * K)
        fvx.profile_enable(None)
    t = {}
    for cat, e0, e1 in recs.marks:
        t[cat] = t.get(cat, 0.0) + e0.elapsed_time(e1) / 1e3
    t_conv = sum(v for c_, v in t.items() if c_.startswith("conv"))
    t_total = t["build"] + t["kmap"] + t_conv
    # per conv: its kernel's launches (launch order within a step = conv order)
    per_conv = []
    esz = 4 if wl.fp32 else 2
    n_in = wl.U
    for i, (c, p) in enumerate(zip(wl.convs, pairs)):
        kn = kernels[i]
        same = [j for j in range(len(wl.convs)) if kernels[j] == kn]
        durs = each[kn]
        per_step = len(durs) // K if K else 0
        mine = []
        L = 1  # launches per conv (the halo-staged kernel runs one per 32 input channels)
        if per_step and per_step % len(same) == 0:
            L = per_step // len(same)
            pos = same.index(i)
            mine = [sum(durs[k * per_step + pos * L:k * per_step + (pos + 1) * L]) for k in range(K)]
        sec = sum(mine) / 1e3 if mine else t[f"conv{i}"]
        nk = len(mine) if mine else K
        # algorithmic bytes: feats read once, output written once (4 B fp32 /
        # 2 B bf16), weights once, plus what locates the inputs: the kernel
        # map's (in, out) int32 pair for the pair-list kernels, the output
        # leaf's 80-byte record for the leaf-densified kernel, that record and
        # the leaf's 27 int32 neighbour-leaf ids for the halo-staged kernel
        where = (80 * wl.leaves_out[i] if kn == "conv_leaf" else 188 * wl.leaves_out[i] if kn == "conv_halo"
                 else 8 * p)
        alg = (n_in * c["cin"] * esz + wl.n_out[i] * c["cout"] * wl.ys[i].element_size()
               + 27 * c["cin"] * c["cout"] * esz + where)
        rl = conv_roofline(flops_i[i] * nk, alg * nk, sec, wl.fp32, peaks, peak_kind, sm_count)
        per_conv.append(dict(conv=f"{c['cin']}->{c['cout']} stride {c['stride']}", kernel=kn, pairs=int(p),
                             mean_pairs_per_output=round(p / wl.n_out[i], 3),
                             kernel_ms=round(sec / nk * 1e3, 5), launches=L, call_ms=round(t[f"conv{i}"] / K * 1e3, 5),
                             active_pair_tflops=round(flops_i[i] * nk / sec / 1e12, 3),
                             algorithmic_bytes=int(alg), flops=int(flops_i[i]), roofline=rl,
                             kernel_timing="CUDA events around each launch" if mine else "call events"))
        n_in = wl.n_out[i]
    # build + kernel map against HBM, as effective bandwidth: per input row
    # 170 B (key encode, about five radix passes, flag scans, sidecars; the
    # one-tile bitmap path sorts nothing but is credited the same bytes), per
    # output voxel 76 B plus 8 B per pair (coordinates, leaf words, mask,
    # scans; the pair lists written once)
    rows = wl.w["coords"].shape[0]
    b_bytes = 170.0 * rows
    k_bytes = sum(76.0 * n + 8.0 * p for n, p in zip(wl.n_out, pairs))
    hbm = peaks["hbm_gbs"]
    s1 = [c for c in range(len(wl.convs)) if wl.convs[c]["stride"] == 1]
    entry = dict(
        workload=wl.w["name"], rows=int(rows), active_voxels=int(wl.U), batch=int(len(wl.offs) - 1),
        mean_active_neighbours=(round(pairs[s1[0]] / wl.n_out[s1[0]] - 1.0, 3) if s1 else None),
        step_ms=round(t_total / K * 1e3, 4), build_ms=round(t["build"] / K * 1e3, 4),
        kmap_ms=round(t["kmap"] / K * 1e3, 4), conv_ms=round(t_conv / K * 1e3, 4),
        step_mvoxels_s=round(wl.U * K / t_total / 1e6, 2),
        build_kmap_mvoxels_s=round(wl.U * K / (t["build"] + t["kmap"]) / 1e6, 2),
        build_kmap_hbm=dict(
            kind="effective bandwidth: fixed per-unit bytes over measured time",
            build_bytes=int(b_bytes), kmap_bytes=int(k_bytes),
            build_gbs=round(b_bytes * K / t["build"] / 1e9, 1), kmap_gbs=round(k_bytes * K / t["kmap"] / 1e9, 1),
            build_frac=round(b_bytes * K / t["build"] / 1e9 / hbm, 4),
            kmap_frac=round(k_bytes * K / t["kmap"] / 1e9 / hbm, 4),
            frac=round((b_bytes + k_bytes) * K / (t["build"] + t["kmap"]) / 1e9 / hbm, 4)),
        conv_active_pair_tflops=round(sum(flops_i) * K / t_conv / 1e12, 4),
        convs=per_conv)
    raw = dict(t_total=t_total, pairs=pairs, kernels=kernels, launches=launches, clocks=clk, main_kernel=main_k)
    return entry, raw


def e2e_forward(fvx, torch, wl, K, world):
    """End to end through the public API with host buffers: every step copies
    its inputs in from pinned host memory and its result back out, all inside
    the timed region.  Steps are pipelined two deep, as a serving loop would
    run them: each slot has its own stream (build -> kernel map -> conv ->
    result download) and an upload stream (features and weights) that
    overlaps the slot's build; step k's download overlaps step k+1's work."""
    dev = wl.dev
    n_e2e = max(2, min(K, 10))
    main_s = [torch.cuda.Stream(device=dev) for _ in range(2)]
    up_s = [torch.cuda.Stream(device=dev) for _ in range(2)]
    cd_slot = [torch.empty_like(wl.coords) for _ in range(2)]
    xd_slot = [torch.empty_like(wl.x) for _ in range(2)]
    Wd_slot = [[torch.empty_like(t_) for t_ in wl.Ws] for _ in range(2)]
    ys_slot = [[torch.empty_like(y_) for y_ in wl.ys] for _ in range(2)]
    y_h = [torch.empty(wl.ys[-1].shape, dtype=wl.ys[-1].dtype).pin_memory() for _ in range(2)]
    conv_done = [None, None]
    up_done = [None, None]

    def upload(k):
        sl = k & 1
        us = up_s[sl]
        with torch.cuda.stream(us):
            if conv_done[sl] is not None:
                us.wait_event(conv_done[sl])  # the slot's previous step has read its inputs
            cd_slot[sl].copy_(wl.coords_h, non_blocking=True)
            xd_slot[sl].copy_(wl.x_h, non_blocking=True)
            for d_, h_ in zip(Wd_slot[sl], wl.W_h):
                d_.copy_(h_, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(us)
            up_done[sl] = ev

    def compute(k):
        sl = k & 1
        ms = main_s[sl]
        with torch.cuda.stream(ms):
            ms.wait_event(up_done[sl])
            handles = forward_step(fvx, wl, NoRec(), cd_slot[sl], xd_slot[sl], Wd_slot[sl], ys_slot[sl], stream=ms)
            done = torch.cuda.Event()
            done.record(ms)
            conv_done[sl] = done
            y_h[sl].copy_(ys_slot[sl][-1], non_blocking=True)
        release(handles)  # frees are ordered on the slot's stream

    def run(n):
        # the host issues step k+1's uploads before step k's build (whose
        # count reads block the host)
        upload(0)
        for k in range(n):
            if k + 1 < n:
                upload(k + 1)
            compute(k)

    run(2)  # warm the pipeline (allocator pools, streams)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(main_s[0])
    for st in (main_s[1], up_s[0], up_s[1]):
        st.wait_event(e_start)
    run(n_e2e)
    for st in (main_s[1], up_s[0], up_s[1]):
        main_s[0].wait_stream(st)
    e_end.record(main_s[0])
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(e_start.elapsed_time(e_end) / 1e3, world)
    return dict(value=round(wl.U * n_e2e * world / t_e2e / 1e6, 2), unit=UNIT,
                h2d_bytes_per_step=int(wl.coords_h.numel() * 4 + wl.x_h.numel() * wl.x_h.element_size()
                                       + sum(t_.numel() * t_.element_size() for t_ in wl.W_h)),
                d2h_bytes_per_step=int(y_h[0].numel() * y_h[0].element_size()),
                steps=n_e2e, pipeline="2 steps in flight on 2 streams; step k+1's uploads overlap step k")


def time_rays(fvx, torch, synth, box, K, warmup, flush, peaks):
    """Voxels along rays (HDDA) on the narrow-band scene of side ``box`` with
    a 1024 x 1024 pinhole camera: K whole calls (count pass, scan, one
    synchronisation for the total, output allocation, write pass), each timed
    with CUDA events after an L2 flush; per kernel, its launch durations."""
    w = synth.ray_scene(box)
    o_h, d_h = synth.camera_rays(box, 1024)
    dev = torch.device("cuda", torch.cuda.current_device())
    g = fvx.Grid.build(torch.from_numpy(w["coords"]).to(dev), w["batch_offsets"])
    o = torch.from_numpy(o_h).to(dev)
    d = torch.from_numpy(d_h).to(dev)
    for _ in range(max(1, warmup)):
        fvx.Hits(g, o, d).destroy()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts, hits = [], 0
    for k in range(K):
        flush.fill_(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h = fvx.Hits(g, o, d)
        e1.record(stream)
        hits = h.n_hits
        h.destroy()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    kern = {}
    for kn in ("rays_count", "rays_write"):
        fvx.profile_enable(kn)
        for k in range(K):
            flush.fill_(float(k))
            fvx.Hits(g, o, d).destroy()
        torch.cuda.synchronize()
        ms, nl = fvx.profile_read()
        fvx.profile_enable(None)
        kern[kn + "_ms"] = round(ms / max(1, nl), 5)
    fvx.device_status()
    n = o_h.shape[0]
    ms = statistics.median(ts)
    # bytes the call must move: rays read by both passes (24 B each), counts
    # written and read, offsets written (8 B per ray), hits written (4 B
    # index + 8 B times)
    alg = 2 * 24 * n + 8 * n + 8 * (n + 1) + 12 * hits
    out = dict(scene=w["name"], voxels=int(g.n_active), rays=int(n), hits=int(hits),
               rays_with_hits=int(np.count_nonzero(np.diff(ray_offsets(fvx, g, o, d)) > 0)),
               ms_per_call=round(ms, 4), mrays_per_s=round(n / ms / 1e3, 2), mhits_per_s=round(hits / ms / 1e3, 2),
               kernels=kern,
               hbm=dict(algorithmic_bytes=int(alg), achieved_gbs=round(alg / ms / 1e6, 1),
                        frac=round(alg / ms / 1e6 / peaks["hbm_gbs"], 4),
                        note="the walk is bound by dependent node loads per ray, not by bytes"))
    g.destroy()
    return out


def ray_offsets(fvx, g, o, d):
    h = fvx.Hits(g, o, d)
    off = h.arrays()[0].cpu().numpy()
    h.destroy()
    return off


def bench_fvx(args, world, rank, local):
    import torch

    from sparse_convolution_gb300 import build_lib
    import sparse_convolution_gb300 as fvx
    from sparse_convolution_gb300 import synth

    torch.cuda.set_device(local)
    build_lib.build()
    fvx.load()
    dev = torch.device("cuda", local)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    peaks, peak_kind = measured_peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    K = args.steps

    w = make_workload(args.workload, args.scale)
    wl = Workload(fvx, torch, synth, w, dev)
    clocks = ClockSampler(local)
    entry, raw = time_forward(fvx, torch, wl, K, args.warmup, flush, peaks, peak_kind, sm_count, world, clocks)
    t_total = max_over_ranks(raw["t_total"], world)
    value = wl.U * K * world / t_total / 1e6
    # the line's roofline: the conv kernel doing the most arithmetic
    big = max(range(len(entry["convs"])), key=lambda i: entry["convs"][i]["flops"])
    cv = entry["convs"][big]
    roofline = dict(cv["roofline"])
    same = [c for c in entry["convs"] if c["kernel"] == cv["kernel"]]
    roofline.update(kernel=cv["kernel"], conv=cv["conv"],
                    traffic=profiled_traffic(cv["kernel"], w["name"]) if len(same) == 1 else None,
                    algorithmic_bytes=cv["algorithmic_bytes"], flops=cv["flops"],
                    avg_launch_ms=round(cv["kernel_ms"] / cv["launches"], 5), launches_per_step=cv["launches"],
                    per="conv call (all its launches)")
    e2e = e2e_forward(fvx, torch, wl, K, world)
    del wl

    # the other workloads (parity-test sizes of the same generators at full
    # size), each timed the same way; the headline's entry comes first
    per_workload = [entry]
    if args.all_workloads and args.scale == 1.0 and rank == 0:
        for name in synth.WORKLOADS:
            if name == args.workload:
                continue
            wo = Workload(fvx, torch, synth, make_workload(name), dev)
            e, _ = time_forward(fvx, torch, wo, K, args.warmup, flush, peaks, peak_kind, sm_count, 1, None)
            per_workload.append(e)
            del wo
            torch.cuda.empty_cache()

    rays = []
    if args.all_workloads and args.scale == 1.0 and rank == 0:
        for box in (128, 1024):
            rays.append(time_rays(fvx, torch, synth, box, K, args.warmup, flush, peaks))
            torch.cuda.empty_cache()

    out = dict(metric=METRIC, value=round(value, 2), unit=UNIT, n_gpus=world, steps=K, warmup=args.warmup,
               ms_per_step=round(t_total / K * 1e3, 4), higher_is_better=True, scaling="weak",
               vs_baseline=None, dtype="f32" if w["dtype"] == "f32" else "bf16", data="synthetic",
               config=dict(workload=w["name"], rows=int(w["coords"].shape[0]), active_voxels=entry["active_voxels"],
                           pairs=[c["pairs"] for c in entry["convs"]],
                           convs=[c["conv"] for c in entry["convs"]],
                           mean_active_neighbours=entry["mean_active_neighbours"],
                           batch=entry["batch"],
                           l2="flushed between steps (256 MB write outside the step events)",
                           parallelism=f"replicas x{world}", sm_count=sm_count),
               components=dict(build_kmap_mvoxels_s=entry["build_kmap_mvoxels_s"],
                               conv_active_pair_tflops=entry["conv_active_pair_tflops"],
                               build_ms=entry["build_ms"], kmap_ms=entry["kmap_ms"], conv_ms=entry["conv_ms"],
                               conv_kernels=raw["kernels"], build_kmap_hbm=entry["build_kmap_hbm"],
                               per_workload=per_workload, rays=rays),
               roofline=roofline, e2e=e2e, gpu_launches=int(raw["launches"]), clocks=raw["clocks"])
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w)
    return out


# ---------------------------------------------------------------- backward pass
BWD_METRIC = "sparse conv3d backward (input + weight gradient) active-pair TFLOP/s"


def oracle_backward(coords, offs, convs, seed):
    """The oracle's backward of the workload's first conv on a sample: the
    transposed map, dx = conv of dy over it with W^T, and dW.  Returns the
    active-pair flops (4 * pairs * cin * cout)."""
    import oracle
    from sparse_convolution_gb300 import synth

    c = convs[0]
    g = oracle.Grid.build(coords, offs)
    go = g if c["stride"] == 1 else g.coarsen(c["stride"])
    km = oracle.KernelMap(g, go, c["stride"])
    kt = oracle.KernelMap(go, g, c["stride"], transposed=True)
    x = synth.features(seed, g.n_active, c["cin"]).astype(np.float64)
    dy = synth.features(seed + 1, go.n_active, c["cout"]).astype(np.float64)
    W = synth.weights(seed + 2, c["cin"], c["cout"]).astype(np.float64)
    oracle.conv(kt, dy, np.ascontiguousarray(W.transpose(0, 2, 1)))
    oracle.conv_wgrad(km, x, dy)
    return 4.0 * km.n_pairs * c["cin"] * c["cout"]


def bench_backward(args, world, rank, local):
    """Backward of the workload's convs with the forward pass's grids and
    kernel maps given (built once, outside the timed region).  A step, per
    conv: the transposed kernel map (gout -> gin), dx = fvx_sparse_conv_dgrad,
    dW = fvx_sparse_conv_wgrad.  value = active-pair flops of the two
    gradients (2 * 2 * pairs * cin * cout) per second."""
    import torch

    from sparse_convolution_gb300 import build_lib
    import sparse_convolution_gb300 as fvx
    from sparse_convolution_gb300 import synth

    torch.cuda.set_device(local)
    build_lib.build()
    fvx.load()
    w = make_workload(args.workload, args.scale)
    convs = w["convs"]
    fp32 = w["dtype"] == "f32"
    dev = torch.device("cuda", local)
    fdt = torch.float32 if fp32 else torch.bfloat16
    g = fvx.Grid.build(torch.from_numpy(w["coords"]).to(dev), w["batch_offsets"])
    grids, kms, pairs = [g], [], []
    for c in convs:
        gin = grids[-1]
        gout = gin if c["stride"] == 1 else gin.coarsen(c["stride"])
        grids.append(gout)
        km = fvx.KernelMap(gin, gout, c["stride"])
        kms.append(km)
        pairs.append(km.n_pairs)
    gi = [grids[i] for i in range(len(convs))]
    go = [grids[i + 1] for i in range(len(convs))]
    x_h = [torch.from_numpy(synth.features(w["seed"] + 30 + i, gi[i].n_active, c["cin"], w["feat_kind"])).to(fdt)
           .pin_memory() for i, c in enumerate(convs)]
    dy_h = [torch.from_numpy(synth.features(w["seed"] + 40 + i, go[i].n_active, c["cout"], w["feat_kind"])).to(fdt)
            .pin_memory() for i, c in enumerate(convs)]
    W_h = [torch.from_numpy(synth.weights(w["seed"] + 20 + i, c["cin"], c["cout"])).to(fdt).pin_memory()
           for i, c in enumerate(convs)]
    xs = [t.to(dev) for t in x_h]
    dys = [t.to(dev) for t in dy_h]
    Ws = [t.to(dev) for t in W_h]
    dxs = [torch.empty((gi[i].n_active, c["cin"]), dtype=torch.float32, device=dev) for i, c in enumerate(convs)]
    dWs = [torch.empty((27, c["cin"], c["cout"]), dtype=torch.float32, device=dev) for c in convs]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def wgrad_kernel(c):  # the library's choice for this layer
        if c["cin"] * c["cout"] <= 1024 and c["cin"] + c["cout"] <= 64:
            return "conv_wgrad_small"
        if not fp32 and c["cin"] % 8 == 0 and c["cout"] % 8 == 0:
            return "conv_wgrad_tc"
        return "conv_wgrad"

    marks = []

    def rec(cat, fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        r = fn()
        e1.record(stream)
        marks.append((cat, e0, e1))
        return r

    def step(x_in, dy_in, W_in, dx_out, dW_out, timed):
        for i, c in enumerate(convs):
            if timed:
                kt = rec("kmap_t", lambda: fvx.KernelMap(go[i], gi[i], c["stride"], transposed=True))
                rec("dgrad", lambda: fvx.sparse_conv_dgrad(gi[i], go[i], kt, dy_in[i], W_in[i], out=dx_out[i]))
                rec("wgrad", lambda: fvx.sparse_conv_wgrad(gi[i], go[i], kms[i], x_in[i], dy_in[i], out=dW_out[i]))
            else:
                kt = fvx.KernelMap(go[i], gi[i], c["stride"], transposed=True)
                fvx.sparse_conv_dgrad(gi[i], go[i], kt, dy_in[i], W_in[i], out=dx_out[i])
                fvx.sparse_conv_wgrad(gi[i], go[i], kms[i], x_in[i], dy_in[i], out=dW_out[i])
            kt.destroy()

    for _ in range(args.warmup):
        step(xs, dys, Ws, dxs, dWs, False)
    torch.cuda.synchronize()
    fvx.device_status()
    flops_i = [4.0 * p * c["cin"] * c["cout"] for c, p in zip(convs, pairs)]
    big = max(range(len(convs)), key=lambda i: flops_i[i])
    prof_kernel = args.profile_kernel or wgrad_kernel(convs[big])
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    fvx.profile_enable(prof_kernel)
    l0 = fvx.launch_count()
    K = args.steps
    for k in range(K):
        flush.fill_(float(k))
        step(xs, dys, Ws, dxs, dWs, True)
    torch.cuda.synchronize()
    launches = fvx.launch_count() - l0
    prof_ms, prof_n = fvx.profile_read()
    fvx.profile_enable(None)
    barrier(world)
    clk = clocks.stop()
    fvx.device_status()
    t = {"kmap_t": 0.0, "dgrad": 0.0, "wgrad": 0.0}
    for cat, e0, e1 in marks:
        t[cat] += e0.elapsed_time(e1) / 1e3
    t_total = max_over_ranks(sum(t.values()), world)
    value = sum(flops_i) * K * world / t_total / 1e12

    peaks, peak_kind = measured_peaks()
    roofline = None
    if prof_n:
        mine = [i for i, c in enumerate(convs) if wgrad_kernel(c) == prof_kernel]
        wflops = sum(flops_i[i] / 2 for i in mine)  # the weight gradient's half
        ach = wflops * K / (prof_ms / 1e3) / 1e12
        if prof_kernel == "conv_wgrad_tc":
            roofline = dict(bound="tensor", achieved=round(ach, 2), peak=peaks["bf16_tflops"], unit="TFLOP/s",
                            peak_source=f"{peak_kind} (bf16_tflops, burst)")
        else:
            peak, src = ffma_peak(torch.cuda.get_device_properties(dev).multi_processor_count, peaks)
            roofline = dict(bound="alu", achieved=round(ach, 3), peak=round(peak, 1), unit="TFLOP/s",
                            peak_source=src)
        roofline.update(kernel=prof_kernel, frac=round(roofline["achieved"] / roofline["peak"], 4),
                        traffic=profiled_traffic(prof_kernel, w["name"]) if len(mine) == 1 else None,
                        flops=int(wflops / max(1, prof_n // K)), avg_launch_ms=round(prof_ms / prof_n, 5),
                        launches_per_step=int(prof_n // K))

    # end to end: every step uploads x, dy and W from pinned host memory and
    # downloads dx and dW, inside the timed region (one stream)
    n_e2e = max(2, min(K, 10))
    xd = [torch.empty_like(t_) for t_ in xs]
    dyd = [torch.empty_like(t_) for t_ in dys]
    Wd = [torch.empty_like(t_) for t_ in Ws]
    dx_h = [torch.empty(t_.shape, dtype=t_.dtype).pin_memory() for t_ in dxs]
    dW_h = [torch.empty(t_.shape, dtype=t_.dtype).pin_memory() for t_ in dWs]

    def e2e_step():
        for d_, h_ in zip(xd + dyd + Wd, x_h + dy_h + W_h):
            d_.copy_(h_, non_blocking=True)
        step(xd, dyd, Wd, dxs, dWs, False)
        for h_, d_ in zip(dx_h + dW_h, dxs + dWs):
            h_.copy_(d_, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e = dict(value=round(sum(flops_i) * n_e2e * world / t_e2e / 1e12, 3), unit="TFLOP/s",
               h2d_bytes_per_step=int(sum(t_.numel() * t_.element_size() for t_ in x_h + dy_h + W_h)),
               d2h_bytes_per_step=int(sum(t_.numel() * t_.element_size() for t_ in dx_h + dW_h)), steps=n_e2e)
    out = dict(metric=BWD_METRIC, value=round(value, 3), unit="TFLOP/s", n_gpus=world, steps=K, warmup=args.warmup,
               ms_per_step=round(t_total / K * 1e3, 4), higher_is_better=True, scaling="weak", vs_baseline=None,
               dtype="f32" if fp32 else "bf16", data="synthetic",
               config=dict(workload=w["name"], active_voxels=int(g.n_active), pairs=[int(p) for p in pairs],
                           convs=[f"{c['cin']}->{c['cout']} stride {c['stride']}" for c in convs],
                           step="per conv: transposed kernel map, input gradient, weight gradient",
                           l2="flushed between steps (256 MB write outside the step events)",
                           parallelism=f"replicas x{world}"),
               components=dict(kmap_t_ms=round(t["kmap_t"] / K * 1e3, 4), dgrad_ms=round(t["dgrad"] / K * 1e3, 4),
                               wgrad_ms=round(t["wgrad"] / K * 1e3, 4),
                               dgrad_tflops=round(sum(flops_i) / 2 * K / t["dgrad"] / 1e12, 3),
                               wgrad_tflops=round(sum(flops_i) / 2 * K / t["wgrad"] / 1e12, 3),
                               wgrad_kernels=[wgrad_kernel(c) for c in convs]),
               roofline=roofline, e2e=e2e, gpu_launches=int(launches), clocks=clk)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        coords, offs, desc = oracle_sample(w, target_rows=60_000)
        t0 = time.perf_counter()
        fl = oracle_backward(coords, offs, convs, 1)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = dict(value=fl / dt / 1e12, unit="TFLOP/s", cores=1, kind="oracle",
                                   sample=f"{desc}: backward of the first conv (transposed map, dx, dW), "
                                          f"single-threaded, {dt:.1f} s", host_cores=os.cpu_count())
    for km in kms:
        km.destroy()
    for gr in grids[1:]:
        if gr is not g:
            gr.destroy()
    g.destroy()
    return out


# ---------------------------------------------------------------- reference arm (the oracle)
def bench_reference(args, world, rank):
    """The oracle, as it stands, single-threaded on the host: W + K passes
    over the crop that the fvx line's cpu_baseline times (oracle_sample), each
    pass build + kernel map + conv of the workload's layers."""
    if rank != 0:
        return None
    import oracle

    oracle.build()
    w = make_workload(args.workload, args.scale)
    coords, offs, desc = oracle_sample(w)
    for _ in range(args.warmup):
        run_oracle_step(coords, offs, w["convs"], 1)
    n, tb, tc, fl = 0, 0.0, 0.0, 0.0
    for _ in range(args.steps):
        n, b, c, fl = run_oracle_step(coords, offs, w["convs"], 1)
        tb, tc = tb + b, tc + c
    tot = tb + tc
    value = n * args.steps / tot / 1e6
    cb = dict(value=round(value, 6), unit=UNIT, cores=1, kind="oracle",
              sample=f"{desc}: oracle build + kernel map + conv of {n} voxels per pass, {args.steps} passes, "
                     f"single-threaded",
              build_kmap_mvoxels_s=round(n * args.steps / tb / 1e6, 6),
              conv_active_pair_gflops=round(fl * args.steps / tc / 1e9, 4), host_cores=os.cpu_count())
    return dict(impl="reference", metric=METRIC, value=round(value, 6), unit=UNIT, n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(tot / args.steps * 1e3, 2), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                config=dict(workload=w["name"], sample=desc,
                            convs=[f"{c['cin']}->{c['cout']} stride {c['stride']}" for c in w["convs"]]),
                cpu_baseline=cb, e2e=dict(value=round(value, 6), unit=UNIT, h2d_bytes_per_step=0,
                                          d2h_bytes_per_step=0))


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        out = bench_reference(args, world, rank)
    elif args.which == "backward":
        out = bench_backward(args, world, rank, local)
    else:
        out = bench_fvx(args, world, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

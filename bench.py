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
sample of the same workload instead.  `--pass backward` times the training
backward of the workload's convs instead (transposed kernel map, input and
weight gradients; its own metric, in TFLOP/s).
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

    src = {"conv_bf16_tc": "conv.cu", "conv_bf16_tma": "conv.cu", "conv_leaf": "conv.cu",
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


def oracle_sample(w, target_rows=250_000):
    """A spatially contiguous crop of the workload (first batch, lowest i)
    with about target_rows rows (fewer for wide convs, whose fp64 oracle cost
    grows with cin*cout): same density and structure, bounded CPU work."""
    coords, offs = w["coords"], w["batch_offsets"]
    width = sum(c["cin"] * c["cout"] for c in w["convs"])
    target_rows = max(2000, int(target_rows * min(1.0, 2048.0 / width)))
    c = coords[offs[0]:offs[1]]
    if c.shape[0] <= target_rows:
        return c, np.array([0, c.shape[0]], np.int64), "whole first batch element"
    cut = np.partition(c[:, 0], target_rows)[target_rows]
    sel = c[c[:, 0] < cut]
    return sel, np.array([0, sel.shape[0]], np.int64), f"crop i < {int(cut)} of batch 0 ({sel.shape[0]} rows)"


def run_oracle_step(coords, offs, convs, seed):
    """The oracle's pass over one input: build, then per conv of the workload
    (coarsen for stride 2) kernel map and conv, each conv reading the last."""
    import oracle
    from sparse_convolution_gb300 import synth

    g = oracle.Grid.build(coords, offs)
    x = synth.features(seed, g.n_active, convs[0]["cin"]).astype(np.float64)
    gin = g
    for i, c in enumerate(convs):
        gout = gin if c["stride"] == 1 else gin.coarsen(c["stride"])
        km = oracle.KernelMap(gin, gout, c["stride"])
        W = synth.weights(seed + 1 + i, c["cin"], c["cout"]).astype(np.float64)
        x, _ = oracle.conv(km, x, W)
        gin = gout
    return g.n_active


def cpu_baseline(w, budget_s=20.0):
    coords, offs, desc = oracle_sample(w)
    t0 = time.perf_counter()
    n = run_oracle_step(coords, offs, w["convs"], 1)
    dt = time.perf_counter() - t0
    return dict(value=n / dt / 1e6, unit=UNIT, cores=1, kind="oracle",
                sample=f"{desc}: build+kmap+conv of {n} voxels, single-threaded, {dt:.1f} s",
                host_cores=os.cpu_count())


# ---------------------------------------------------------------- GPU arm
def bench_fvx(args, world, rank, local):
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
    coords_h = torch.from_numpy(w["coords"]).pin_memory()
    offs = w["batch_offsets"]
    coords = coords_h.to(dev)
    g0 = fvx.Grid.build(coords, offs)
    U = g0.n_active
    n_out, leaves_out = [U], [g0.n_leaf]
    if len(convs) > 1:
        gc0 = g0.coarsen(2)
        n_out.append(gc0.n_active)
        leaves_out.append(gc0.n_leaf)
        gc0.destroy()
    g0.destroy()
    # feature rows follow the active-voxel index order; values are i.i.d., so any order is a valid input
    fdt = torch.float32 if fp32 else torch.bfloat16
    x_h = torch.from_numpy(synth.features(w["seed"] + 10, U, convs[0]["cin"], w["feat_kind"])).to(fdt).pin_memory()
    W_h = [torch.from_numpy(synth.weights(w["seed"] + 20 + i, c["cin"], c["cout"])).to(fdt).pin_memory()
           for i, c in enumerate(convs)]
    x = x_h.to(dev)
    Ws = [t.to(dev) for t in W_h]
    # outputs: fp32 (bf16 operands, fp32 accumulation: the mode whose error meets
    # 2e-3 * sum|w*x|); a conv that feeds the next one writes bf16
    ys = []
    for i, c in enumerate(convs):
        odt = torch.float32 if (fp32 or i == len(convs) - 1) else torch.bfloat16
        ys.append(torch.empty((n_out[i], c["cout"]), dtype=odt, device=dev))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    algos = []  # kernel family each conv ran (recorded on the first step)
    pair_counts = []  # pairs of each conv's kernel map (first step)

    def step(rec, coords_in, x_in, W_in):
        """One pass of the path.  rec(category) brackets each call with events."""
        handles = []
        with rec("build"):
            g = fvx.Grid.build(coords_in, offs)
        handles.append(g)
        src, gin = x_in, g
        for i, c in enumerate(convs):
            if c["stride"] == 1:
                gout = gin
            else:
                with rec("build"):
                    gout = gin.coarsen(c["stride"])
                handles.append(gout)
            with rec("kmap"):
                km = fvx.KernelMap(gin, gout, c["stride"])
            handles.append(km)
            if len(pair_counts) < len(convs):  # read once (the read synchronises)
                pair_counts.append(km.n_pairs)
            with rec("conv"):
                fvx.sparse_conv(gin, gout, km, src, W_in[i], out=ys[i])
            if len(algos) < len(convs):
                algos.append(fvx.last_conv_algo())
            src, gin = ys[i], gout
        return handles, pair_counts

    class NoRec:
        def __call__(self, cat):
            return self

        def __enter__(self):
            return self

        def __exit__(self, *a):
            return False

    class EventRec:
        def __init__(self):
            self.marks = []

        def __call__(self, cat):
            self.cat = cat
            return self

        def __enter__(self):
            self.e0 = torch.cuda.Event(enable_timing=True)
            self.e0.record(stream)
            return self

        def __exit__(self, *a):
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(stream)
            self.marks.append((self.cat, self.e0, e1))
            return False

    def release(handles):
        for hnd in reversed(handles):
            hnd.destroy()

    for _ in range(args.warmup):
        hs, pairs = step(NoRec(), coords, x, Ws)
        release(hs)
    torch.cuda.synchronize()
    fvx.device_status()

    def kernel_of(i):
        if fp32:
            return "conv_f32"
        if algos[i] == fvx.FVX_CONV_LEAF:
            return "conv_leaf"
        return "conv_bf16_tma" if convs[i]["cin"] % 16 == 0 else "conv_bf16_tc"

    conv_kernels = [kernel_of(i) for i in range(len(convs))]
    # the roofline follows the conv kernel doing the most arithmetic
    prof_kernel = args.profile_kernel or conv_kernels[0]
    recs = EventRec()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    fvx.profile_enable(prof_kernel)
    l0 = fvx.launch_count()
    for k in range(args.steps):
        flush.fill_(float(k))  # evict L2 between steps (outside the step's events)
        hs, pairs = step(recs, coords, x, Ws)
        release(hs)
    torch.cuda.synchronize()
    launches = fvx.launch_count() - l0
    prof_ms, prof_n = fvx.profile_read()
    fvx.profile_enable(None)
    barrier(world)
    clk = clocks.stop()
    fvx.device_status()
    t = {"build": 0.0, "kmap": 0.0, "conv": 0.0}
    for cat, e0, e1 in recs.marks:
        t[cat] += e0.elapsed_time(e1) / 1e3
    t_total = max_over_ranks(sum(t.values()), world)
    K = args.steps
    value = U * K * world / t_total / 1e6
    esz = 4 if fp32 else 2
    flops_i = [2.0 * c["cin"] * c["cout"] * p for c, p in zip(convs, pairs)]
    flops = sum(flops_i)
    # algorithmic bytes of each conv: feats read once, output written once
    # (4 B fp32 / 2 B bf16), weights once, plus what locates the inputs: the
    # kernel map's (in, out) int32 pair for the pair-list kernels, the output
    # leaf's 80-byte record for the leaf-densified kernel
    bytes_i = []
    n_in = U
    for i, (c, p) in enumerate(zip(convs, pairs)):
        where = 80 * leaves_out[i] if conv_kernels[i] == "conv_leaf" else 8 * p
        bytes_i.append(n_in * c["cin"] * esz + n_out[i] * c["cout"] * ys[i].element_size()
                       + 27 * c["cin"] * c["cout"] * esz + where)
        n_in = n_out[i]
    if not args.profile_kernel and len(convs) > 1:
        prof_kernel = conv_kernels[max(range(len(convs)), key=lambda i: flops_i[i])]
    mine = [i for i in range(len(convs)) if conv_kernels[i] == prof_kernel]
    flops_p = sum(flops_i[i] for i in mine)
    alg_bytes = sum(bytes_i[i] for i in mine)
    # build + kernel map against HBM: per input row 170 B (key encode, radix
    # passes, flag scans, sidecars), per output voxel 76 B plus 8 B per pair
    # (coordinates, leaf words, mask, scans; the pair lists written once)
    bk_bytes = 170.0 * w["coords"].shape[0] + sum(76.0 * n + 8.0 * p for n, p in zip(n_out, pairs))

    # roofline of the profiled kernel (all of its launches in the timed region)
    peaks, peak_kind = measured_peaks()
    roofline = None
    if prof_n and mine:
        flops = flops_p
        sec = prof_ms / 1e3
        per_launch = prof_n / K  # launches of the kernel per step
        intensity = flops / alg_bytes
        if fp32:
            # FFMA: 152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz (max SM clock)
            peak = 152 * 128 * 2 * 2.07e9 / 1e12
            roofline = dict(bound="alu", achieved=round(flops * K / sec / 1e12, 3), peak=round(peak, 1),
                            unit="TFLOP/s", peak_source="derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz")
        elif intensity > peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9):
            peak = peaks["bf16_tflops"]
            roofline = dict(bound="tensor", achieved=round(flops * K / sec / 1e12, 2), peak=peak, unit="TFLOP/s",
                            peak_source=f"{peak_kind} (bf16_tflops, burst)")
        else:
            peak = peaks["hbm_gbs"]
            roofline = dict(bound="hbm", achieved=round(alg_bytes * K / sec / 1e9, 1), peak=peak, unit="GB/s",
                            peak_source=f"{peak_kind} (hbm_gbs)")
        roofline.update(kernel=prof_kernel, frac=round(roofline["achieved"] / roofline["peak"], 4),
                        traffic=profiled_traffic(prof_kernel, w["name"]) if len(mine) == 1 else None,
                        algorithmic_bytes=int(alg_bytes / per_launch), flops=int(flops / per_launch),
                        avg_launch_ms=round(prof_ms / prof_n, 5), launches_per_step=int(per_launch))

    # end to end through the public API with host buffers: every step copies
    # its inputs in from pinned host memory and its result back out, all inside
    # the timed region.  Steps are pipelined two deep, as a serving loop would
    # run them: each slot has its own stream (build -> kernel map -> conv ->
    # result download) and an upload stream (features and weights) that
    # overlaps the slot's build; step k's download overlaps step k+1's work.
    n_e2e = max(2, min(K, 10))
    main_s = [torch.cuda.Stream(device=dev) for _ in range(2)]
    up_s = [torch.cuda.Stream(device=dev) for _ in range(2)]
    cd_slot = [torch.empty_like(coords) for _ in range(2)]
    xd_slot = [torch.empty_like(x) for _ in range(2)]
    Wd_slot = [[torch.empty_like(t_) for t_ in Ws] for _ in range(2)]
    ys_slot = [[torch.empty_like(y_) for y_ in ys] for _ in range(2)]
    y_h = [torch.empty(ys[-1].shape, dtype=ys[-1].dtype).pin_memory() for _ in range(2)]
    conv_done = [None, None]
    up_done = [None, None]

    def upload(k):
        sl = k & 1
        us = up_s[sl]
        with torch.cuda.stream(us):
            if conv_done[sl] is not None:
                us.wait_event(conv_done[sl])  # the slot's previous step has read its inputs
            cd_slot[sl].copy_(coords_h, non_blocking=True)
            xd_slot[sl].copy_(x_h, non_blocking=True)
            for d_, h_ in zip(Wd_slot[sl], W_h):
                d_.copy_(h_, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(us)
            up_done[sl] = ev

    def compute(k):
        sl = k & 1
        ms = main_s[sl]
        with torch.cuda.stream(ms):
            ms.wait_event(up_done[sl])
            handles = []
            g = fvx.Grid.build(cd_slot[sl], offs, stream=ms)
            handles.append(g)
            src, gin = xd_slot[sl], g
            for i, c in enumerate(convs):
                gout = gin if c["stride"] == 1 else gin.coarsen(c["stride"], stream=ms)
                if gout is not gin:
                    handles.append(gout)
                km = fvx.KernelMap(gin, gout, c["stride"], stream=ms)
                handles.append(km)
                fvx.sparse_conv(gin, gout, km, src, Wd_slot[sl][i], out=ys_slot[sl][i], stream=ms)
                src, gin = ys_slot[sl][i], gout
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
    e2e = dict(value=round(U * n_e2e * world / t_e2e / 1e6, 2), unit=UNIT,
               h2d_bytes_per_step=int(coords_h.numel() * 4 + x_h.numel() * x_h.element_size()
                                      + sum(t_.numel() * t_.element_size() for t_ in W_h)),
               d2h_bytes_per_step=int(y_h[0].numel() * y_h[0].element_size()),
               steps=n_e2e, pipeline="2 steps in flight on 2 streams; step k+1's uploads overlap step k")

    out = dict(metric=METRIC, value=round(value, 2), unit=UNIT, n_gpus=world, steps=K, warmup=args.warmup,
               ms_per_step=round(t_total / K * 1e3, 4), higher_is_better=True, scaling="weak",
               vs_baseline=None, dtype="f32" if fp32 else "bf16", data="synthetic",
               config=dict(workload=w["name"], rows=int(w["coords"].shape[0]), active_voxels=U,
                           pairs=[int(p) for p in pairs],
                           convs=[f"{c['cin']}->{c['cout']} stride {c['stride']}" for c in convs],
                           batch=int(len(offs) - 1),
                           l2="flushed between steps (256 MB write outside the step events)",
                           parallelism=f"replicas x{world}"),
               components=dict(build_kmap_mvoxels_s=round(U * K / (t["build"] + t["kmap"]) / 1e6, 2),
                               conv_active_pair_tflops=round(sum(flops_i) * K / t["conv"] / 1e12, 4),
                               build_ms=round(t["build"] / K * 1e3, 4), kmap_ms=round(t["kmap"] / K * 1e3, 4),
                               conv_ms=round(t["conv"] / K * 1e3, 4), conv_kernels=conv_kernels,
                               build_kmap_hbm=dict(algorithmic_bytes=int(bk_bytes),
                                                   achieved_gbs=round(bk_bytes * K / (t["build"] + t["kmap"]) / 1e9, 1),
                                                   frac=round(bk_bytes * K / (t["build"] + t["kmap"]) / 1e9
                                                              / peaks["hbm_gbs"], 4))),
               roofline=roofline, e2e=e2e, gpu_launches=int(launches), clocks=clk)
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
            peak = 152 * 128 * 2 * 2.07e9 / 1e12
            roofline = dict(bound="alu", achieved=round(ach, 3), peak=round(peak, 1), unit="TFLOP/s",
                            peak_source="derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz")
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
    if rank != 0:
        return None
    import oracle

    oracle.build()
    w = make_workload(args.workload, args.scale)
    coords, offs, desc = oracle_sample(w, target_rows=120_000)
    cv = w["convs"][0]
    for _ in range(args.warmup):
        run_oracle_step(coords, offs, w["convs"], 1)
    times, n = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        n = run_oracle_step(coords, offs, w["convs"], 1)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = n * args.steps / tot / 1e6
    cb = dict(value=round(value, 4), unit=UNIT, cores=1, kind="oracle",
              sample=f"{desc}: build+kmap+conv of {n} voxels per step, single-threaded", host_cores=os.cpu_count())
    return dict(impl="reference", metric=METRIC, value=round(value, 4), unit=UNIT, n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(tot / args.steps * 1e3, 2), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                config=dict(workload=w["name"], sample=desc,
                            convs=[f"{c['cin']}->{c['cout']} stride {c['stride']}" for c in w["convs"]]),
                cpu_baseline=cb, e2e=dict(value=round(value, 4), unit=UNIT, h2d_bytes_per_step=0,
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

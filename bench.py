"""Benchmark of libfnorm on GB300: effective HBM GB/s (algorithmic bytes: read
x once, write y once) and the fraction of the measured HBM peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--shape N,C,H,W] [--no-extra] [--dry-run]
                    [--phases]

``--gpus N`` runs one process per GPU: launched without torchrun, the script
re-launches itself under ``torch.distributed.run`` with N processes; under a
launcher, WORLD_SIZE must equal N. ``--dry-run`` prints that plan and exits.
At least 3 warm-up steps run; the line's ``warmup`` is the number used (and
``warmup_requested`` the one asked for, when they differ).

One step is one call of the hot path over one batch of the workload. The
default workload is InstanceNorm2d forward, fp32, x[112,64,512,512] ~ N(0,1)
(7168 slices of 512x512; 7.5 GB read, 7.5 GB written). The input is larger
than L2, so no flush is needed between steps. Under torchrun each rank runs
its own copy of the workload on its own GPU (weak scaling; the slices are
independent, so there is no collective) and the time is the max over ranks.

``--impl reference`` times the CPU oracle (single-threaded, float64) on a
bounded sample of the same workload on the host cores.

Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import normalization_reduction_gb300 as fn  # noqa: E402
from normalization_reduction_gb300 import dist, inputs  # noqa: E402

METRIC = "effective HBM GB/s (min bytes/time) and % of GB300 peak per normalization config"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
L2_BYTES = 126 * 1024 * 1024

# DRAM bytes (read + write) per launch of each workload's dominant kernel from
# one ncu capture (dram__bytes_read.sum + dram__bytes_write.sum); None until
# measured for the current kernel.
NCU_TRAFFIC = {
    # the split InstanceNorm kernel: 1.073823 GB read + 1.018198 GB written for
    # 1024 slices (x[16,64,512,512]), scaled by 7 to the 7168-slice launch
    "instancenorm2d_fp32_112x64x512x512": 14644147000,
    # the eval BatchNorm kernel at full size
    "batchnorm2d_eval_fp32_128x64x126x126": 984366848,
    # both launches of a training BatchNorm step (caches flushed between them
    # by ncu, so without the apply pass's L2 reuse)
    "batchnorm2d_train_fp32_128x64x126x126": 1505662464,
    # the L2-form epilogue kernel at full size: 112.564480 MB read + 3.587328 MB
    # written (the rest of y still dirty in L2 at kernel end)
    "epilogue_fp32_128x16x14x30x30": 116151808,
}


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------ workloads
class Workload:
    name = ""
    launches = 1          # our kernel launches per step
    dtype = "f32"
    kernel = ""

    def bytes_per_step(self) -> int:
        raise NotImplementedError

    def l2_note(self) -> str:
        return "input larger than L2, no flush"

    def step(self, stream):
        raise NotImplementedError


class InstanceNormLarge(Workload):
    kernel = "in_split_kernel"

    def __init__(self, dev, shape=inputs.SHAPE_LARGE):
        self.shape = shape
        self.name = "instancenorm2d_fp32_" + "x".join(str(v) for v in shape)
        self.x = inputs.instancenorm_large(dev, shape)
        self.y = torch.empty_like(self.x)
        self.N, self.C = shape[0], shape[1]
        self.S = shape[2] * shape[3]

    def bytes_per_step(self):
        return self.x.numel() * 8

    def step(self, stream):
        fn.fnorm_instancenorm(self.x, self.y, self.N, self.C, self.S, fn.FNORM_F32, fn.FNORM_F32,
                              1e-5, None, None, stream)


class Epilogue(Workload):
    name = "epilogue_fp32_128x16x14x30x30"
    kernel = "epi_range_l2_kernel"
    graph = True   # ~30 us per step: timed as a CUDA graph of `steps` launches

    def __init__(self, dev, copies=None, want_arg=False):
        x, m = inputs.epilogue(dev)
        self.N, self.C = x.shape[0], x.shape[1]
        self.S = x[0, 0].numel()
        nbytes = x.numel() * 4
        copies = copies or max(1, -(-4 * L2_BYTES // nbytes))   # rotate >= 4x L2
        self.xs = [x] + [x.clone() for _ in range(copies - 1)]
        self.ys = [torch.empty((self.N, self.S), device=dev) for _ in range(copies)]
        # with the argmax output (int64 channel index per position)
        self.args = ([torch.empty((self.N, self.S), dtype=torch.int64, device=dev)
                      for _ in range(copies)] if want_arg else None)
        if want_arg:
            self.name = self.name + "_argmax"
        self.m = m
        self.i = 0

    def bytes_per_step(self):
        b = self.N * self.C * self.S * 4 + self.N * self.S * 4 + self.C * 4
        return b + (self.N * self.S * 8 if self.args is not None else 0)

    def l2_note(self):
        return f"{len(self.xs)} rotating input/output copies (>= 4x L2)"

    def step(self, stream):
        k = self.i % len(self.xs)
        self.i += 1
        fn.fnorm_instancenorm_epilogue(self.xs[k], self.m, self.ys[k],
                                       self.args[k] if self.args is not None else None, self.N,
                                       self.C, self.S, 1e-5, -1.0, 1.0, stream)


class BatchNorm(Workload):
    name = "batchnorm2d_train_fp32_128x64x126x126"
    kernel = "bn_stats_split_kernel+bn_apply_staged_kernel"
    launches = 2

    def __init__(self, dev):
        self.x, self.g, self.b, self.rm, self.rv = inputs.batchnorm(dev)
        self.y = torch.empty_like(self.x)
        self.N, self.C = self.x.shape[0], self.x.shape[1]
        self.S = self.x[0, 0].numel()
        nb = fn.fnorm_batchnorm_workspace_size(self.N, self.C, self.S)
        self.ws = torch.empty(nb, dtype=torch.uint8, device=dev)

    def bytes_per_step(self):
        return self.x.numel() * 8

    def step(self, stream):
        fn.fnorm_batchnorm_train(self.x, self.y, self.g, self.b, 2.0, self.rm, self.rv, 0.1, 1e-5,
                                 None, None, self.N, self.C, self.S, self.ws, self.ws.numel(),
                                 stream)


class InstanceNormWs(InstanceNormLarge):
    """fnorm_instancenorm_ws (caller workspace): few fp32 slices too long for a
    cluster take the BatchNorm-kernel route over the [1, N*C, S] view."""

    def __init__(self, dev, shape):
        super().__init__(dev, shape)
        self.name = "instancenorm2d_ws_fp32_" + "x".join(str(v) for v in shape)
        self.nb = fn.fnorm_instancenorm_workspace_size(self.N, self.C, self.S)
        self.ws = torch.empty(max(self.nb, 1), dtype=torch.uint8, device=dev)

    def step(self, stream):
        fn.fnorm_instancenorm_ws(self.x, self.y, self.N, self.C, self.S, fn.FNORM_F32,
                                 fn.FNORM_F32, 1e-5, None, None, self.ws, self.nb, stream)


class InstanceNormAffine(InstanceNormLarge):
    """InstanceNorm2d(64, affine=True) on x[112,64,512,512]."""

    def __init__(self, dev, shape=inputs.SHAPE_LARGE):
        self.shape = shape
        self.name = "instancenorm2d_affine_fp32_" + "x".join(str(v) for v in shape)
        self.x, self.g, self.b = inputs.instancenorm_affine(dev, shape)
        self.y = torch.empty_like(self.x)
        self.N, self.C = shape[0], shape[1]
        self.S = shape[2] * shape[3]

    def step(self, stream):
        fn.fnorm_instancenorm_affine(self.x, self.y, self.g, self.b, self.N, self.C, self.S,
                                     fn.FNORM_F32, fn.FNORM_F32, 1e-5, None, None, stream)


class BatchNormEval(Workload):
    """Eval-mode BatchNorm2d(64) then x*2.0 on x[128,64,126,126]."""
    name = "batchnorm2d_eval_fp32_128x64x126x126"
    kernel = "bn_eval_staged_kernel"

    def __init__(self, dev):
        self.x, self.g, self.b, self.rm, self.rv = inputs.batchnorm_eval(dev)
        self.y = torch.empty_like(self.x)
        self.N, self.C = self.x.shape[0], self.x.shape[1]
        self.S = self.x[0, 0].numel()

    def bytes_per_step(self):
        return self.x.numel() * 8

    def step(self, stream):
        fn.fnorm_batchnorm_eval(self.x, self.y, self.g, self.b, 2.0, self.rm, self.rv, 1e-5,
                                self.N, self.C, self.S, stream)


class Sweep(Workload):
    kernel = "in_*_kernel"
    dtype = "bf16"

    def __init__(self, dev, S, total=inputs.SWEEP_TOTAL):
        self.name = f"instancenorm_bf16_sweep_S{S}" + ("" if total == inputs.SWEEP_TOTAL
                                                       else f"_total{total}")
        self.x = inputs.instancenorm_sweep(S, dev, total=total)
        self.y = torch.empty_like(self.x)
        self.N, self.C, self.S = self.x.shape

    def bytes_per_step(self):
        return self.x.numel() * 4

    def step(self, stream):
        fn.fnorm_instancenorm(self.x, self.y, self.N, self.C, self.S, fn.FNORM_BF16, fn.FNORM_BF16,
                              1e-5, None, None, stream)


class Floor(Workload):
    """Reference floors for the roofline (not the library): a plain read of
    BYTES bytes (torch's sum over an fp32 tensor) or a copy (torch's copy_),
    rotating over input copies of at least 4x L2 in total when BYTES is below
    that, so every step reads HBM. The epilogue's workload reads 103 MB and
    writes 6.5 MB; its floor is about a 103 MB read."""
    kernel = "torch reference (not libfnorm)"
    launches = 0
    graph = True

    def __init__(self, dev, kind, nbytes):
        self.kind = kind
        self.name = f"floor_{kind}_{nbytes}B"
        n = max(1, nbytes // 4)
        copies = max(1, -(-4 * L2_BYTES // (n * 4)))
        self.xs = [torch.ones(n, device=dev) for _ in range(copies)]
        self.ys = [torch.empty(n, device=dev) for _ in range(copies)] if kind == "copy" else []
        self.out = torch.empty((), device=dev)
        self.n = n
        self.i = 0

    def bytes_per_step(self):
        return self.n * 4 * (2 if self.kind == "copy" else 1)

    def l2_note(self):
        return f"{len(self.xs)} rotating copies (>= 4x L2 in total)"

    def step(self, stream):
        k = self.i % len(self.xs)
        self.i += 1
        if self.kind == "copy":
            self.ys[k].copy_(self.xs[k])
        else:
            torch.sum(self.xs[k], dim=0, out=self.out)


# ------------------------------------------------------------------ timing
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.proc = None
        self.dev = dev_index

    def __enter__(self):
        try:
            ident = str(self.dev)
            try:
                u = torch.cuda.get_device_properties(self.dev).uuid
                ident = "GPU-" + str(u)
            except Exception:
                pass
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not getattr(self, "out", ""):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_info():
    w = dist.world_from_env()
    return w.size, w.rank, w.local_rank


def barrier(ws):
    dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    return dist.max_over_ranks(v, device="cuda")


def make_workload(args, dev) -> Workload:
    shape = tuple(int(v) for v in args.shape.split(",")) if args.shape else None
    if args.workload == "in_large":
        return InstanceNormLarge(dev, shape or inputs.SHAPE_LARGE)
    if args.workload == "epilogue":
        return Epilogue(dev)
    if args.workload == "epilogue_argmax":
        return Epilogue(dev, want_arg=True)
    if args.workload == "batchnorm":
        return BatchNorm(dev)
    if args.workload == "in_ws":
        return InstanceNormWs(dev, shape or inputs.SHAPE_LARGE)
    if args.workload == "in_affine":
        return InstanceNormAffine(dev, shape or inputs.SHAPE_LARGE)
    if args.workload == "bn_eval":
        return BatchNormEval(dev)
    if args.workload.startswith("floor_read:") or args.workload.startswith("floor_copy:"):
        kind, nbytes = args.workload[len("floor_"):].split(":")
        return Floor(dev, kind, int(nbytes))
    if args.workload.startswith("sweep:"):
        parts = args.workload.split(":")
        total = int(parts[2]) if len(parts) > 2 else inputs.SWEEP_TOTAL
        return Sweep(dev, int(parts[1]), total)
    raise SystemExit(f"unknown workload {args.workload}")


def time_workload(wl: Workload, steps: int, warmup: int, ws: int, sample_clocks=False):
    """Device time per step (ms) with CUDA events on the launching stream.

    Workloads whose steps take tens of microseconds (``wl.graph``) are captured
    into one CUDA graph of ``steps`` launches and replayed, so host launch
    latency does not gate the GPU; the per-step time is then the graph's time
    divided by ``steps``.
    """
    if getattr(wl, "graph", False):
        return time_graph(wl, steps, warmup, ws, sample_clocks)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        wl.step(stream)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    per = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    sampler = ClockSampler(torch.cuda.current_device()) if sample_clocks else None
    if sampler:
        sampler.__enter__()
        time.sleep(0.3)
    start.record(stream)
    for i in range(steps):
        per[i][0].record(stream)
        wl.step(stream)
        per[i][1].record(stream)
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    barrier(ws)
    if sampler:
        sampler.__exit__()
    total_ms = start.elapsed_time(end)
    step_ms = [a.elapsed_time(b) for a, b in per]
    return total_ms, step_ms, (sampler.summary() if sampler else None)


def time_graph(wl: Workload, steps: int, warmup: int, ws: int, sample_clocks=False):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warmup):          # plans, attributes and occupancy queries
            wl.step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream()
        for _ in range(steps):
            wl.step(cap)
    g.replay()                            # warm replay
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()) if sample_clocks else None
    if sampler:
        sampler.__enter__()
        time.sleep(0.3)
    start.record(stream)
    g.replay()
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    barrier(ws)
    if sampler:
        sampler.__exit__()
    total_ms = start.elapsed_time(end)
    return total_ms, [total_ms / steps] * steps, (sampler.summary() if sampler else None)


def gpu_local_cpus(dev):
    """CPUs of the NUMA node the GPU is attached to (sysfs), or None."""
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open(f"/sys/bus/pci/devices/{bus}/local_cpulist") as f:
            text = f.read().strip()
        cpus = set()
        for part in text.split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
        return cpus & os.sched_getaffinity(0) or None
    except Exception:
        return None


def e2e_instancenorm(wl: InstanceNormLarge, steps: int, chunk_slices: int = 224,
                     nstreams: int = 4):
    """Binds the process to the GPU-local CPUs (when sysfs names them) while
    the pinned buffers are allocated and used, then runs the timed loop."""
    saved = os.sched_getaffinity(0)
    local = gpu_local_cpus(wl.x.device)
    if local:
        os.sched_setaffinity(0, local)
    try:
        res = _e2e_instancenorm(wl, steps, chunk_slices, nstreams)
    finally:
        os.sched_setaffinity(0, saved)
    res["host_cpus"] = f"{len(local)} GPU-local" if local else "unbound"
    return res


def _e2e_instancenorm(wl: InstanceNormLarge, steps: int, chunk_slices: int = 224,
                      nstreams: int = 4):
    """Same metric through the C ABI with the input and output in pinned HOST
    memory: every step copies x host->device, normalises, copies y back.
    Chunks of slices go round-robin over several streams so the copies in both
    directions overlap each other and the kernel (the host link, not the GPU,
    bounds this number)."""
    NC = wl.N * wl.C
    S = wl.S
    xh = torch.empty((NC, S), dtype=torch.float32, pin_memory=True)
    yh = torch.empty((NC, S), dtype=torch.float32, pin_memory=True)
    xh.copy_(wl.x.view(NC, S)[:NC])
    dx = wl.x.view(NC, S)
    dy = wl.y.view(NC, S)
    streams = [torch.cuda.Stream() for _ in range(nstreams)]
    chunks = [(a, min(NC, a + chunk_slices)) for a in range(0, NC, chunk_slices)]

    def one_step():
        for i, (a, b) in enumerate(chunks):
            s = streams[i % len(streams)]
            with torch.cuda.stream(s):
                dx[a:b].copy_(xh[a:b], non_blocking=True)
                fn.fnorm_instancenorm(dx[a:b], dy[a:b], 1, b - a, S, fn.FNORM_F32, fn.FNORM_F32,
                                      1e-5, None, None, s)
                yh[a:b].copy_(dy[a:b], non_blocking=True)

    one_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        one_step()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    nbytes = NC * S * 4
    return {"value": round(wl.bytes_per_step() / dt / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(dt * 1e3, 3), "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": nbytes,
            "pipeline": f"{len(chunks)} chunks over {nstreams} streams"}


def cpu_baseline(x_dev: torch.Tensor, S: int, budget_s: float = 10.0, batch: int = 256):
    """The oracle on a bounded sample of the workload's slices (host cores)."""
    import oracle
    orc = oracle.get()
    NC = x_dev.numel() // S
    xv = x_dev.view(NC, S)
    done = 0
    elapsed = 0.0
    while done < NC and elapsed < budget_s:
        b = min(batch, NC - done)
        xs = xv[done:done + b].cpu().numpy()
        t0 = time.perf_counter()
        orc.instancenorm(xs)
        elapsed += time.perf_counter() - t0
        done += b
    nbytes = done * S * 8
    return {"value": round(nbytes / elapsed / 1e9, 3), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{done} of {NC} slices ({done * S} elements), float64 single-threaded"}


PHASE_NAMES = ["statistics", "exchange", "coefficients", "kept_output", "l2_output"]


def epilogue_phases():
    """Per-phase times of the L2-form epilogue kernel's last launch, from the
    instrumented library (libfnorm_phases.so): median duration of each phase
    over the CTAs, and each phase's end relative to the earliest CTA start."""
    import ctypes
    import numpy as np
    lib = fn.lib()
    n_ctas, n_ph = 2048, len(PHASE_NAMES) + 1
    buf = (ctypes.c_ulonglong * (n_ctas * n_ph))()
    lib.fnorm_phase_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.fnorm_phase_trace_read.restype = ctypes.c_int
    if lib.fnorm_phase_trace_read(ctypes.addressof(buf), n_ctas * n_ph) != 0:
        return {"error": "trace read failed"}
    t = np.frombuffer(buf, dtype=np.uint64).astype(np.int64).reshape(n_ctas, n_ph)
    t = t[(t > 0).all(axis=1)]
    if not len(t):
        return {"error": "no stamps (not the L2-form kernel?)"}
    d = np.diff(t, axis=1)
    t0 = t[:, 0].min()
    out = {"ctas": int(len(t)), "unit": "us"}
    for j, name in enumerate(PHASE_NAMES):
        end = t[:, j + 1] - t0
        out[name] = {"median": round(float(np.median(d[:, j])) / 1e3, 3),
                     "end_min": round(float(end.min()) / 1e3, 3),
                     "end_median": round(float(np.median(end)) / 1e3, 3),
                     "end_max": round(float(end.max()) / 1e3, 3)}
    return out


def run_ours(args):
    ws, rank, local = dist_info()
    if args.phases:
        # the instrumented library: per-phase stamps (timing is perturbed a little)
        from normalization_reduction_gb300 import build as nbuild
        fn.LIBRARY = nbuild.build(phases=True)
    if ws > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    peak, peak_kind = peak_hbm()

    wl = make_workload(args, dev)
    total_ms, step_ms, clocks = time_workload(wl, args.steps, args.warmup, ws, sample_clocks=True)
    total_ms = max_over_ranks(total_ms, ws)
    ms = total_ms / args.steps
    nbytes = wl.bytes_per_step()
    value = nbytes * ws / (ms * 1e-3) / 1e9
    kernel_ms = statistics.mean(step_ms)
    achieved = nbytes / (kernel_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, generated on device)",
        "config": {"workload": wl.name, "shape": list(getattr(wl, "shape", ())), "eps": 1e-5,
                   "bytes_per_step": nbytes, "l2": wl.l2_note(),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "pct_of_peak": round(100 * value / ws / peak, 2),
        "pct_of_nominal": round(100 * value / ws / NOMINAL_HBM_GBS, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": NCU_TRAFFIC.get(wl.name), "peak_source": peak_kind,
                     "kernel": wl.kernel},
        "gpu_launches": wl.launches * args.steps,
        "clocks": clocks,
    }
    if args.warmup_requested != args.warmup:
        res["warmup_requested"] = args.warmup_requested
    if args.phases:
        res["phases"] = epilogue_phases() if isinstance(wl, Epilogue) else {
            "error": "phase stamps exist for the epilogue workload only"}
        res["phases"]["library"] = "libfnorm_phases.so (instrumented)"
    res["dtype"] = wl.dtype
    if rank == 0 and not args.no_extra and isinstance(wl, InstanceNormLarge):
        res["e2e"] = e2e_instancenorm(wl, max(2, min(args.steps, 5)))
        res["cpu_baseline"] = cpu_baseline(wl.x, wl.S)
    del wl
    torch.cuda.empty_cache()
    if not args.no_extra and args.workload == "in_large" and args.shape is None:
        res["per_config"] = other_configs(dev, ws, peak)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def other_configs(dev, ws, peak):
    """The other workloads, same timing rules (reported alongside)."""
    out = {}
    cases = [("epilogue", lambda: Epilogue(dev), 200, 20),
             ("epilogue_argmax", lambda: Epilogue(dev, want_arg=True), 200, 20),
             ("batchnorm", lambda: BatchNorm(dev), 20, 5),
             ("batchnorm_eval", lambda: BatchNormEval(dev), 20, 5),
             ("instancenorm_affine", lambda: InstanceNormAffine(dev), 20, 5)]
    cases += [(f"sweep_S{S}", (lambda S=S: Sweep(dev, S)), 20, 5) for S in inputs.SWEEP_S]
    for key, make, steps, warm in cases:
        wl = make()
        total_ms, step_ms, _ = time_workload(wl, steps, warm, ws)
        ms = max_over_ranks(total_ms, ws) / steps
        gbs = wl.bytes_per_step() / (ms * 1e-3) / 1e9
        out[key] = {"workload": wl.name, "ms_per_step": round(ms, 4), "GB/s": round(gbs, 1),
                    "pct_of_peak": round(100 * gbs / peak, 2), "launches_per_step": wl.launches}
        if isinstance(wl, BatchNorm):
            out[key]["GB/s_two_read_basis"] = round(gbs * 1.5, 1)
        del wl
        torch.cuda.empty_cache()
    return out


def run_reference(args):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    import numpy as np
    import oracle
    orc = oracle.get()
    shape = inputs.SHAPE_LARGE
    S = shape[2] * shape[3]
    NC = shape[0] * shape[1]
    sample = 24   # slices per step: a bounded sample of the workload
    x = inputs.normal((sample, S), inputs.SEED_LARGE, "cpu").numpy()
    for _ in range(args.warmup):
        orc.instancenorm(x)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        orc.instancenorm(x)
        times.append(time.perf_counter() - t0)
    per = statistics.mean(times)
    gbs = sample * S * 8 / per / 1e9
    res = {"impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
           "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1))",
           "config": {"workload": "instancenorm2d_fp32_112x64x512x512", "shape": list(shape),
                      "sample_slices_per_step": sample, "of_slices": NC},
           "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                            "sample": f"{sample} of {NC} slices per step, float64 single-threaded"},
           "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    if args.warmup_requested != args.warmup:
        res["warmup_requested"] = args.warmup_requested
    print(json.dumps(res), flush=True)
    del np


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true",
                    help="skip e2e, cpu baseline and the other workloads")
    ap.add_argument("--workload", default="in_large",
                    help="in_large | in_ws | in_affine | epilogue | epilogue_argmax | batchnorm | "
                         "bn_eval | "
                         "sweep:S[:TOTAL] "
                         "(S a power of 4, 256..4^10; TOTAL elements, default 2^30) | "
                         "floor_read:BYTES | floor_copy:BYTES (torch reference floors)")
    ap.add_argument("--shape", default=None,
                    help="N,C,H,W for in_large (e.g. a smaller case for ncu)")
    ap.add_argument("--phases", action="store_true",
                    help="epilogue workload: time it with the instrumented library and add "
                         "the per-phase breakdown of the last launch")
    ap.add_argument("--dry-run", action="store_true",
                    help="print how the run would start (one line of JSON) and exit")
    args = ap.parse_args()
    plan = dist.launch_plan(args.gpus, os.environ, sys.argv[1:], os.path.abspath(__file__),
                            sys.executable)
    if args.dry_run:
        print(json.dumps(plan), flush=True)
        return 0 if plan["action"] != "error" else 2
    if plan["action"] == "error":
        print(f"bench.py: {plan['why']}", file=sys.stderr, flush=True)
        return 2
    if plan["action"] == "relaunch":
        # one process per GPU under torch.distributed.run; rank 0 prints the line
        return subprocess.run(plan["cmd"]).returncode
    # at least 3 untimed warm-up steps; the line reports the number used
    args.warmup_requested = args.warmup
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())

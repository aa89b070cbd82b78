#!/usr/bin/env python3
"""Benchmark of the attention forward pass on GB300 -- one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload suite|NAME] [--impl ours|reference]

A step is one fa_fwd call over the whole workload (every query row of every head and batch).
By default (``--workload suite``) the run times five workloads one after another: the largest
one, B=1 Hq=32 Hkv=8 S=16384 D=128 bf16 causal, whose figures are the top level of the line,
then the 4096-token GQA causal one, the non-causal fp16 one (S=2000, large logits), the D=64
causal one and the smallest one; ``per_config`` holds each workload's value, step time,
roofline (fractions of the burst and of the sustained peak), clocks and CPU-oracle baseline.
``value`` is attention TFLOP/s (4*B*Hq*Sq*Sk*D, halved when causal) over the K timed steps,
timed with CUDA events on the launching stream with the inputs resident in HBM; the L2 is
flushed (a 256 MiB write) between timed steps, outside the events.  ``e2e`` is the same
metric through the host-memory entry point (fa_fwd_host) on pinned host buffers: every step
copies q, k, v host->device, runs the attention and copies o and lse back, all inside the
events, with the copies of one chunk of heads overlapped with the kernels of another
(``--chunks`` sets the pipeline depth).  Two calls are kept in flight (alternate steps use their
own staging buffers, host outputs and stream, so one step's uploads overlap the previous step's
kernels and downloads; 2 chunks per call unless ``--chunks`` says otherwise);
``serial_ms_per_step`` is the same with one call at a time (the library's default depth).

``roofline`` compares the kernel against the measured dense bf16 tensor peak of the pool's
GB300s (MEASURED_PEAKS.json when present, else the fallback figure, as stated in the line).
``cpu_baseline`` times the float64 CPU oracle on a bounded sample of the same workload's
query rows, on all host cores.

``--impl reference`` times that oracle instead (the reference arm: there is no other
implementation of these pages to run): each step evaluates a bounded sample of query rows of
the headline workload.

``--op gemm | gemm_gelu | softmax`` measures the standalone building blocks instead of the
attention call (same JSON fields): the tiled matrix product (bf16, M = N = K = 8192 by
default; ``gemm_gelu`` adds the fused bias + tanh-GELU epilogue), against the tensor roofline,
and the row softmax (fp32, 65536 x 4096 by default), against the HBM roofline.

Multi-GPU (torchrun, one process per GPU): every rank runs its own replica of the workload
(independent inputs, no collective on the data path); timings are max-reduced across ranks
and ``value`` counts the work of all ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s at 1 GB300 and % of dense BF16 tensor peak (causal / non-causal)"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
E2E_INFLIGHT_CHUNKS = 2      # fa_fwd_host pipeline depth per call when two calls are in flight
PROFILE_GLOB = os.path.join(ROOT, "profiles", "*.md")
# The default run: the largest single-GPU workload first (the headline of the line), then the
# other benchmark workloads -- the 4096-token GQA causal one, the non-causal fp16 one with
# large logits and a ragged tail, the D = 64 causal one and the smallest one.
# The five benchmark configurations, the largest first (the headline), then the two head-dim-256
# workloads of the one-query-tile kernel.
SUITE = ("gqa_causal_b1_h32kv8_s16384", "gqa_causal_b2_h32kv8_s4096", "mha_fp16_b8_h16_s2000_std2",
         "mha_causal_b4_h16_s1024_d64", "mha_b1_h2_s128_d64",
         "gqa_causal_b2_h32kv8_s4096_d256", "mha_b4_h16_s2048_d256")
TARGET_FRAC = 0.60    # of the dense bf16 peak, stated for the D = 128 workloads


# ----------------------------------------------------------------------------- helpers
# The sources each timed kernel is built from: its own translation unit plus the shared
# device headers and the host code that encodes its tensor maps and launch shape.
COMMON_SOURCES = ("ptx.cuh", "watchdog.cuh", "fa_internal.h", "fa_api.cpp")
KERNEL_SOURCES = {
    "fa::fa_fwd_kernel": ("fa_fwd_sm103.cu", "schedule.h"),
    "fa::fa_fwd1_kernel": ("fa_fwd1_sm103.cu", "schedule.h"),
    "fa::gemm::gemm_kernel": ("gemm_sm103.cu",),
    "fa::sm::softmax_regs_kernel": ("softmax_sm103.cu",),
}


def strip_comments(src: str) -> str:
    """C/C++ source without // and /* */ comments and without blank lines (string and
    character literals are kept as they are), so that editing a comment does not count as a
    change of the code."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            while i < n and src[i] != "\n":
                i += 1
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash(kernel: str) -> str:
    """sha256 of the sources `kernel` is built from, comments removed: ties an ncu traffic
    figure to the code it measured (a change to another kernel leaves it valid)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "programming_flashattention_fwd_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel] + COMMON_SOURCES):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def attention_kernel(w, kernel: int) -> str:
    """The kernel fa_fwd_select runs for this workload and variant (0 = automatic)."""
    k = kernel or (2 if w.D == 256 else 1)
    return "fa::fa_fwd1_kernel" if k >= 2 else "fa::fa_fwd_kernel"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, None, "fallback"


def measured_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes from a committed ncu summary of `kernel` on this workload and
    this exact kernel source (lines 'kernel: K', 'workload: W', 'kernel_source_sha: H' and
    'traffic_bytes_per_launch: N'), else None."""
    want = kernel_source_hash(kernel)
    for p in sorted(glob.glob(PROFILE_GLOB)):
        lines = [ln.strip() for ln in open(p).read().splitlines()]
        if (f"workload: {workload}" not in lines or f"kernel_source_sha: {want}" not in lines
                or f"kernel: {kernel}" not in lines):
            continue
        for line in lines:
            if line.startswith("traffic_bytes_per_launch:"):
                try:
                    return float(line.split(":", 1)[1])
                except ValueError:
                    return None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in a background process."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self._th = threading.Thread(target=self._read, daemon=True)
        self._th.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        """Ends sampling; window() then summarises any interval of the run."""
        if self.proc is None:
            return
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def window(self, t0, t1):
        """Median SM clock, maximum clock and throttle reasons seen in [t0, t1] (or the samples
        nearest to it when the interval is shorter than the sampling period)."""
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 - 0.06 <= r[0] <= t1 + 0.06]
        where = "during timed region"
        if not inside and rows:
            inside = sorted(rows, key=lambda r: abs(r[0] - t1))[:3]
            where = "nearest samples to the timed region (region shorter than the sampling period)"
        if not inside:
            return None
        sm = sorted(float(r[1][2]) for r in inside if r[1][2].replace(".", "").isdigit())
        mx = [float(r[1][3]) for r in inside if r[1][3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[1][6 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "where": where}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """Max of a float over all ranks (identity for one process)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle
def oracle_row_flops(w, rows) -> float:
    """4 * |allowed keys| * D floating-point operations per evaluated query row."""
    i = rows[:, 2]
    n = (i + 1).clip(max=w.Sk) if w.causal else i * 0 + w.Sk
    return float(4.0 * n.sum() * w.D)


def time_oracle(w, q, k, v, target_s: float, seed: int):
    """Time the oracle on a seeded row sample sized to take about target_s seconds."""
    import numpy as np
    import oracle
    from programming_flashattention_fwd_gb300.inputs import sample_rows
    orc = oracle.load()
    cores = orc.max_threads()
    probe = sample_rows(w, n=max(cores * 4, 64), seed=seed, edge=False)
    t0 = time.perf_counter()
    orc.rows(q, k, v, w.is_fp16, w.causal, w.softmax_scale, probe)
    dt = max(time.perf_counter() - t0, 1e-6)
    n = int(min(w.B * w.Hq * w.Sq, max(len(probe), len(probe) * target_s / dt)))
    rows = sample_rows(w, n=n, seed=seed + 1, edge=False)
    t0 = time.perf_counter()
    orc.rows(q, k, v, w.is_fp16, w.causal, w.softmax_scale, rows)
    dt = time.perf_counter() - t0
    flops = oracle_row_flops(w, rows)
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} seeded query rows of {w.name} (all heads/batches), "
                      f"float64 C oracle with OpenMP, {dt:.1f} s",
            "rows": int(len(rows)), "seconds": round(dt, 3), "rows_per_s": round(len(rows) / dt, 1),
            "float64_gflops": round(flops / dt / 1e9, 2),
            "full_workload_s_extrapolated": round(w.flops() / (flops / dt), 2)}


def run_reference(args, w, world, rank):
    """Reference arm: the float64 oracle, each step a bounded sample of query rows."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from programming_flashattention_fwd_gb300.inputs import make_qkv, sample_rows
    q, k, v = make_qkv(w)
    orc = oracle.load()
    cores = orc.max_threads()
    # size the per-step sample so that warmup + steps take about args.ref_seconds in total
    probe = sample_rows(w, n=max(cores * 4, 64), seed=99, edge=False)
    t0 = time.perf_counter()
    orc.rows(q, k, v, w.is_fp16, w.causal, w.softmax_scale, probe)
    dt = max(time.perf_counter() - t0, 1e-6)
    per_step_s = args.ref_seconds / max(1, args.steps + args.warmup)
    n = int(min(w.B * w.Hq * w.Sq, max(len(probe), len(probe) * per_step_s / dt)))
    flops_total, t_total = 0.0, 0.0
    for s in range(args.warmup + args.steps):
        rows = sample_rows(w, n=n, seed=1000 + s, edge=False)
        t0 = time.perf_counter()
        orc.rows(q, k, v, w.is_fp16, w.causal, w.softmax_scale, rows)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            flops_total += oracle_row_flops(w, rows)
            t_total += dt
    value = flops_total / t_total / 1e12
    sample = f"{n} seeded query rows of {w.name} per step, float64 C oracle with OpenMP"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def workload_config(w, args):
    return {"workload": w.name, "kernel": getattr(args, "kernel", 0), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
            "dtype": w.dtype, "causal": w.causal, "scale": w.softmax_scale, "seed": w.seed,
            "l2": "flushed between timed steps (256 MiB write)",
            "parallelism": "replicas" if args.gpus > 1 else "single GPU"}


# ----------------------------------------------------------------------------- GPU arm
def time_device(args, w, world, rank, dev, fn):
    """Device-timed calls of `fn` on workload `w` (inputs resident in HBM): W warm-up calls, then K
    calls each bracketed by CUDA events on the launching stream with a 256 MiB L2 flush between
    them (outside the events), then up to 50 calls back to back (warm L2, for reference).
    Returns the timing record and the host/device tensors for the end-to-end leg."""
    import numpy as np
    import torch
    from programming_flashattention_fwd_gb300 import binding
    from programming_flashattention_fwd_gb300.inputs import make_qkv

    wr = w.with_(seed=w.seed + 7919 * rank) if rank else w     # independent replica per rank
    q_h, k_h, v_h = make_qkv(wr)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        fn(q, k, v, o, lse, w.causal, w.softmax_scale)
    torch.cuda.synchronize(dev)
    st, word = binding.fa_device_status()
    if st != 0:
        raise RuntimeError(f"device watchdog fired during warm-up of {w.name} (word {word:#x})")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for s in range(args.steps):
        flush.zero_()
        starts[s].record(stream)
        fn(q, k, v, o, lse, w.causal, w.softmax_scale)
        ends[s].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    barrier(world)
    times = [a.elapsed_time(b) * 1e-3 for a, b in zip(starts, ends)]
    t_step = max_over_ranks(sum(times) / len(times), world)
    st, word = binding.fa_device_status()
    if st != 0:
        raise RuntimeError(f"device watchdog fired during the timed steps of {w.name} (word {word:#x})")

    # the same calls back to back without the L2 flush (warm L2), for reference only
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_warm = min(args.steps, 50)
    w0.record(stream)
    for _ in range(n_warm):
        fn(q, k, v, o, lse, w.causal, w.softmax_scale)
    w1.record(stream)
    torch.cuda.synchronize(dev)
    t_warm = max_over_ranks(w0.elapsed_time(w1) * 1e-3 / n_warm, world)
    rec = {"t_step": t_step, "times": times, "t_warm": t_warm, "n_warm": n_warm, "window": (t0, t1)}
    return rec, (q_h, k_h, v_h), (q, k, v, o, lse)


def roofline_record(w, args, t_step):
    """Achieved TFLOP/s of the attention kernel against the measured dense bf16 peaks: `frac` is
    of the burst figure (the kernel is timed alone), `frac_sustained` of the sustained one."""
    peak, peak_sus, peak_src = measured_peaks()
    achieved = w.flops() / t_step / 1e12
    kname = attention_kernel(w, args.kernel)
    rec = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
           "frac": achieved / peak, "traffic": ncu_traffic(w.name, kname),
           "peak_source": f"{peak_src} dense bf16 (burst)" + (f"; sustained {peak_sus}" if peak_sus else ""),
           "kernel": kname}
    if peak_sus:
        rec["peak_sustained"] = peak_sus
        rec["frac_sustained"] = achieved / peak_sus
    return rec


def timing_record(rec, w, world):
    import numpy as np
    times, t_warm = rec["times"], rec["t_warm"]
    return {"ms_mean": rec["t_step"] * 1e3, "ms_median": float(np.median(times)) * 1e3,
            "ms_min": min(times) * 1e3, "ms_max": max(times) * 1e3,
            "warm_l2_ms_per_step": t_warm * 1e3, "warm_l2_value": w.flops() * world / t_warm / 1e12,
            "note": "value uses ms_mean over L2-flushed calls (rank max); the warm figure times "
                    f"{rec['n_warm']} calls back to back without the flush"}


def time_e2e(args, w, world, dev, fn, host, devt):
    """End to end through the host-memory entry point (fa_fwd_host): pinned host q, k, v in,
    o and lse back, copies inside the events; two calls in flight and one at a time."""
    import torch
    from programming_flashattention_fwd_gb300 import binding
    q_h, k_h, v_h = host
    q, k, v, o, lse = devt
    stream = torch.cuda.current_stream(dev)
    q_p, k_p, v_p = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    o_p = torch.empty(q_h.shape, dtype=q_h.dtype).pin_memory()
    l_p = torch.empty(q_h.shape[:3], dtype=torch.float32).pin_memory()
    q2, k2, v2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    o2 = torch.empty_like(o)
    l2 = torch.empty_like(lse)

    # pipeline depth of fa_fwd_host: one call at a time takes the library's default (4 chunks);
    # with two calls in flight the neighbouring call already fills the link, and 2 chunks per
    # call measured best (456 against 430 TFLOP/s with 4 on the 4096-token workload)
    chunks_serial = args.chunks
    chunks_inflight = args.chunks if args.chunks else E2E_INFLIGHT_CHUNKS

    def e2e_step(bufs=(q2, k2, v2, o2, l2), outs=(o_p, l_p), st=stream, chunks=None):
        qd, kd, vd, od, ld = bufs
        oh, lh = outs
        if args.kernel:   # an explicit variant: copies in, the kernel, copies back, one after another
            with torch.cuda.stream(st):
                qd.copy_(q_p, non_blocking=True)
                kd.copy_(k_p, non_blocking=True)
                vd.copy_(v_p, non_blocking=True)
                fn(qd, kd, vd, od, ld, w.causal, w.softmax_scale)
                oh.copy_(od, non_blocking=True)
                lh.copy_(ld, non_blocking=True)
        else:             # the host-memory entry point: copies and kernels overlapped chunk by chunk
            binding.fa_fwd_host(q_p, k_p, v_p, oh, lh, qd, kd, vd, od, ld, w.causal, w.softmax_scale,
                                chunks=chunks_serial if chunks is None else chunks, stream=st)

    def timed(run_steps):
        torch.cuda.synchronize(dev)
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run_steps()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return max_over_ranks(a.elapsed_time(b) * 1e-3 / args.steps, world)

    # one call at a time (each step's copies, kernels and copies back before the next step)
    for _ in range(max(1, args.warmup)):
        e2e_step()
    t_serial = timed(lambda: [e2e_step() for _ in range(args.steps)])
    assert torch.equal(o_p, o.cpu()) and torch.equal(l_p, lse.cpu()), "e2e result differs from the device run"

    # two calls in flight: alternate steps use their own staging buffers, host outputs and stream,
    # so one step's uploads overlap the previous step's kernels and downloads
    q3, k3, v3, o3 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(o)
    l3 = torch.empty_like(lse)
    o_p2 = torch.empty(q_h.shape, dtype=q_h.dtype).pin_memory()
    l_p2 = torch.empty(q_h.shape[:3], dtype=torch.float32).pin_memory()
    side = torch.cuda.Stream(dev)
    sets = [((q2, k2, v2, o2, l2), (o_p, l_p), stream), ((q3, k3, v3, o3, l3), (o_p2, l_p2), side)]

    def pipelined():
        ev = torch.cuda.Event()
        ev.record(stream)
        side.wait_event(ev)
        for i in range(args.steps):
            bufs, outs, st = sets[i % 2]
            e2e_step(bufs, outs, st, chunks_inflight)
        stream.wait_stream(side)

    for i in range(max(2, args.warmup)):
        e2e_step(*sets[i % 2], chunks_inflight)
    t_e2e = timed(pipelined)
    for oh, lh in ((o_p, l_p), (o_p2, l_p2)):
        assert torch.equal(oh, o.cpu()) and torch.equal(lh, lse.cpu()), "e2e result differs from the device run"
    h2d = (q_h.numel() + k_h.numel() + v_h.numel()) * q_h.element_size()
    d2h = o_p.numel() * o_p.element_size() + l_p.numel() * 4
    flops = w.flops()
    return {"value": flops * world / t_e2e / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
            "calls_in_flight": 2, "chunks_per_call": chunks_inflight or 4,
            "serial_chunks_per_call": chunks_serial or 4, "serial_ms_per_step": t_serial * 1e3,
            "serial_value": flops * world / t_serial / 1e12,
            "api": "fa_fwd_host" if not args.kernel else "torch copies + fa_fwd_select"}


def run_ours(args, workloads, world, rank, local):
    """Times every workload in `workloads` on the device; the first is the headline of the JSON
    line (its value, config, roofline, e2e and cpu_baseline at the top level) and every one,
    the headline included, gets an entry in `per_config`."""
    import torch
    from programming_flashattention_fwd_gb300 import binding

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.load_library()
    sampler = ClockSampler(local) if (rank == 0 and not args.no_clocks) else None
    if sampler:
        sampler.start()

    results = []
    e2e = None
    for i, w in enumerate(workloads):
        if args.kernel:
            fn = lambda q_, k_, v_, o_, l_, c_, s_: binding.fa_fwd_select(q_, k_, v_, o_, l_, c_, s_, args.kernel)
        else:
            fn = binding.fa_fwd_fp16 if w.is_fp16 else binding.fa_fwd
        rec, host, devt = time_device(args, w, world, rank, dev, fn)
        if i == 0:
            e2e = time_e2e(args, w, world, dev, fn, host, devt)
        results.append((w, rec, host))
        del devt
        torch.cuda.empty_cache()
    if sampler:
        sampler.stop()
        time.sleep(0.05)
    if rank != 0:
        return

    per_config = {}
    for i, (w, rec, host) in enumerate(results):
        rec["clocks"] = sampler.window(*rec["window"]) if sampler else None
        entry = {"value": w.flops() * world / rec["t_step"] / 1e12, "unit": UNIT,
                 "ms_per_step": rec["t_step"] * 1e3, "config": workload_config(w, args),
                 "roofline": roofline_record(w, args, rec["t_step"]), "clocks": rec["clocks"],
                 "timing": timing_record(rec, w, world), "gpu_launches": args.steps,
                 "target_frac": TARGET_FRAC if w.D == 128 else None}
        if not args.no_cpu_baseline and world == 1:   # the oracle baseline is timed at N = 1 only
            budget = args.cpu_seconds if i == 0 else args.cpu_seconds_per_config
            entry["cpu_baseline"] = time_oracle(w, *host, budget, seed=w.seed + 100)
        per_config[w.name] = entry

    w, rec, _ = results[0]
    head = per_config[w.name]
    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": head["config"],
        "e2e": e2e,
        "gpu_launches": args.steps,
        "timing": head["timing"],
        "roofline": head["roofline"],
        "clocks": head["clocks"],
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if len(results) > 1:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)


def run_op(args, world, rank, local):
    """Standalone building blocks: tiled matrix product (+ fused epilogue) or row softmax."""
    import numpy as np
    import torch
    import oracle
    from programming_flashattention_fwd_gb300 import binding

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    binding.load_library()
    g = torch.Generator().manual_seed(1234 + 7919 * rank)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    if args.op in ("gemm", "gemm_gelu"):
        M, N, K = args.M, args.N, args.K
        epi = 2 if args.op == "gemm_gelu" else 0
        a_h = torch.randn((M, K), generator=g).to(torch.bfloat16)
        b_h = torch.randn((K, N), generator=g).to(torch.bfloat16)
        bias_h = torch.randn((N,), generator=g)
        a, b, bias = a_h.to(dev), b_h.to(dev), bias_h.to(dev)
        c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        call = lambda: binding.gemm(a, b, bias if epi else None, epi, False, c)
        work = 2.0 * M * N * K
        name = f"{args.op}_bf16_{M}x{N}x{K}"
        metric, unit, bound = ("matrix product TFLOP/s" + (" (bias + tanh-GELU epilogue)" if epi else ""),
                               "TFLOP/s", "tensor")
        scale = 1e12
        cfg = {"workload": name, "M": M, "N": N, "K": K, "dtype": "bf16", "out": "bf16", "epilogue": epi}
        h2d = (a_h.numel() + b_h.numel()) * 2 + (bias_h.numel() * 4 if epi else 0)
        d2h = c.numel() * 2
    else:
        R, C = args.rows, args.cols
        sdt = torch.bfloat16 if args.softmax_dtype == "bf16" else torch.float32
        esz = 2 if args.softmax_dtype == "bf16" else 4
        x_h = (torch.randn((R, C), generator=g) * 4.0).to(sdt)
        x = x_h.to(dev)
        y = torch.empty_like(x)
        call = lambda: binding.softmax_rows(x, y)
        work = 2.0 * R * C * esz
        name = f"softmax_{args.softmax_dtype}_{R}x{C}"
        metric, unit, bound = "row softmax GB/s (bytes read + written)", "GB/s", "hbm"
        scale = 1e9
        cfg = {"workload": name, "rows": R, "cols": C, "dtype": args.softmax_dtype}
        h2d, d2h = x_h.numel() * esz, x_h.numel() * esz

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local) if (rank == 0 and not args.no_clocks) else None
    if sampler:
        sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = time.time()
    for s_ in range(args.steps):
        flush.zero_()
        starts[s_].record(stream)
        call()
        ends[s_].record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    barrier(world)
    clocks = None
    if sampler:
        sampler.stop()
        clocks = sampler.window(t_start, t_end)
    t_step = max_over_ranks(sum(a_.elapsed_time(b_) * 1e-3 for a_, b_ in zip(starts, ends)) / args.steps, world)
    st, word = binding.fa_device_status()
    if st != 0:
        raise RuntimeError(f"device watchdog fired (word {word:#x})")

    # end to end: pinned host inputs in, result out, inside the events
    if args.op in ("gemm", "gemm_gelu"):
        a_p, b_p, bias_p = a_h.pin_memory(), b_h.pin_memory(), bias_h.pin_memory()
        c_p = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()

        def e2e():
            a.copy_(a_p, non_blocking=True)
            b.copy_(b_p, non_blocking=True)
            if epi:
                bias.copy_(bias_p, non_blocking=True)
            call()
            c_p.copy_(c, non_blocking=True)
    else:
        x_p = x_h.pin_memory()
        y_p = torch.empty_like(x_h).pin_memory()

        def e2e():
            x.copy_(x_p, non_blocking=True)
            call()
            y_p.copy_(y, non_blocking=True)
    for _ in range(max(1, args.warmup)):
        e2e()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_e2e = max_over_ranks(e0.elapsed_time(e1) * 1e-3 / args.steps, world)
    if rank != 0:
        return

    kname = "fa::gemm::gemm_kernel" if bound == "tensor" else "fa::sm::softmax_regs_kernel"
    if bound == "tensor":
        peak, _, src = measured_peaks()
        peak_unit = "TFLOP/s"
    else:
        peak, src = measured_hbm()
        peak_unit = "GB/s"
    achieved = work / t_step / scale
    orc = oracle.load()
    t0 = time.perf_counter()
    if args.no_cpu_baseline:
        cpu_work, sample = None, None
    elif args.op in ("gemm", "gemm_gelu"):
        rng = np.random.default_rng(5)
        n_ent = max(64, int(4e8 / K / 8))   # sized for a few seconds of float64 work on the host
        ent = np.stack([rng.integers(0, M, n_ent), rng.integers(0, N, n_ent)], 1)
        orc.gemm_entries(a_h, b_h, False, ent, bias_h if epi else None, epi)
        cpu_work, sample = 2.0 * K * n_ent, f"{n_ent} seeded output entries of {name}, float64 C oracle"
    else:
        ids = np.random.default_rng(5).integers(0, R, 512)
        orc.softmax_rows(x_h, ids)
        cpu_work, sample = 2.0 * len(ids) * C * esz, f"{len(ids)} seeded rows of {name}, float64 C oracle"
    dt = time.perf_counter() - t0
    line = {
        "metric": metric, "value": work * world / t_step / scale, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": cfg["dtype"], "data": "synthetic",
        "config": dict(cfg, l2="flushed between timed steps (256 MiB write)",
                       parallelism="replicas" if world > 1 else "single GPU"),
        "e2e": {"value": work * world / t_e2e / scale, "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3},
        "gpu_launches": args.steps,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": peak_unit,
                     "frac": achieved / peak, "traffic": ncu_traffic(name, kname),
                     "peak_source": f"{src}" + (" dense bf16 (burst)" if bound == "tensor" else " HBM copy"),
                     "kernel": kname},
        "clocks": clocks,
    }
    if cpu_work is not None:
        line["cpu_baseline"] = {"value": cpu_work / dt / scale, "unit": unit, "cores": orc.max_threads(),
                                "kind": "oracle", "sample": sample + f", {dt:.1f} s"}
    print(json.dumps(line), flush=True)


def main():
    from programming_flashattention_fwd_gb300.inputs import ALL_WORKLOADS as WORKLOADS
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="suite", choices=["suite"] + sorted(WORKLOADS),
                    help="one workload, or 'suite': the headline (the largest, 16384-token GQA causal) "
                         "followed by the other four benchmark workloads, each in per_config")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle CPU-baseline budget (headline)")
    ap.add_argument("--cpu-seconds-per-config", type=float, default=4.0,
                    help="oracle CPU-baseline budget of each other workload of the suite")
    ap.add_argument("--ref-seconds", type=float, default=90.0, help="reference-arm total budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--kernel", type=int, default=0, choices=[0, 1, 2, 3],
                    help="attention kernel variant: 0 automatic, 1 two tiles / 128-key steps, "
                         "2 one tile / 64-key steps, 3 one tile / 128-key steps (D 128)")
    ap.add_argument("--chunks", type=int, default=0,
                    help="pipeline depth of the host-memory (e2e) call; 0 = the library's default one call "
                         "at a time and 2 per call with two calls in flight")
    ap.add_argument("--op", default="attention", choices=["attention", "gemm", "gemm_gelu", "softmax"])
    ap.add_argument("--M", type=int, default=8192)
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--K", type=int, default=8192)
    ap.add_argument("--rows", type=int, default=65536)
    ap.add_argument("--cols", type=int, default=4096)
    ap.add_argument("--softmax-dtype", default="fp32", choices=["fp32", "bf16"])
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    names = SUITE if args.workload == "suite" else (args.workload,)
    workloads = [WORKLOADS[n] for n in names]
    w = workloads[0]
    world, rank, local = dist_init()
    if world != args.gpus and world > 1:
        args.gpus = world
    if args.op != "attention":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the reference arm covers the attention call only"}))
        else:
            run_op(args, world, rank, local)
    elif args.impl == "reference":
        run_reference(args, w, world, rank)
    else:
        run_ours(args, workloads, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

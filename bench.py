#!/usr/bin/env python3
"""Benchmark of the fused attention forward on GB300.

Default workload: B=2, H=16, N=4096, d=128, causal, bf16 (the headline
configuration).  One step = one fa_fwd call over the whole batch (every
(batch, head, query tile) unit).  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--impl ours (default): CUDA-event time of K launches with inputs resident in
HBM and L2 flushed (a 256 MiB write and a 256 MiB read) between launches; the end-to-end
figure adds, every step, the pinned-host -> device copy of Q, K, V and the
device -> host copy of O and LSE.  --impl reference: the fp64 CPU oracle on
a fixed seeded sample of query rows of the same workload (the baseline
program), on the host cores.  Under torchrun each rank runs the workload on
its own GPU (independent replicas: weak scaling); timing is the max over
ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "attention fwd TFLOPS & % of GB300 BF16 tensor peak (N=4096,d=128,causal)"
UNIT = "TFLOPS"
# The split-KV decode workloads are bound by HBM: GB/s of algorithmic bytes.
DECODE_METRIC = "split-KV decode attention GB/s of algorithmic HBM bytes & % of measured HBM bandwidth"
DECODE_UNIT = "GB/s"
# The backward pass: nominal FLOPs are 2.5x the forward's (five N x N x d
# products against two), the convention of the FlashAttention line of work.
BWD_METRIC = "attention bwd TFLOPS (nominal 2.5x forward FLOPs) & % of GB300 BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
# NVIDIA's published dense (no 2:4 sparsity) BF16/FP16 tensor rate of one
# Blackwell Ultra (GB300) GPU, reported beside the measured peak.
NOMINAL_BF16_TFLOPS = 2250.0
# exp2 (MUFU) throughput per SM per clock, measured on GB300 with a
# microbenchmark of back-to-back ex2.approx.ftz.f32: the forward's secondary
# ceiling (one exponential per visible score).
EX2_PER_CLK_PER_SM = 32
NUM_SMS = 152


class L2Flush:
    """Evicts the inputs from L2 between timed launches, untimed: a 256 MiB
    write, then a 256 MiB read of a second buffer.  The read also evicts the
    write's dirty lines, so their write-back happens here and not inside the
    next timed launch (which would charge an HBM-bound kernel for ~126 MB of
    someone else's writes)."""

    def __init__(self, dev):
        import torch

        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()
# DRAM bytes (read + write) of one split-KV call (the clustered split pass),
# from one ncu capture per workload (profiles/); a workload is left out
# until a capture of the kernel as benchmarked exists.
NCU_TRAFFIC_BYTES_DECODE = {
    "decode_b4h16q16k16384d128_causal": 538_348_715,
    "decode_b4h16q1k16384d128": 538_085_120,
}
# DRAM bytes (read + write) of one backward step (three launches), from an
# ncu capture; a workload is left out until a capture of the kernels as
# benchmarked exists.
NCU_TRAFFIC_BYTES_BWD = {
    "b2h16n4096d128_causal": 436_226_816,
}
# Per-launch DRAM traffic of the forward kernel per workload, from an ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum); a workload is left
# out until a capture of the kernel as benchmarked exists.
NCU_TRAFFIC_BYTES = {
    "b2h16n4096d128_causal": 137_546_752,
    "b2h16n4096d256_causal": 575_460_352,
    "b2h16n4096d128_causal_fp16": 137_477_973,
    "b2h16n4096d96_causal": 77_837_909,
    "b2h16n4096d64_causal": 50_824_704,
    "b4h8n1024d64": 12_651_179,
    "b1h16n16000d128_causal": 560_115_371,
    "b1h32n8192d128_causal_qk3": 574_306_987,
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples the SM clock, the clock-event (throttle) reasons and the power
    draw of one GPU through NVML's read-only queries (libnvidia-ml, called
    with ctypes), in a background thread every ~2 ms and on demand
    (sample()); only samples taken between mark_start() and mark_stop() count.
    Changes no setting of the GPU."""

    NVML_CLOCK_SM = 1
    # nvmlClocksEventReason* bits (NVML API)
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, dev_index: int):
        self.samples = []  # (perf_counter, sm_mhz, reasons_mask, power_mw)
        self.t_start = self.t_stop = None
        self.error = None
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._lock = threading.Lock()
        self.nvml = self.handle = None
        try:
            import ctypes

            self.ct = ctypes
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            self.handle = self._find_handle(dev_index)
            mx = ctypes.c_uint(0)
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, self.NVML_CLOCK_SM,
                                                   ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) \
                or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError) as e:
            self.error = f"NVML unavailable: {e}"
            self.nvml = self.handle = None

    def _find_handle(self, dev_index: int):
        """NVML handle of the CUDA device: by UUID, else by the index that
        CUDA_VISIBLE_DEVICES maps it to."""
        import torch

        ct = self.ct
        handle = ct.c_void_p()
        uuid = getattr(torch.cuda.get_device_properties(dev_index), "uuid", None)
        if uuid is not None:
            text = str(uuid)
            if not text.startswith("GPU-"):
                text = "GPU-" + text
            if self.nvml.nvmlDeviceGetHandleByUUID(text.encode(), ct.byref(handle)) == 0:
                return handle
        index = dev_index
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if ids and all(x.isdigit() for x in ids) and dev_index < len(ids):
            index = int(ids[dev_index])
        if self.nvml.nvmlDeviceGetHandleByIndex_v2(ct.c_uint(index), ct.byref(handle)) != 0:
            raise OSError("no NVML handle for the device")
        return handle

    def sample(self):
        if self.handle is None:
            return
        ct = self.ct
        mhz, mask, mw = ct.c_uint(0), ct.c_ulonglong(0), ct.c_uint(0)
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, ct.byref(mhz)) != 0:
            return
        self._reasons_fn(self.handle, ct.byref(mask))
        self.nvml.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw))
        with self._lock:
            self.samples.append((time.perf_counter(), float(mhz.value), int(mask.value),
                                 float(mw.value)))

    def _run(self):
        while not self._stop.is_set():
            self.sample()
            self._stop.wait(0.002)

    def start(self):
        if self.handle is None:
            return
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def mark_start(self):
        self.t_start = time.perf_counter()

    def mark_stop(self):
        self.t_stop = time.perf_counter()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)
        return self.summary()

    def summary(self):
        if self.handle is None:
            return {"sm_mhz": None, "samples_in_timed_region": 0, "error": self.error}
        with self._lock:
            inside = [x for x in self.samples
                      if self.t_start is not None and self.t_stop is not None
                      and self.t_start <= x[0] <= self.t_stop]
        out = {"source": "NVML (read-only queries, ~2 ms period, in process)",
               "sm_max_mhz": self.max_mhz, "samples_in_timed_region": len(inside)}
        if not inside:
            out.update({"sm_mhz": None, "reasons": [],
                        "note": "no sample fell inside the timed region"})
            return out
        mhz = [x[1] for x in inside]
        reasons = sorted({name for x in inside for name, bit in self.REASONS.items()
                          if x[2] & bit})
        out.update({"sm_mhz": statistics.median(mhz), "sm_mhz_min": min(mhz),
                    "sm_mhz_max": max(mhz), "reasons": reasons,
                    "power_w_max": max(x[3] for x in inside) / 1000.0})
        return out


def timed_launches(step, flush, steps: int, warmup: int, stream, dev, world: int, sampler):
    """Warm-up, then `steps` timed steps, each bracketed by CUDA events on
    `stream` and followed by an untimed L2 flush; barrier + synchronize on
    both sides of the timed region.  The clock sampler runs from before the
    warm-up, and one untimed flush keeps the GPU busy up to the first timed
    step (as every later step follows a flush), so no timed step starts on an
    idle GPU.  While the GPU works through the queued steps the host samples
    the clocks too.  Returns (per-step ms list, clock summary or None)."""
    import torch

    if sampler:
        sampler.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for _ in range(warmup):
        step()
        flush()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark_start()
    flush()
    for i in range(steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        flush()
    while not ends[-1].query():
        if sampler:
            sampler.sample()
        time.sleep(0.0005)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark_stop()
    if world > 1:
        torch.distributed.barrier()
    per_launch_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    clocks = sampler.stop() if sampler else None
    if clocks and clocks.get("sm_mhz"):
        med = statistics.median(per_launch_ms)
        clocks["step_kcycles_at_median_mhz"] = med * clocks["sm_mhz"]  # ms x MHz = kcycles
    return per_launch_ms, clocks


def reduce_max_over_ranks(values, device=None):
    """Element-wise max of a list of floats over all ranks (identity when the
    process group is not initialised).  Used for the per-rank timings."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_tflops(world: int, flops_per_step: float, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank runs `steps` steps of `flops_per_step`;
    the job takes the slowest rank's `ms`."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def order1_bytes(w) -> float:
    """Algorithmic HBM bytes of the K/V-outer loop order (64 x 64 tiles):
    K and V read once; per visible (query tile, key tile) step Q_i read and
    the running fp32 O_i, m_i, l_i read (after the first step) and written
    (before the last); O (bf16) and LSE written once."""
    t = -(-w.N // 64)
    steps = t * (t + 1) // 2 if w.causal else t * t
    per_tile_q = 64 * w.d * 2
    state = 64 * (w.d + 2) * 4
    bh = w.B * w.H
    return bh * (2 * w.N * w.d * 2 + steps * per_tile_q + 2 * (steps - t) * state
                 + w.N * w.d * 2 + w.N * 4)


def cpu_oracle_sample_decode(w, qkv, heads: int, threads: int = 0, min_seconds: float = 0.0):
    """Time the fp64 oracle on the first `heads` (batch, head) slices of a
    decode workload, repeated until `min_seconds` have passed (at least
    once); returns (seconds, algorithmic bytes processed, repetitions,
    cores)."""
    import oracle

    q, k, v = (np.ascontiguousarray(a.reshape(w.B * w.H, *a.shape[2:])[:heads]) for a in qkv)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.attention(q, k, v, w.causal, w.scale, threads=threads)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    nbytes = reps * w.io_bytes * heads / (w.B * w.H)
    return dt, nbytes, reps, oracle.max_threads() if threads <= 0 else threads


def cpu_oracle_sample(w, qkv, rows_per_head: int, seed: int, threads: int = 0,
                      min_seconds: float = 0.0):
    """Time the fp64 oracle on a fixed seeded sample of query rows (all rows
    when rows_per_head is 0 or >= N), repeated until min_seconds have passed
    (at least once).

    Returns (seconds, flops, rows per head, repetitions, cores).  FLOPs count
    the same work the metric counts: 4·d per (query, visible key) pair (2·d
    for the score, 2·d for the P·V row)."""
    import oracle

    q, k, v = qkv
    if rows_per_head <= 0 or rows_per_head >= w.N:
        rows = None
        idx = np.arange(w.N, dtype=np.int64)
    else:
        rng = np.random.Generator(np.random.PCG64(seed))
        rows = np.sort(rng.permutation(w.N)[:rows_per_head]).astype(np.int64)
        idx = rows
    visible = (idx + 1) if w.causal else np.full(idx.size, w.N)
    flops = float(4.0 * w.d * visible.sum() * w.B * w.H)
    reps = 0
    t0 = time.perf_counter()
    while True:
        oracle.attention(q, k, v, w.causal, w.scale, rows=rows, threads=threads,
                         dtype=getattr(w, "dtype", "bf16"))
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    cores = oracle.max_threads() if threads <= 0 else threads
    return dt, flops * reps, idx.size, reps, cores


def run_reference(args, w):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    if isinstance(w, workloads.DecodeWorkload):
        return run_reference_decode(args, w)
    rows_per_head = args.ref_rows
    qkv = workloads.generate(w)
    times = []
    flops = 0.0
    cores = 0
    for i in range(args.warmup + args.steps):
        dt, flops, n_rows, _, cores = cpu_oracle_sample(w, qkv, rows_per_head, seed=1000 + w.seed)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = flops * len(times) / total / 1e12
    sample = (f"{rows_per_head} seeded query rows per head x {w.B * w.H} heads "
              f"({100.0 * rows_per_head / w.N:.2f}% of the rows) per step, fp64 oracle, "
              f"{cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_decode(args, w):
    world, _, _ = dist_setup()
    qkv = workloads.generate_decode(w)
    times, nbytes, heads, cores = [], 0.0, 1, 0
    for i in range(args.warmup + args.steps):
        heads = 2
        dt, nbytes, _, cores = cpu_oracle_sample_decode(w, qkv, heads=heads)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    sample = (f"{heads} of {w.B * w.H} (batch, head) slices per step, all {w.Nq} queries "
              f"against {w.Nk} keys, fp64 oracle, {cores} threads")
    line = {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": DECODE_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": DECODE_UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": DECODE_UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w):
    import torch

    import tiled_attention_forward_attn_gb300 as fa

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.load_library()

    decode = isinstance(w, workloads.DecodeWorkload)
    q, k, v = workloads.generate_decode(w) if decode else workloads.generate(w)
    elem = getattr(w, "dtype", "bf16")
    qd, kd, vd = (workloads.as_torch(a, elem).to(dev) for a in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty(tuple(qd.shape[:3]), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    if decode:
        ws_bytes = fa.fa_fwd_splitkv_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, 0)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        n_splits = fa.fa_fwd_splitkv_num_splits(w.B, w.H, w.Nq, w.Nk, w.d, 0)

        def step():
            fa.fa_fwd_splitkv(qd, kd, vd, o, lse, w.causal, w.scale, 0, workspace, stream)
    elif args.loop_order:
        ws_ord = torch.empty(max(16, fa.load_library().fa_fwd_order_ablation_workspace_bytes(
            w.B, w.H, w.N, w.d, args.loop_order)), dtype=torch.uint8, device=dev)

        def step():
            fa.attention_forward_order_ablation(qd, kd, vd, w.causal, w.scale, args.loop_order,
                                                workspace=ws_ord, out=(o, lse), stream=stream)
    else:
        def step():
            fa.fa_fwd(qd, kd, vd, o, lse, w.causal, w.scale, stream)

    sampler = ClockSampler(local) if rank == 0 else None
    per_launch_ms, clocks = timed_launches(step, flush, args.steps, args.warmup, stream, dev,
                                           world, sampler)
    kernel_ms = sum(per_launch_ms)

    # End to end, every step from pinned host inputs to pinned host outputs.
    # The forward goes through the C ABI's host-buffer entry point
    # (fa_fwd_host: three uploads, the kernel, two downloads on one stream),
    # steps alternating between two streams with their own device staging, so
    # step i+1's uploads overlap step i's kernel and downloads.  The other
    # paths copy with torch around their device-pointer call.
    hq, hk, hv = (workloads.as_torch(a, elem).pin_memory() for a in (q, k, v))
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    hl = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho[0].numel() * ho[0].element_size() + hl[0].numel() * hl[0].element_size()
    host_path = not args.loop_order
    streams = [stream, torch.cuda.Stream(dev)]
    if host_path and decode:
        ws_host = [torch.empty(fa.fa_fwd_splitkv_host_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d, 0),
                               dtype=torch.uint8, device=dev) for _ in range(2)]
    elif host_path:
        ws_host = [torch.empty(fa.fa_fwd_host_workspace_bytes(w.B, w.H, w.N, w.d),
                               dtype=torch.uint8, device=dev) for _ in range(2)]

    def e2e_step(i):
        if host_path and decode:
            fa.fa_fwd_splitkv_host(hq, hk, hv, ho[i % 2], hl[i % 2], w.causal, w.scale, 0,
                                   ws_host[i % 2], streams[i % 2])
            return
        if host_path:
            fa.fa_fwd_host(hq, hk, hv, ho[i % 2], hl[i % 2], w.causal, w.scale, ws_host[i % 2],
                           streams[i % 2])
            return
        qd.copy_(hq, non_blocking=True)
        kd.copy_(hk, non_blocking=True)
        vd.copy_(hv, non_blocking=True)
        step()
        ho[0].copy_(o, non_blocking=True)
        hl[0].copy_(lse, non_blocking=True)

    for i in range(max(3, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_steps = max(10, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(streams[0])
    streams[1].wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    streams[0].wait_stream(streams[1])
    e1.record(streams[0])
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)

    kernel_ms, e2e_ms = reduce_max_over_ranks([kernel_ms, e2e_ms], device=dev)

    if rank == 0 and decode:
        peaks, peaks_src = load_peaks()
        per_step = float(w.io_bytes)
        value = world * per_step * args.steps / (kernel_ms * 1e-3) / 1e9
        achieved = per_step / (kernel_ms * 1e-3 / args.steps) / 1e9
        peak = float(peaks["hbm_gbs"])
        e2e_value = world * per_step * e2e_steps / (e2e_ms * 1e-3) / 1e9
        cpu = None
        if world == 1 and not args.skip_cpu_baseline:
            dt, nbytes, reps, cores = cpu_oracle_sample_decode(w, (q, k, v), heads=w.B * w.H,
                                                               min_seconds=10.0)
            cpu = {"value": nbytes / dt / 1e9, "unit": DECODE_UNIT, "cores": cores,
                   "kind": "oracle",
                   "sample": (f"the whole workload ({w.B * w.H} (batch, head) slices, {w.Nq} "
                              f"queries against {w.Nk} keys) {reps} times, fp64 oracle, "
                              f"{dt:.1f} s")}
        line = {
            "metric": DECODE_METRIC, "value": value, "unit": DECODE_UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": kernel_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                       "causal": w.causal, "splits": n_splits,
                       "l2": "flushed between launches (256 MiB write + 256 MiB read, untimed); K+V exceed L2",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "pct_of_peak": 100.0 * achieved / peak,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": f"{peaks_src} hbm_gbs",
                         "timed": "the whole split-KV call (one or two launches), per step",
                         "traffic": NCU_TRAFFIC_BYTES_DECODE.get(w.name)},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": DECODE_UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step": e2e_ms / e2e_steps,
                    "path": "fa_fwd_splitkv_host (C ABI, host buffers), steps alternating "
                            "between two streams"},
            # one clustered launch per step when the ranges fit in a cluster
            # (<= 8), else the split pass and the combine pass
            "gpu_launches": (1 if n_splits <= 8 else 2) * args.steps,
            "launch_ms": {"min": min(per_launch_ms), "median": statistics.median(per_launch_ms),
                          "max": max(per_launch_ms)},
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    elif rank == 0:
        peaks, peaks_src = load_peaks()
        flops_step = w.flops
        value = job_tflops(world, flops_step, args.steps, kernel_ms)
        avg_launch_s = kernel_ms * 1e-3 / args.steps
        achieved = flops_step / avg_launch_s / 1e12
        peak = float(peaks["bf16_tflops"])
        e2e_value = job_tflops(world, flops_step, e2e_steps, e2e_ms)

        cpu = None
        if world == 1 and not args.skip_cpu_baseline:
            dt, fl, n_rows, reps, cores = cpu_oracle_sample(
                w, (q, k, v), args.cpu_rows, seed=2000 + w.seed, min_seconds=args.cpu_seconds)
            what = ("the whole workload (every row of every head)" if n_rows == w.N else
                    f"{n_rows} seeded query rows per head x {w.B * w.H} heads "
                    f"({100.0 * n_rows / w.N:.2f}% of the rows)")
            full_exact = 4.0 * w.d * w.B * w.H * (w.N * (w.N + 1) / 2 if w.causal else w.N * w.N)
            cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
                   "sample": f"{what}, {reps} time(s), fp64 oracle, {dt:.1f} s",
                   "extrapolated_full_s": dt * full_exact / fl,
                   "extrapolation": "time of the whole workload at the sample's FLOP rate "
                                    "(an extrapolation, not a measurement)"}
        # One exponential per visible score element (the exact causal count).
        n_exp = w.B * w.H * (w.N * (w.N + 1) / 2 if w.causal else w.N * w.N)
        sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
        ex2_peak = EX2_PER_CLK_PER_SM * NUM_SMS * sm_mhz * 1e6 / 1e9
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_source": f"{peaks_src} bf16_tflops (burst)" + (
                        "; fp16 x 1: its nominal dense rate equals bf16's"
                        if elem == "f16" else ""),
                    "traffic": None if args.loop_order else NCU_TRAFFIC_BYTES.get(w.name),
                    "secondary": {"what": "exp2 (MUFU) rate, one per visible score",
                                  "achieved": n_exp / avg_launch_s / 1e9, "peak": ex2_peak,
                                  "unit": "Gexp/s", "frac": n_exp / avg_launch_s / 1e9 / ex2_peak,
                                  "peak_source": f"{EX2_PER_CLK_PER_SM}/clk/SM measured x "
                                                 f"{NUM_SMS} SMs x {sm_mhz:.0f} MHz"}}
        if args.loop_order == 1:
            # The K/V-outer order moves the running state through HBM every
            # step: its own algorithmic bytes bound it.
            nbytes = order1_bytes(w)
            roofline = {"bound": "hbm", "achieved": nbytes / avg_launch_s / 1e9,
                        "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                        "frac": nbytes / avg_launch_s / 1e9 / float(peaks["hbm_gbs"]),
                        "peak_source": f"{peaks_src} hbm_gbs",
                        "algorithmic_bytes": nbytes, "traffic": None}
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": kernel_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": elem, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "scale": w.scale,
                       "l2": "flushed between launches (256 MiB write + 256 MiB read, untimed)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       **({"loop_order": {1: "K/V outer (v1)", 2: "Q outer (v2)"}[args.loop_order],
                           "kernel": "fa_fwd_order_ablation (64x64 tiles, warp MMAs)"}
                          if args.loop_order else {})},
            "pct_of_peak": 100.0 * achieved / peak,
            "pct_of_nominal": 100.0 * achieved / NOMINAL_BF16_TFLOPS,
            "nominal_peak": {"value": NOMINAL_BF16_TFLOPS, "unit": "TFLOP/s",
                             "source": "NVIDIA Blackwell Ultra (GB300) dense BF16 tensor rate "
                                       "per GPU, without 2:4 sparsity"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step": e2e_ms / e2e_steps,
                    "path": ("fa_fwd_host (C ABI, host buffers), steps alternating between two "
                             "streams" if host_path else "torch copies around the C ABI call")},
            "gpu_launches": args.steps,
            "launch_ms": {"min": min(per_launch_ms), "median": statistics.median(per_launch_ms),
                          "max": max(per_launch_ms)},
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_reference_bwd(args, w):
    """The oracle's backward on one (batch, head) slice of the workload per
    step (one slice runs on one thread); rank 0 only."""
    import oracle

    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    q, k, v = workloads.generate(w)
    do = workloads.generate_shape(w.B, w.H, w.N, w.d, seed=5000 + w.seed)[0]
    sl = [np.ascontiguousarray(a[:1, :1]) for a in (q, k, v, do)]
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.attention_bwd(*sl, w.causal, w.scale)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    fl = 2.5 * w.flops / (w.B * w.H)
    value = fl * len(times) / total / 1e12
    sample = f"gradients of 1 of the {w.B * w.H} (batch, head) slices per step, fp64 oracle, 1 thread"
    print(json.dumps({
        "impl": "reference", "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "pass": "bwd", "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0}), flush=True)
    return 0


def run_ours_bwd(args, w):
    """Time fa_bwd (pre-pass, dK/dV pass, dQ pass) on the workload's shape;
    O and LSE come from one untimed fa_fwd, dO is seeded."""
    import torch

    import tiled_attention_forward_attn_gb300 as fa

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.load_library()
    elem = getattr(w, "dtype", "bf16")
    q, k, v = workloads.generate(w)
    do = workloads.generate_shape(w.B, w.H, w.N, w.d, seed=5000 + w.seed, dtype=elem)[0]
    qd, kd, vd, dod = (workloads.as_torch(a, elem).to(dev) for a in (q, k, v, do))
    o, lse = fa.attention_forward(qd, kd, vd, causal=w.causal, scale=w.scale)
    dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.fa_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, w.causal, w.scale, ws, stream)

    sampler = ClockSampler(local) if rank == 0 else None
    per_launch_ms, clocks = timed_launches(step, flush, args.steps, args.warmup, stream, dev,
                                           world, sampler)
    kernel_ms = sum(per_launch_ms)

    # End to end: Q, K, V, O, LSE, dO in from pinned host memory, dQ, dK, dV out.
    hosts_in = [workloads.as_torch(a, elem).pin_memory() for a in (q, k, v)]
    hosts_in += [o.cpu().pin_memory(), lse.cpu().pin_memory(),
                 workloads.as_torch(do, elem).pin_memory()]
    hosts_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in hosts_in)
    d2h = sum(t.numel() * t.element_size() for t in hosts_out)

    # Every step through the C ABI's host-buffer entry point (fa_bwd_host: six
    # uploads, the three backward launches, three downloads on one stream),
    # steps alternating between two streams with their own device staging.
    outs2 = [hosts_out, [torch.empty_like(t).pin_memory() for t in hosts_out]]
    streams = [stream, torch.cuda.Stream(dev)]
    ws_host = [torch.empty(fa.fa_bwd_host_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                           device=dev) for _ in range(2)]

    def e2e_step(i):
        fa.fa_bwd_host(*hosts_in, *outs2[i % 2], w.causal, w.scale, ws_host[i % 2], streams[i % 2])

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    e2e_steps = max(10, min(args.steps, 100))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(streams[0])
    streams[1].wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    streams[0].wait_stream(streams[1])
    e1.record(streams[0])
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)
    kernel_ms, e2e_ms = reduce_max_over_ranks([kernel_ms, e2e_ms], device=dev)

    if rank == 0:
        import oracle

        peaks, peaks_src = load_peaks()
        flops_step = 2.5 * w.flops
        value = job_tflops(world, flops_step, args.steps, kernel_ms)
        achieved = flops_step / (kernel_ms * 1e-3 / args.steps) / 1e12
        peak = float(peaks["bf16_tflops"])
        cpu = None
        if world == 1 and not args.skip_cpu_baseline:
            sl = [np.ascontiguousarray(a[:1, :1]) for a in (q, k, v, do)]
            t0 = time.perf_counter()
            oracle.attention_bwd(*sl, w.causal, w.scale, dtype=elem)
            dt = time.perf_counter() - t0
            cpu = {"value": 2.5 * w.flops / (w.B * w.H) / dt / 1e12, "unit": UNIT,
                   "cores": 1, "kind": "oracle",
                   "sample": (f"gradients of one of the {w.B * w.H} (batch, head) slices, fp64 "
                              f"oracle (one slice runs on one thread), {dt:.1f} s")}
        line = {
            "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": kernel_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": elem,
            "data": "synthetic",
            "config": {"workload": w.name, "pass": "bwd", "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "scale": w.scale,
                       "l2": "flushed between launches (256 MiB write + 256 MiB read, untimed)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "pct_of_peak": 100.0 * achieved / peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "peak_source": f"{peaks_src} bf16_tflops (burst)" + (
                             "; fp16 x 1: its nominal dense rate equals bf16's"
                             if elem == "f16" else ""),
                         "timed": "pre-pass, dK/dV pass and dQ pass together, per step",
                         # DRAM bytes of the three launches of one step (ncu, profiles/).
                         "traffic": NCU_TRAFFIC_BYTES_BWD.get(w.name),
                         "traffic_scope": "pre-pass + dK/dV pass + dQ pass, per step"},
            "cpu_baseline": cpu,
            "e2e": {"value": job_tflops(world, flops_step, e2e_steps, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step": e2e_ms / e2e_steps,
                    "path": "fa_bwd_host (C ABI, host buffers), steps alternating between two "
                            "streams"},
            "gpu_launches": 3 * args.steps,
            "launch_ms": {"min": min(per_launch_ms), "median": statistics.median(per_launch_ms),
                          "max": max(per_launch_ms)},
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=workloads.HEADLINE.name,
                    choices=[x.name for x in workloads.WORKLOADS + workloads.VARIANT_WORKLOADS
                             + workloads.DECODE_WORKLOADS])
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="query rows per head timed for the CPU baseline (0: all rows, the "
                         "whole workload, repeated for at least --cpu-seconds)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="query rows per head per step of --impl reference")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--loop-order", type=int, choices=(1, 2), default=0,
                    help="time the loop-order ablation kernel instead of fa_fwd: 1 = K/V "
                         "outer (v1), 2 = Q outer (v2)")
    ap.add_argument("--pass", dest="pass_", choices=("fwd", "bwd"), default="fwd",
                    help="bwd: time the backward pass of the (square) workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = workloads.by_name(args.workload)
    if args.pass_ == "bwd":
        if not isinstance(w, workloads.Workload) or w.d > 128 or w.d % 16:
            ap.error("--pass bwd takes a square workload with d a multiple of 16 up to 128")
        if args.impl == "reference":
            return run_reference_bwd(args, w)
        return run_ours_bwd(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())

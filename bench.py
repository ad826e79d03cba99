"""Benchmark: product-VQ encode throughput (sub-vectors encoded per second).

One step = one encode of the whole workload (default: the Falcon3-7B-shape
prefill, 4096 tokens x 4 KV heads x head_dim 256 -> N = 1,048,576 fp16
sub-vectors of length 4 against 256 centroids), launched through the C ABI
with inputs resident in HBM.  L2 is flushed before every step (a 256 MiB
write, larger than the 129 MB L2) and each step is timed with CUDA events on
the launching stream.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank encodes its own full workload (independent problems,
no data-path collective: weak scaling); with ``--partition`` the ranks split
one workload instead (``vq_partition``: each encodes its share against
replicated codebooks, no collective: strong scaling).  Rank 0 prints.
``--impl reference`` times the CPU oracle on this host's cores instead (the
baseline arm).  The default line also carries ``other_workloads``: the Llama
decode step, long-context and grouped-adversarial encodes, timed the same way.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "sub-vectors encoded/sec (1xGB300) and % of FP32 CUDA-core peak"
UNIT = "sub-vectors/s"
# The pages' own number for this exact workload (Falcon3-7B shape, S=4096,
# D=256, sub_dim 4, 256 centroids, N = 1,048,576): 7.98 ms per call on an
# Apple M-series GPU -> 131.4 M sub-vectors/s.  Context only (other hardware).
PAGES_FALCON_SUBVEC_PER_S = 1_048_576 / 7.98e-3
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture, keyed by the exact launch description it was taken on; a
# kernel that has changed since reports null (see profiles/).
MEASURED_TRAFFIC = {
    "kernel=encode_tc dtype=f16 sub_dim=4 tmem_cols=64 tiles_per_block=14 tiles_per_step=2 "
    "centroid_group=16 grid=586 smem=47718": 8_425_984,
    "kernel=encode_tc dtype=f16 sub_dim=8 tmem_cols=64 tiles_per_block=3 tiles_per_step=1 "
    "centroid_group=8 grid=704 smem=34880": 4_364_800,
}
# The same for the other ops' dominant kernels, keyed by (op, workload, input dtype):
# attn_partial, hadamard_rows, scalar_scan (fp32 keys).
MEASURED_OP_TRAFFIC = {
    ("attention", "llama_attention", "f16"): 67_280_384 + 391_936,
    ("hadamard", "turboquant_keys", "f16"): 67_156_992 + 4_517_376,
    ("scalar", "turboquant_keys", "f32"): 134_288_384 + 12_928_256,
}
L2_FLUSH_BYTES = 256 << 20
# How the encode rooflines count work.
ENCODE_ACCOUNTING = ("effective: brute-force F = n_centroids * 3 * sub_dim fp32 operations per "
                     "sub-vector over the measured time; the screening kernels do less "
                     "arithmetic and return the same index, so frac can exceed 1")
L2_POLICY = "flushed before every step (256 MiB write); per-step CUDA events on the launching stream"
# Workloads timed beside the headline one in the default line: (name, steps).
OTHER_WORKLOADS = (("tiny", 300), ("llama_decode", 300), ("long_context", 100),
                   ("grouped_adversarial", 20))
FP32_LANES_PER_SM = 128
CLOCK_REASON_BITS = {
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
    0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
    0x100: "display_clock_setting",
}


def flops_per_subvector(w: workloads.Workload) -> int:
    """Algorithmic fp32 operations per encoded sub-vector: for each centroid,
    sub_dim subtractions, sub_dim squares, sub_dim - 1 additions and one
    comparison = 3 * sub_dim."""
    return w.n_centroids * 3 * w.sub_dim


def bytes_per_subvector(w: workloads.Workload) -> int:
    """Algorithmic HBM bytes per sub-vector: the fp16 row in, the uint32 index
    out (the codebook, a few KiB per group, is negligible)."""
    return 2 * w.sub_dim + 4


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._reader = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._reader is not None:
                self._reader.join(timeout=2)

    def summary(self) -> dict:
        sm, sm_max, reasons = [], None, set()
        for line in self.lines:
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                sm_max = float(f[2])
                active = int(f[4], 16) if f[4].startswith("0x") else int(f[4])
            except ValueError:
                continue
            for bit, name in CLOCK_REASON_BITS.items():
                if active & bit:
                    reasons.add(name)
            for k, name in ((5, "hw_slowdown"), (6, "hw_thermal_slowdown"),
                            (7, "sw_thermal_slowdown"), (8, "sw_power_cap")):
                if f[k].lower() == "active":
                    reasons.add(name)
        busy = [v for v in sm if v > 0]
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": sm_max,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_max(values, device) -> list:
    """Element-wise maximum of ``values`` over all ranks of the default process
    group (the values themselves when running as a single process)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_throughput(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job rate: every rank encodes its own workload of ``units_per_rank``
    sub-vectors; the job takes as long as the slowest rank."""
    return units_per_rank * world / seconds_max


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_baseline(w_name: str, x: np.ndarray, cb: np.ndarray, budget_s: float = 12.0) -> dict:
    """The CPU oracle on this host's cores over a bounded sample of the same
    workload: the first rows of group 0, encoded repeatedly (at least 3 runs)
    until about ``budget_s`` seconds of CPU work are done; the median run."""
    import oracle  # test infrastructure: used here only for the CPU baseline

    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    w = workloads.WORKLOADS[w_name]
    m = x.shape[1]
    probe = min(m, 8192)
    t0 = time.perf_counter()
    oracle.encode(x[:1, :probe], cb[:1], n_threads=cores)
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    rows = int(min(m, max(probe, rate * budget_s / 3)))
    runs = int(min(30, max(3, round(budget_s * rate / rows))))
    xs = np.ascontiguousarray(x[:1, :rows])
    times = []
    for _ in range(runs):
        t0 = time.perf_counter()
        oracle.encode(xs, cb[:1], n_threads=cores)
        times.append(time.perf_counter() - t0)
    med = statistics.median(times)
    # the same oracle on one core, over a tenth of the sample
    rows1 = max(1, rows // 10)
    t0 = time.perf_counter()
    oracle.encode(np.ascontiguousarray(x[:1, :rows1]), cb[:1], n_threads=1)
    one_core = rows1 / max(time.perf_counter() - t0, 1e-9)
    return {"value": rows / med, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {rows} of {w.n} sub-vectors of {w_name} (codebook 0), "
                      f"median of {runs} runs ({sum(times):.1f} s in all), {cores} threads",
            "seconds": med,
            "value_1_core": one_core, "cpu_model": cpu_model()}


def cpu_model() -> str:
    """The host CPU's model name (or its implementer / part on Arm)."""
    try:
        text = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "CPU part"):
        for line in text.splitlines():
            if line.split(":")[0].strip() == key:
                return f"{key}: {line.split(':', 1)[1].strip()}"
    return "unknown"


def bench_reference(args) -> None:
    """The baseline arm: the CPU oracle, as it stands, on this host's cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle  # test infrastructure: the reference arm is the oracle

    oracle.build()
    w = workloads.WORKLOADS[args.workload]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    x, cb = workloads.generate(args.workload)
    g, m, sub = x.shape
    probe = min(m, 4096)
    t0 = time.perf_counter()
    oracle.encode(x[:1, :probe], cb[:1], n_threads=cores)
    rate = probe / max(time.perf_counter() - t0, 1e-6)
    per_step_s = min(1.0, 120.0 / max(1, args.steps + args.warmup))
    rows = int(min(m, max(256, rate * per_step_s)))
    xs = np.ascontiguousarray(x[:1, :rows])
    for _ in range(args.warmup):
        oracle.encode(xs, cb[:1], n_threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.encode(xs, cb[:1], n_threads=cores)
    total = time.perf_counter() - t0
    value = rows * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "strong" if args.partition else "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_block(w, args, world),
        "timing": {"l2": "not applicable: the CPU oracle, wall-clock time over the steps"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {rows} of {w.n} sub-vectors of {args.workload} per "
                                   f"step, {cores} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def config_block(w: workloads.Workload, args, world: int) -> dict:
    """The workload, identical for both arms (timing details go elsewhere)."""
    if world == 1:
        par = "single"
    else:
        par = f"partition{world}" if getattr(args, "partition", False) else f"replicas{world}"
    return {"workload": w.name, "description": w.description, "n_subvectors": w.n,
            "n_groups": w.n_groups, "sub_dim": w.sub_dim, "n_centroids": w.n_centroids,
            "input_dtype": "f16", "tokens": w.tokens, "kv_heads": w.kv_heads,
            "head_dim": w.head_dim, "layers": w.layers, "parallelism": par}


def time_steps(step, steps: int, warmup: int, flush, stream, dev, clock_index=None):
    """Run `warmup` untimed steps, then `steps` timed ones, each after an L2
    flush and bracketed by CUDA events on `stream`.  Returns the per-step
    milliseconds, the wall time of the timed region, and (with clock_index)
    the sampled clocks."""
    import torch

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(clock_index) if clock_index is not None else None
    if sampler:
        sampler.__enter__()
    try:
        region0 = time.perf_counter()
        for k in range(steps):
            flush.zero_()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize(dev)
        region_s = time.perf_counter() - region0
    finally:
        if sampler:
            sampler.__exit__(None, None, None)
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], region_s, (
        sampler.summary() if sampler else None)


def other_workloads(vq, dev, flush, stream, peak_tflops: float) -> dict:
    """The other encode workloads, one grouped launch per step, timed like
    the headline one: the tiny case (launch-bound), the Llama decode step,
    long context, grouped adversarial."""
    import torch

    out = {}
    for name, steps in OTHER_WORKLOADS:
        w = workloads.WORKLOADS[name]
        x, cb = workloads.generate(name)
        xd, cbd = torch.from_numpy(x).to(dev), torch.from_numpy(cb).to(dev)
        idx = torch.empty(x.shape[:2], dtype=torch.uint32, device=dev)
        ms, _, _ = time_steps(lambda: vq.vq_encode_grouped(xd, cbd, out=idx, stream=stream),
                              steps, 3, flush, stream, dev)
        mean = sum(ms) / len(ms)
        achieved = flops_per_subvector(w) * w.n / (mean * 1e-3) / 1e12
        out[name] = {"value": w.n / (mean * 1e-3), "unit": UNIT, "ms_per_step": mean,
                     "ms_median": statistics.median(ms), "steps": steps,
                     "n_subvectors": w.n, "n_groups": w.n_groups, "sub_dim": w.sub_dim,
                     "frac": achieved / peak_tflops, "accounting": ENCODE_ACCOUNTING,
                     "kernel": vq.vq_describe_launch(x.shape[0], x.shape[1], cb.shape[1],
                                                     x.shape[2], torch.float16, xd.data_ptr())}
        del xd, cbd, idx
    return out


def bench_ours(args) -> None:
    import torch
    import torch.distributed as dist

    from product_vq_kv_gb300.build import build

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build()
    if world > 1:
        dist.barrier()
    import product_vq_kv_gb300 as vq

    vq.load_library()
    w = workloads.WORKLOADS[args.workload]
    x, cb = workloads.generate(args.workload)
    if args.centroids:  # a smaller codebook: its first rows
        cb = np.ascontiguousarray(cb[:, : args.centroids])
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[args.dtype]
    xd = torch.from_numpy(x).to(dev).to(tdt)
    cbd = torch.from_numpy(cb).to(dev).to(tdt)
    if args.misalign:  # x one element off its natural alignment: the any-layout kernel
        buf = torch.empty(xd.numel() + 1, dtype=tdt, device=dev)
        buf[1:].copy_(xd.reshape(-1))
        xd = buf[1:].view(xd.shape)
    out = torch.empty(x.shape[:2], dtype=torch.uint32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    units = w.n  # sub-vectors this rank encodes per step
    if args.partition:
        # this rank's share of the one job (codebooks replicated, no collective)
        slices = vq.vq_partition(x.shape[0], x.shape[1], world, rank)
        units = sum(ng * nr for _, ng, _, nr in slices)
        share = torch.empty(units, dtype=torch.uint32, device=dev)

        def step():
            vq.vq_encode_partition(xd, cbd, world, rank, out=share, stream=stream)
    elif args.per_layer:
        # the pages' per-layer dispatch: one vq_encode launch per group
        views = [(xd[g], cbd[g], out[g]) for g in range(x.shape[0])]

        def step():
            for xg, cg, og in views:
                vq.vq_encode(xg, cg, out=og, stream=stream)
    else:
        def step():
            vq.vq_encode_grouped(xd, cbd, out=out, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    step_ms, region_s, clk = time_steps(step, args.steps, 0, flush, stream, dev, clock_index=local)
    if world > 1:
        dist.barrier()
    kernel_ms = sum(step_ms) / len(step_ms)
    median_ms = statistics.median(step_ms)
    kernel_ms, region_s, median_ms = reduce_max([kernel_ms, region_s, median_ms], dev)

    variant = (args.dtype != "f16" or args.centroids or args.misalign or args.per_layer
               or args.partition)
    # end to end through the host entry point: pinned host in, pinned host out
    xh = torch.from_numpy(x).pin_memory()
    cbh = torch.from_numpy(cb).pin_memory()
    outh = torch.empty(x.shape[:2], dtype=torch.uint32).pin_memory()
    e2e_steps = 0 if variant else max(3, min(args.steps, 200))
    for _ in range(3 if e2e_steps else 0):
        vq.vq_encode_grouped_host(xh, cbh, outh, xd, cbd, out, stream=stream)
    if world > 1:
        dist.barrier()
    e0 = time.perf_counter()
    for _ in range(e2e_steps):
        vq.vq_encode_grouped_host(xh, cbh, outh, xd, cbd, out, stream=stream)
    e2e_s = max(time.perf_counter() - e0, 1e-12)
    (e2e_s,) = reduce_max([e2e_s], dev)
    if world > 1:
        dist.barrier()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    props = torch.cuda.get_device_properties(dev)
    peaks = measured_peaks()
    desc = vq.vq_describe_launch(x.shape[0], x.shape[1], cb.shape[1], x.shape[2], tdt,
                                 xd.data_ptr())
    sm_max = peaks.get("sm_max_mhz") or clk["sm_max_mhz"] or 2070.0
    peak_tflops = props.multi_processor_count * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    # replicas: every rank encodes the whole workload; partition: the ranks
    # share one (rank 0's share stands for each rank's launch below)
    value = (w.n / (kernel_ms * 1e-3) if args.partition
             else job_throughput(units, world, kernel_ms * 1e-3))
    flops_unit = cb.shape[1] * 3 * w.sub_dim  # as flops_per_subvector, for the codebook used
    achieved = flops_unit * units / (kernel_ms * 1e-3) / 1e12
    roofline = {
        "bound": "alu", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s",
        "frac": achieved / peak_tflops,
        "traffic": None if args.partition else MEASURED_TRAFFIC.get(desc),
        "kernel": desc if not args.partition else f"{desc} (whole job; this rank: {units} rows)",
        "accounting": ENCODE_ACCOUNTING,
        "flops_per_unit": flops_unit, "units_per_launch": units,
        "peak_basis": f"{props.multi_processor_count} SMs x {FP32_LANES_PER_SM} FP32 lanes x "
                      f"2 (FMA) x {sm_max:.0f} MHz",
        "hbm_gbs": bytes_per_subvector(w) * units / (kernel_ms * 1e-3) / 1e9,
    }
    if clk["sm_mhz"]:
        roofline["frac_at_sampled_clock"] = roofline["frac"] * sm_max / clk["sm_mhz"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": kernel_ms,
        "ms_median": median_ms,
        "higher_is_better": True, "scaling": "strong" if args.partition else "weak",
        "vs_baseline": (value / world / PAGES_FALCON_SUBVEC_PER_S
                        if args.workload == "falcon_prefill" and not variant else None),
        "dtype": "f32", "data": "synthetic (seeded N(0,1) fp16 keys and codebooks"
                                + (f", as {args.dtype})" if args.dtype != "f16" else ")"),
        "config": dict(config_block(w, args, world), n_centroids=int(cb.shape[1]),
                       input_dtype=args.dtype),
        "timing": {"l2": L2_POLICY, "timed_region_s": region_s,
                   "x_misaligned": bool(args.misalign),
                   "dispatch": ("one vq_encode per group" if args.per_layer
                                else f"vq_encode_partition: {len(slices)} grouped launches"
                                if args.partition else "one grouped launch")},
        "gpu_launches": args.steps * (x.shape[0] if args.per_layer
                                      else len(slices) if args.partition else 1),
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "roofline": roofline,
        "e2e": None if variant else {"value": job_throughput(units * e2e_steps, world, e2e_s), "unit": UNIT,
                "h2d_bytes_per_step": x.nbytes + cb.nbytes,
                "d2h_bytes_per_step": int(units * 4),
                "path": "vq_encode_grouped_host with pinned host buffers: the kernel reads x and "
                        "writes the indices across the CPU-GPU link; codebooks copied"},
    }
    if world == 1 and not variant and args.workload == "falcon_prefill" and not args.no_other:
        del xd, cbd, out
        line["other_workloads"] = other_workloads(vq, dev, flush, stream, peak_tflops)
    if world == 1 and not args.no_cpu_baseline and not variant:
        line["cpu_baseline"] = cpu_baseline(args.workload, x, cb)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def bench_dequantize(args) -> None:
    """Decode throughput: 8-bit codes of the workload back to fp16 sub-vectors
    (one ``vq_dequantize_grouped`` per step), against the HBM roofline."""
    import torch

    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as vq

    dev = torch.device("cuda", 0)
    w = workloads.WORKLOADS[args.workload]
    x, cb = workloads.generate(args.workload)
    xd, cbd = torch.from_numpy(x).to(dev), torch.from_numpy(cb).to(dev)
    codes = vq.vq_encode_grouped_u8(xd, cbd)
    out = torch.empty_like(xd)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        flush.zero_()
        vq.vq_dequantize_grouped(codes, cbd, out=out, stream=stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clocks:
        for k in range(args.steps):
            flush.zero_()
            starts[k].record(stream)
            vq.vq_dequantize_grouped(codes, cbd, out=out, stream=stream)
            ends[k].record(stream)
        torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    bytes_per_unit = 1 + 2 * w.sub_dim  # uint8 code in, fp16 row out
    achieved = bytes_per_unit * w.n / (ms * 1e-3) / 1e9
    peak = measured_peaks().get("hbm_gbs") or 6800.0
    clk = clocks.summary()
    line = {
        "metric": "sub-vectors decoded/sec (1xGB300)", "value": w.n / (ms * 1e-3),
        "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8->f16", "data": "synthetic", "op": "dequantize",
        "config": config_block(w, args, 1), "gpu_launches": args.steps,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "bytes_per_unit": bytes_per_unit, "units_per_launch": w.n,
                     "accounting": "algorithmic bytes: one uint8 code read and one fp16 row "
                                   "written per sub-vector (codebooks negligible)"},
        "timing": {"l2": L2_POLICY},
        "e2e": None,
    }
    print(json.dumps(line))


def bench_smooth(args) -> None:
    """Encode fused with per-channel smoothing (uint8 codes out), one
    ``vq_encode_grouped_smooth`` per step, against the FP32 CUDA-core peak
    with the same per-sub-vector accounting as the plain encode."""
    import torch

    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as vq

    dev = torch.device("cuda", 0)
    w = workloads.WORKLOADS[args.workload]
    head_dim = w.sub_vectors_per_head * w.sub_dim
    x, smooth, cb = workloads.generate_smooth(args.workload)
    xd, sd, cbd = (torch.from_numpy(a).to(dev) for a in (x, smooth, cb))
    out = torch.empty(x.shape[:2], dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        vq.vq_encode_grouped_smooth(xd, sd, cbd, head_dim, index_bytes=1, out=out, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clocks:
        for k in range(args.steps):
            flush.zero_()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    props = torch.cuda.get_device_properties(dev)
    clk = clocks.summary()
    sm_max = measured_peaks().get("sm_max_mhz") or clk["sm_max_mhz"] or 2070.0
    peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    achieved = flops_per_subvector(w) * w.n / (ms * 1e-3) / 1e12
    line = {
        "metric": "smoothed sub-vectors encoded to 8-bit codes/sec (1xGB300)",
        "value": w.n / (ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "op": "smooth",
        "config": dict(config_block(w, args, 1), head_dim=head_dim, index_bytes=1),
        "gpu_launches": args.steps,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "flops_per_unit": flops_per_subvector(w), "units_per_launch": w.n,
                     "accounting": ENCODE_ACCOUNTING},
        "timing": {"l2": L2_POLICY},
        "e2e": None,
    }
    print(json.dumps(line))


def bench_sibling(args, fused: bool) -> None:
    """Scalar (sub_dim = 1) quantize of one layer's key cache against a 4-bit
    Lloyd-Max codebook (``--op scalar``: fp16 keys take the bucket-table
    kernel, bf16 keys the 64 KiB table build and lookup pass, fp32 keys the
    per-element search), or the randomised Hadamard rotation fused with it
    (``--op hadamard``); one launch per step (two for bf16 keys), against the
    HBM roofline of the key bytes in and 1 byte out per element."""
    import torch

    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as vq

    dev = torch.device("cuda", 0)
    sw = workloads.SCALAR_WORKLOADS["turboquant_keys"]
    x, c, diag = workloads.generate_scalar(sw.name)
    xd, cd, dd = (torch.from_numpy(a).to(dev) for a in (x, c, diag))
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[args.dtype]
    xd = xd.to(tdt)  # fp32 keys take the per-element exact search instead of the table
    out = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    ws = torch.empty(65536, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if fused:
            vq.vq_hadamard_quantize(xd, dd, cd, out=out, stream=stream)
        else:
            vq.vq_scalar_quantize(xd, cd, out=out, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clocks:
        for k in range(args.steps):
            flush.zero_()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    algo_bytes = (xd.element_size() + 1) * sw.n
    achieved = algo_bytes / (ms * 1e-3) / 1e9
    peak = measured_peaks().get("hbm_gbs") or 6800.0
    clk = clocks.summary()
    line = {
        "metric": ("key elements rotated and quantized/sec (1xGB300)" if fused
                   else "key elements scalar-quantized/sec (1xGB300)"),
        "value": sw.n / (ms * 1e-3), "unit": "elements/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "op": "hadamard" if fused else "scalar",
        "config": {"workload": sw.name, "batch": sw.batch, "heads": sw.heads,
                   "tokens": sw.tokens, "head_dim": sw.head_dim, "bits": sw.bits,
                   "input_dtype": args.dtype},
        "timing": {"l2": L2_POLICY},
        # bf16 keys: the table build and the lookup pass; fp16 keys (bucket
        # table built in the kernel), fp32 keys and the fused rotation: one launch
        "gpu_launches": args.steps * (2 if not fused and args.dtype == "bf16" else 1),
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": MEASURED_OP_TRAFFIC.get(("hadamard" if fused else "scalar", sw.name, args.dtype)),
                     "bytes_per_launch": algo_bytes,
                     "timed": "whole step" + (" (table build + lookup pass)" if not fused and args.dtype == "bf16"
                                              else ""),
                     "accounting": "algorithmic bytes: each key element read once and its "
                                   "uint8 index written once"},
        "e2e": None,
    }
    print(json.dumps(line))


def bench_attention(args) -> None:
    """Decode attention over the 8-bit product-VQ KV cache of the Llama-shape
    workload (one ``vq_attention_decode`` per step: table build, scores,
    softmax and value sum per token slice, then the merge of the slices),
    reported as query-head x cached-token scores per second against the HBM
    roofline of the code bytes it must read."""
    import torch

    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as vq

    dev = torch.device("cuda", 0)
    aw = workloads.ATTENTION_WORKLOADS["llama_attention"]
    arrays = workloads.generate_attention(aw.name)
    q, kc, kcb, vc, vcb = (torch.from_numpy(a).to(dev) for a in arrays)
    out = torch.empty_like(q)
    nbytes = vq.vq_attention_workspace_bytes(aw.batch, aw.heads_q, aw.heads_kv, aw.tokens,
                                             aw.head_dim, aw.sub_dim, aw.n_centroids)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        vq.vq_attention_decode(q, kc, kcb, vc, vcb, out=out, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clocks:
        for k in range(args.steps):
            flush.zero_()
            starts[k].record(stream)
            step()
            ends[k].record(stream)
        torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / args.steps
    scores = aw.batch * aw.heads_q * aw.tokens
    # algorithmic bytes: key and value codes, queries and outputs, codebooks
    small = 2 * aw.batch * aw.heads_q * aw.head_dim * 2 + 2 * aw.heads_kv * aw.n_centroids * aw.sub_dim * 2
    algo_bytes = aw.code_bytes + small
    achieved = algo_bytes / (ms * 1e-3) / 1e9
    peak = measured_peaks().get("hbm_gbs") or 6800.0

    # end to end: queries and codes copied from pinned host memory, the
    # output read back, every step (a decode step that starts from a host cache)
    hosts = [torch.from_numpy(a).pin_memory() for a in arrays]
    dev_in = [torch.empty_like(h, device=dev) for h in hosts]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(h.numel() * h.element_size() for h in hosts)
    d2h = out_h.numel() * out_h.element_size()
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for d_, h_ in zip(dev_in, hosts):
            d_.copy_(h_, non_blocking=True)
        vq.vq_attention_decode(*dev_in, out=out, workspace=ws, stream=stream)
        out_h.copy_(out, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t0) / e2e_steps

    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        qh, kch, kcbh, vch, vcbh = arrays
        t0 = time.perf_counter()
        oracle.attention_decode(qh[:1], kch[:1], kcbh, vch[:1], vcbh)
        dt = time.perf_counter() - t0
        cpu = {"value": aw.heads_q * aw.tokens / dt, "unit": "scores/s", "cores": 1,
               "kind": "oracle", "sample": f"batch row 0 of {aw.batch} ({aw.heads_q} query heads "
               f"x {aw.tokens} tokens), numpy float64"}
    clk = clocks.summary()
    line = {
        "metric": "decode-attention scores/sec over 8-bit VQ codes (1xGB300)",
        "value": scores / (ms * 1e-3), "unit": "scores/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8 codes, f16 q/codebooks, f32 accumulate",
        "data": "synthetic", "op": "attention",
        "config": {"workload": aw.name, "batch": aw.batch, "heads_q": aw.heads_q,
                   "heads_kv": aw.heads_kv, "tokens": aw.tokens, "head_dim": aw.head_dim,
                   "sub_dim": aw.sub_dim, "n_centroids": aw.n_centroids},
        "timing": {"l2": L2_POLICY},
        "gpu_launches": 2 * args.steps,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": MEASURED_OP_TRAFFIC.get(("attention", aw.name, "f16")),
                     "bytes_per_launch": algo_bytes,
                     "timed": "whole step (partial + combine kernels)",
                     "accounting": "algorithmic bytes: every key and value code read once "
                                   "(queries, codebooks and outputs negligible)"},
        "cpu_baseline": cpu,
        "e2e": {"value": scores / e2e_s, "unit": "scores/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
    }
    print(json.dumps(line))


def main() -> None:
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(workloads.WORKLOADS), default="falcon_prefill")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--dtype", choices=["f16", "bf16", "f32"], default="f16",
                   help="encode: input type (f32 rows and codebooks go to the tensor cores as tf32 pieces)")
    p.add_argument("--centroids", type=int, default=0,
                   help="encode: use only the first N codebook rows (below 64: brute force)")
    p.add_argument("--misalign", action="store_true",
                   help="encode: x one element off alignment (the any-layout kernel)")
    p.add_argument("--per-layer", action="store_true",
                   help="encode: one vq_encode launch per group instead of one grouped launch")
    p.add_argument("--partition", action="store_true",
                   help="encode under torchrun: the ranks split one workload (strong scaling) "
                        "instead of each encoding its own (weak scaling)")
    p.add_argument("--no-other", action="store_true",
                   help="encode: skip the other workloads of the default line")
    p.add_argument("--op", choices=["encode", "dequantize", "attention", "smooth", "scalar",
                                    "hadamard"], default="encode")
    args = p.parse_args()
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.impl == "reference":
        bench_reference(args)
    elif args.op == "dequantize":
        bench_dequantize(args)
    elif args.op == "attention":
        bench_attention(args)
    elif args.op == "smooth":
        bench_smooth(args)
    elif args.op in ("scalar", "hadamard"):
        bench_sibling(args, fused=args.op == "hadamard")
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()

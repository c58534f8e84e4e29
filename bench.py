#!/usr/bin/env python3
"""Benchmark: FP32 C = A x B at M = N = K = 4096 on one GB300 (TFLOP/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one call of ``gemm_f32`` (the whole hot path: block-tile
scheduling, shared-memory staging, register-tiled FFMA, epilogue) on the
headline workload, operands resident in HBM, L2 flushed before every step by
writing a buffer twice the L2 size.  Each step is timed with CUDA events on the
launching stream; the JSON line reports the mean.  ``e2e`` repeats the
measurement through the same C-ABI call with the operands in pinned host
memory: every step copies A and B in and C out, pipelined so that a step's
copies overlap its neighbours' products (the serial figure is reported beside
it).

Under torchrun (N > 1) every rank runs an independent replica of the product
on its own GPU (the product has no exchange step); ``value`` is the FLOPs of
all ranks over the slowest rank's time.

``--impl reference`` times the CPU oracle instead (rank 0 only), each step a
bounded sample of rows of the same product, on all host cores.
"""
from __future__ import annotations

import argparse
import json
import math
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

from tiled_matrix_multiply_gb300 import inputs, tiling_model  # noqa: E402

METRIC = "FP32 GEMM TFLOP/s at M=N=K=4096 on 1 GB300; % of FP32 (or tensor-pipe) roofline"
UNIT = "TFLOP/s"
FFMA_PER_CLK_PER_SM = 128          # 4 sub-partitions x 32 FP32 lanes
FALLBACK_SM_MAX_MHZ = 2070.0


# -- distributed plumbing ---------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_over_ranks(dist, local_ms: float, local_flops: float):
    """(max time over ranks, summed FLOPs) -- the whole-job aggregate."""
    if dist is None:
        return local_ms, local_flops
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    f = torch.tensor([local_flops], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(f, op=dist.ReduceOp.SUM)
    return float(t.item()), float(f.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# -- clocks -------------------------------------------------------------------------------

CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
REASON_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs."""

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self._thr = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={','.join(CLOCK_FIELDS)}",
               "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self._thr = threading.Thread(target=self._read, daemon=True)
        self._thr.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._thr:
            self._thr.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(CLOCK_FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(REASON_NAMES, parts[4:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# -- peaks ----------------------------------------------------------------------------------

def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return {}


def ffma_peak_tflops(sm_count: int, peaks: dict) -> tuple[float, str]:
    """SMs x 128 FFMA/clk x 2 FLOP x maximum SM clock."""
    mhz = peaks.get("sm_max_mhz")
    src = "MEASURED_PEAKS.json sm_max_mhz"
    if not mhz:
        mhz, src = FALLBACK_SM_MAX_MHZ, "fallback 2070 MHz"
    return sm_count * FFMA_PER_CLK_PER_SM * 2 * mhz * 1e6 / 1e12, \
        f"{sm_count} SMs x 128 FFMA/clk x 2 FLOP x {mhz:.0f} MHz ({src})"


KERNEL_SOURCES = {"gemm_simt": ["gemm_simt.cu"], "gemm_tc3": ["gemm_tc3.cu"],
                  "tc3_split_a": ["gemm_tc3.cu"], "tc3_split_b": ["gemm_tc3.cu"],
                  "window_sum": ["window_sum.cu"], "sum_partials": ["reduce_softmax.cu"],
                  "softmax_staged": ["reduce_softmax.cu"], "softmax_grid": ["reduce_softmax.cu"]}


def recorded_traffic(kernel: str, workload: str, units: int | None = None):
    """DRAM bytes per launch from the committed ncu capture, if the kernel is unchanged since.

    A capture taken on a smaller case of a bandwidth-bound kernel records the
    units (elements) it processed; its traffic is scaled to `units`, since
    such a kernel's traffic grows in proportion to its input."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(f"{kernel}/{workload}")
    if not rec:
        return None
    from tiled_matrix_multiply_gb300 import build
    if rec.get("source_sha") != build.source_digest(KERNEL_SOURCES[kernel]):
        return None
    traffic = rec.get("dram_bytes_per_launch")
    if traffic is not None and units is not None and rec.get("units"):
        traffic = traffic * units / rec["units"]
    return traffic


# -- the oracle as the CPU baseline / reference arm ---------------------------------------------

def oracle_sample(A: np.ndarray, B: np.ndarray, rows: int, threads: int) -> float:
    """Seconds the oracle takes for the first `rows` rows of C = A x B."""
    import oracle
    t0 = time.perf_counter()
    oracle.gemm(A[:rows], B, threads=threads)
    return time.perf_counter() - t0


def calibrate_rows(A, B, threads: int, target_s: float) -> tuple[int, float]:
    """Rows of C whose oracle time is about target_s (at least one row per thread)."""
    M = A.shape[0]
    rows = min(M, max(threads, 1))
    t = oracle_sample(A, B, rows, threads)
    while t < 0.2 * target_s and rows < M:
        rows = min(M, rows * 4)
        t = oracle_sample(A, B, rows, threads)
    want = int(rows * target_s / max(t, 1e-9))
    want = max(threads, (want // threads) * threads)
    return min(M, want), t / rows


def cpu_baseline(A, B, w, target_s=10.0) -> dict:
    """The oracle on the first rows of the product (all of it if that is quick), repeated to
    about target_s seconds of wall time."""
    import oracle
    threads = oracle.default_threads()
    rows, _ = calibrate_rows(A, B, threads, min(2.0, target_s / 5))
    rows = min(w.M, max(threads, int(rows * target_s / 2.0) // threads * threads))
    reps, total = 0, 0.0
    while reps == 0 or total < 0.8 * target_s:
        total += oracle_sample(A, B, rows, threads)
        reps += 1
    t = total / reps
    flops = 2.0 * rows * w.N * w.K
    return {"value": flops / t / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {rows} of {w.M} rows of C ({rows}x{w.N}x{w.K}, FP64 accumulation), "
                      f"{reps} run(s), {t:.2f} s each on {threads} OpenMP threads"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    w = inputs.WORKLOADS[args.workload]
    A, B = inputs.workload_operands(w)
    threads = oracle.default_threads()
    total_steps = args.steps + args.warmup
    per_step = max(0.05, min(5.0, 90.0 / total_steps))
    rows, _ = calibrate_rows(A, B, threads, per_step)
    for _ in range(args.warmup):
        oracle_sample(A, B, rows, threads)
    times = [oracle_sample(A, B, rows, threads) for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(times)
    flops = 2.0 * rows * w.N * w.K
    value = flops / (ms / 1e3) / 1e12
    sample = (f"each step: first {rows} of {w.M} rows of C ({rows}x{w.N}x{w.K}), "
              f"FP64 accumulation on {threads} OpenMP threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, "CPU oracle (row sample)"),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, path: str) -> dict:
    return {"workload": f"{w.name}: {w.describe()}", "M": w.M, "N": w.N, "K": w.K,
            "layout": "row-major, lda=K, ldb=N, ldc=N", "path": path,
            "l2": "flushed before every step (memset of 2x L2 bytes, outside the events)"}


# -- the GPU arm ------------------------------------------------------------------------------

def time_device(step_fn, flush_fn, steps: int, warmup: int, stream, dist) -> list[float]:
    """Per-step device times (ms) of step_fn, L2 flushed before each step."""
    import torch
    for _ in range(warmup):
        flush_fn()
        step_fn()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush_fn()
        starts[i].record(stream)
        step_fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def e2e_pipelined(A_pin, B_pin, w, dev, stream, steps: int, warmup: int, dist) -> float:
    """Mean ms per step of `steps` host-to-host products (pinned A, B in; C out) through
    gemm_f32, pipelined over two device slots: copies in on one stream, the product on
    `stream`, copies out on a third, ordered by events."""
    import torch
    from tiled_matrix_multiply_gb300 import _abi
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    slots = [(torch.empty((w.M, w.K), dtype=torch.float32, device=dev),
              torch.empty((w.K, w.N), dtype=torch.float32, device=dev),
              torch.empty((w.M, w.N), dtype=torch.float32, device=dev)) for _ in range(2)]
    outs = [torch.empty((w.M, w.N), dtype=torch.float32).pin_memory() for _ in range(2)]

    def run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_mm = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            a, b, c = slots[i % 2]
            if i >= 2:
                s_in.wait_event(ev_mm[i - 2])          # slot i % 2's inputs are free
            with torch.cuda.stream(s_in):
                a.copy_(A_pin, non_blocking=True)
                b.copy_(B_pin, non_blocking=True)
            ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])       # slot i % 2's result has left
            _abi.check("gemm_f32", w.M, w.N, w.K, a.data_ptr(), w.K, b.data_ptr(), w.N,
                       c.data_ptr(), w.N, stream.cuda_stream)
            ev_mm[i].record(stream)
            s_out.wait_event(ev_mm[i])
            with torch.cuda.stream(s_out):
                outs[i % 2].copy_(c, non_blocking=True)
            ev_out[i].record(s_out)

    run(max(warmup, 3))
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    run(steps)
    end.record(s_out)          # after the last copy out, which follows every earlier step
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def run_ours(args, world, rank, local):
    import torch
    import tiled_matrix_multiply_gb300 as tmm
    from tiled_matrix_multiply_gb300 import _abi, build

    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}), flush=True)
        return 1
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    build.build()
    _abi.load()

    w = inputs.WORKLOADS[args.workload]
    A_h, B_h = inputs.workload_operands(w)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    stream = torch.cuda.current_stream(dev)
    A = torch.from_numpy(A_h).to(dev)
    B = torch.from_numpy(B_h).to(dev)
    C = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20) or (128 << 20))
    flush_buf = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    launches = {"n": 0}

    def step():
        _abi.check("gemm_f32", w.M, w.N, w.K, A.data_ptr(), w.K, B.data_ptr(), w.N,
                   C.data_ptr(), w.N, stream.cuda_stream)
        launches["n"] += 1

    def flush():
        flush_buf.zero_()

    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid else None)
    sampler.start()
    time.sleep(0.3)
    launches["n"] = 0
    times = time_device(step, flush, args.steps, args.warmup, stream, dist)
    timed_launches = launches["n"] - args.warmup
    clocks = sampler.stop()
    local_ms = statistics.mean(times)
    ms, total_flops = reduce_over_ranks(dist, local_ms, float(w.flops))
    value = total_flops / (ms / 1e3) / 1e12

    # End to end through the same call: pinned host operands in, result out, per step.
    A_pin = torch.from_numpy(A_h).pin_memory()
    B_pin = torch.from_numpy(B_h).pin_memory()
    C_pin = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()

    def e2e_step():
        A.copy_(A_pin, non_blocking=True)
        B.copy_(B_pin, non_blocking=True)
        step()
        C_pin.copy_(C, non_blocking=True)

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 50))
        # Serial: each step copies in, multiplies, copies out, one after another.
        serial_times = time_device(e2e_step, flush, e2e_steps, args.warmup, stream, dist)
        serial_ms, serial_flops = reduce_over_ranks(dist, statistics.mean(serial_times),
                                                    float(w.flops))
        # Pipelined: the same per-step work with step i+1's inputs copied in and step
        # i-1's result copied out while step i multiplies (two device slots, three streams).
        pipe_ms = e2e_pipelined(A_pin, B_pin, w, dev, stream, e2e_steps, args.warmup, dist)
        e2e_ms, e2e_flops = reduce_over_ranks(dist, pipe_ms, float(w.flops))
        e2e = {"value": e2e_flops / (e2e_ms / 1e3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": A_h.nbytes + B_h.nbytes,
               "d2h_bytes_per_step": w.M * w.N * 4, "ms_per_step": e2e_ms,
               "steps": e2e_steps,
               "schedule": "pipelined: H2D of step i+1 and D2H of step i-1 overlap step i's "
                           "gemm_f32; one event pair around all steps, every step's copies inside",
               "serial_ms_per_step": serial_ms,
               "serial_value": serial_flops / (serial_ms / 1e3) / 1e12}

    # The same steps with L2 left warm (no flush), after the timed region.
    warm_times = time_device(step, lambda: None, max(3, min(args.steps, 50)), args.warmup,
                             stream, dist)
    warm_ms, warm_flops = reduce_over_ranks(dist, statistics.mean(warm_times), float(w.flops))
    warm = {"value": warm_flops / (warm_ms / 1e3) / 1e12, "unit": UNIT, "ms_per_step": warm_ms,
            "steps": len(warm_times), "l2": "not flushed between steps"}

    # Roofline of the one kernel a step launches.
    peaks = measured_peaks()
    peak, peak_src = ffma_peak_tflops(props.multi_processor_count, peaks)
    achieved = w.flops / (local_ms / 1e3) / 1e12
    roofline = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "traffic": recorded_traffic("gemm_simt", w.name),
                "peak_source": peak_src,
                "algorithmic": f"2MNK = {w.flops:.4e} FLOP per launch",
                "frac_at_measured_clock": (achieved / (peak * clocks["sm_mhz"] /
                                                       (peaks.get("sm_max_mhz") or
                                                        FALLBACK_SM_MAX_MHZ))
                                           if clocks.get("sm_mhz") else None)}

    extra = {}
    gpu_id = f"GPU-{uuid}" if uuid else None
    sm_count = props.multi_processor_count
    if not args.no_tc3 and rank == 0:
        extra["tc3"] = tc3_leg(args, w, A, B, C, flush, stream, peaks, gpu_id, sm_count)
    if not args.no_layouts and rank == 0:
        extra["layouts"] = layouts_leg(args, w, A, B, C, flush, stream)
    if not args.no_window and rank == 0:
        extra["window5"] = window_leg(args, flush, stream, peaks)
    if not args.no_reduce and rank == 0:
        extra.update(reduction_legs(args, flush, stream, peaks))
    if not args.no_contrast and rank == 0:
        extra["contrast"] = contrast_paths(args, w, A, B, C, flush, stream, props, peaks)
    if not args.no_configs and rank == 0:
        extra["configs"] = configs_leg(args, flush, stream, peaks, gpu_id, sm_count)

    if rank == 0:
        cpu = (cpu_baseline(A_h, B_h, w, args.cpu_seconds)
               if world == 1 and args.cpu_seconds > 0 else None)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": workload_config(w, "gemm_f32 (tiled SIMT FFMA)"),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": timed_launches,
            "ms_per_step_min": min(times), "ms_per_step_max": max(times),
            "ms_per_step_median": statistics.median(times),
            "warm_l2": warm,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


TF32_PER_BF16 = 1.1 / 2.25       # nominal dense TF32 / BF16 tensor rates of the part
TF32_FLOP_PER_CLK_PER_SM = 4096   # dense TF32 tensor FLOP per clock per SM (ncu's instruction rate)


def tf32_peak(peaks) -> tuple[float, str]:
    bf16 = peaks.get("bf16_tflops")
    if bf16:
        return bf16 * TF32_PER_BF16, ("MEASURED_PEAKS.json bf16_tflops x 1.1/2.25 (nominal "
                                      "TF32/BF16 dense ratio)")
    return 1900.0 * TF32_PER_BF16, "fallback 1.9 PFLOP/s bf16 x 1.1/2.25"


def tf32_instruction_rate(sm_count: int, mhz) -> float | None:
    """TF32 tensor FLOP/s at the sampled SM clock: 4096 FLOP per clock per SM."""
    return sm_count * TF32_FLOP_PER_CLK_PER_SM * mhz * 1e6 / 1e12 if mhz else None


def tc3_traffic(workload: str):
    """DRAM bytes of one gemm_f32_tc3 step: the product kernel and both split
    kernels, each from its committed ncu capture (None unless all three are
    recorded for the current sources)."""
    parts = {k: recorded_traffic(k, workload)
             for k in ("gemm_tc3", "tc3_split_a", "tc3_split_b")}
    total = sum(parts.values()) if all(v is not None for v in parts.values()) else None
    return total, parts


def tc3_leg(args, w, A, B, C, flush, stream, peaks, gpu_id, sm_count) -> dict:
    """gemm_f32_tc3 on the same workload: three TF32 tensor-core products per
    output term; reported as effective FP32 TFLOP/s and against the TF32 pipe."""
    import torch
    from tiled_matrix_multiply_gb300 import _abi
    lib = _abi.load()
    need = int(lib.gemm_f32_tc3_workspace_size(w.M, w.N, w.K))
    ws = torch.empty(need + 256, dtype=torch.uint8, device=A.device)
    wptr = (ws.data_ptr() + 255) // 256 * 256
    launches = {"n": 0}

    def step():
        rc = lib.gemm_f32_tc3(w.M, w.N, w.K, A.data_ptr(), w.K, B.data_ptr(), w.N, C.data_ptr(),
                              w.N, wptr, need, stream.cuda_stream)
        if rc != _abi.TMM_OK:
            raise _abi.TmmError("gemm_f32_tc3", rc, _abi.last_error())
        launches["n"] += 3   # split of A, split of B, product kernel

    steps = max(3, min(args.steps, 200))
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)
    launches["n"] = 0
    times = time_device(step, flush, steps, args.warmup, stream, None)
    clocks = sampler.stop()
    if lib.tmm_check_device(stream.cuda_stream) != _abi.TMM_OK:
        raise _abi.TmmError("tmm_check_device", _abi.TMM_ERR_DEVICE_TIMEOUT, _abi.last_error())
    ms = statistics.mean(times)
    peak, peak_src = tf32_peak(peaks)
    tensor_tflops = 3 * w.flops / (ms / 1e3) / 1e12
    inst_rate = tf32_instruction_rate(sm_count, clocks.get("sm_mhz"))
    traffic, traffic_parts = tc3_traffic(w.name)
    return {"path": "gemm_f32_tc3 (tcgen05, 3 x TF32 split products, FP32 accumulation)",
            "value": w.flops / (ms / 1e3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "steps": steps, "gpu_launches": launches["n"] - 3 * args.warmup,
            "workspace_bytes": need, "clocks": clocks,
            "roofline": {"bound": "tensor", "achieved": tensor_tflops, "peak": peak, "unit": UNIT,
                         "frac": tensor_tflops / peak,
                         "frac_at_instruction_rate": (tensor_tflops / inst_rate
                                                      if inst_rate else None),
                         "instruction_rate": inst_rate,
                         "instruction_rate_source": (f"{sm_count} SMs x 4096 TF32 FLOP/clk x "
                                                     "median sampled SM clock"),
                         "traffic": traffic, "traffic_parts": traffic_parts,
                         "peak_source": peak_src,
                         "algorithmic": f"3 x 2MNK = {3 * w.flops:.4e} tensor FLOP per step "
                                        "(split pre-pass included in the step time; traffic "
                                        "counts the split kernels and the product kernel)"}}


#: The workloads of the configs leg: every product configuration, at full size.
CONFIG_WORKLOADS = ["square256", "square1024", "square4096", "ragged4000x3001x2047",
                    "rect8192x8192x1024", "rect16384x1024x4096", "rect1024x16384x4096",
                    "square8192"]


def configs_leg(args, flush, stream, peaks, gpu_id, sm_count) -> dict:
    """Every product configuration at full size, operands in HBM, L2 flushed before
    every step: gemm_f32 (FFMA roofline) and gemm_f32_tc3 (TF32 tensor roofline), and
    gemm_f32_naive where a few of its steps take well under a second.  Steps per
    configuration are sized to about 0.2 s of work per path (5 to 50)."""
    import torch
    from tiled_matrix_multiply_gb300 import _abi
    lib = _abi.load()
    ffma_peak, ffma_src = ffma_peak_tflops(sm_count, peaks)
    tf32, tf32_src = tf32_peak(peaks)
    out = {"peaks": {"gemm_f32": ffma_peak, "gemm_f32_source": ffma_src,
                     "gemm_f32_tc3": tf32, "gemm_f32_tc3_source": tf32_src,
                     "unit": UNIT},
           "l2": "flushed before every step (memset of 2x L2 bytes, outside the events)"}
    sampler = ClockSampler(gpu_id)
    sampler.start()
    for name in CONFIG_WORKLOADS:
        w = inputs.WORKLOADS[name]
        A_h, B_h = inputs.workload_operands(w)
        dev = torch.device("cuda", torch.cuda.current_device())
        A = torch.from_numpy(A_h).to(dev)
        B = torch.from_numpy(B_h).to(dev)
        C = torch.empty((w.M, w.N), dtype=torch.float32, device=dev)
        need = int(lib.gemm_f32_tc3_workspace_size(w.M, w.N, w.K))
        ws = torch.empty(need + 256, dtype=torch.uint8, device=dev)
        wptr = (ws.data_ptr() + 255) // 256 * 256
        s = stream.cuda_stream

        def simt():
            _abi.check("gemm_f32", w.M, w.N, w.K, A.data_ptr(), w.K, B.data_ptr(), w.N,
                       C.data_ptr(), w.N, s)

        def tc3():
            rc = lib.gemm_f32_tc3(w.M, w.N, w.K, A.data_ptr(), w.K, B.data_ptr(), w.N,
                                  C.data_ptr(), w.N, wptr, need, s)
            if rc != _abi.TMM_OK:
                raise _abi.TmmError("gemm_f32_tc3", rc, _abi.last_error())

        def naive():
            _abi.check("gemm_f32_naive", w.M, w.N, w.K, A.data_ptr(), w.K, B.data_ptr(), w.N,
                       C.data_ptr(), w.N, s)

        rec = {"M": w.M, "N": w.N, "K": w.K, "workload": w.describe()}
        for label, fn, rate, peak in (("gemm_f32", simt, 60e12, ffma_peak),
                                      ("gemm_f32_tc3", tc3, 250e12, tf32 / 3),
                                      ("gemm_f32_naive", naive, 6e12, ffma_peak)):
            est_s = w.flops / rate
            if label == "gemm_f32_naive" and est_s > 0.05:
                continue
            steps = int(min(50, max(5, 0.2 / est_s)))
            ms = statistics.mean(time_device(fn, flush, steps, 3, stream, None))
            tflops = w.flops / (ms / 1e3) / 1e12
            rec[label] = {"value": tflops, "unit": UNIT, "ms_per_step": ms, "steps": steps,
                          "frac": tflops / peak}
            if label == "gemm_f32_tc3":
                rec[label]["frac_note"] = "effective FP32 TFLOP/s over (TF32 peak / 3)"
        if lib.tmm_check_device(s) != _abi.TMM_OK:
            raise _abi.TmmError("tmm_check_device", _abi.TMM_ERR_DEVICE_TIMEOUT,
                                _abi.last_error())
        out[name] = rec
        del A, B, C, ws
        torch.cuda.empty_cache()
    clocks = sampler.stop()
    out["clocks"] = clocks
    inst = tf32_instruction_rate(sm_count, clocks.get("sm_mhz"))
    if inst:
        for name in CONFIG_WORKLOADS:
            r = out[name].get("gemm_f32_tc3")
            if r:
                r["frac_at_instruction_rate"] = 3 * r["value"] / inst
    return out


def layouts_leg(args, w, A, B, C, flush, stream) -> dict:
    """The same product with A and/or B stored transposed (gemm_f32_ex, gemm_f32_tc3_ex):
    op(A) = A^T reads A stored K x M, the layout of "CMU DLSys Lecture 12" section 4."""
    import torch
    from tiled_matrix_multiply_gb300 import _abi
    lib = _abi.load()
    At = A.t().contiguous()     # stored K x M
    Bt = B.t().contiguous()     # stored N x K
    need = int(lib.gemm_f32_tc3_workspace_size(w.M, w.N, w.K))
    ws = torch.empty(need + 256, dtype=torch.uint8, device=A.device)
    wptr = (ws.data_ptr() + 255) // 256 * 256
    out = {}
    steps = max(3, min(args.steps, 50))
    for name, ta, tb in (("tn", 1, 0), ("nt", 0, 1), ("tt", 1, 1)):
        a, lda = (At, w.M) if ta else (A, w.K)
        b, ldb = (Bt, w.K) if tb else (B, w.N)

        def simt():
            rc = lib.gemm_f32_ex(ta, tb, w.M, w.N, w.K, a.data_ptr(), lda, b.data_ptr(), ldb,
                                 C.data_ptr(), w.N, stream.cuda_stream)
            assert rc == _abi.TMM_OK, _abi.last_error()

        def tc3():
            rc = lib.gemm_f32_tc3_ex(ta, tb, w.M, w.N, w.K, a.data_ptr(), lda, b.data_ptr(), ldb,
                                     C.data_ptr(), w.N, wptr, need, stream.cuda_stream)
            assert rc == _abi.TMM_OK, _abi.last_error()
        rec = {}
        for label, fn in (("gemm_f32_ex", simt), ("gemm_f32_tc3_ex", tc3)):
            ms = statistics.mean(time_device(fn, flush, steps, args.warmup, stream, None))
            rec[label] = {"value": w.flops / (ms / 1e3) / 1e12, "unit": UNIT, "ms_per_step": ms}
        out[name] = rec
    return {"steps": steps, "transa_transb": {"tn": [1, 0], "nt": [0, 1], "tt": [1, 1]}, **out}


AUX_LOG2N = 28     # the window, sum and softmax legs each move 2^28 floats per call by default


def window_leg(args, flush, stream, peaks) -> dict:
    """window_sum_f32 ("CMU DLSys Lecture 12" section 3, W = 5) on 2^28 outputs:
    HBM-bound, 4 (n + W - 1) bytes read and 4 n written per call."""
    import torch
    from tiled_matrix_multiply_gb300 import _abi
    lib = _abi.load()
    W = 5
    n = 1 << args.aux_log2n
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.rand(n + W - 1, device="cuda", generator=g)
    y = torch.empty(n, device="cuda")

    def step():
        rc = lib.window_sum_f32(n, W, x.data_ptr(), y.data_ptr(), stream.cuda_stream)
        assert rc == _abi.TMM_OK, _abi.last_error()
    steps = max(3, min(args.steps, 100))
    ms = statistics.mean(time_device(step, flush, steps, args.warmup, stream, None))
    nbytes = 4 * (n + W - 1) + 4 * n
    gbs = nbytes / (ms / 1e3) / 1e9
    peak = peaks.get("hbm_gbs") or 6800.0
    del x, y
    torch.cuda.empty_cache()
    return {"workload": f"window sum W={W}, n=2^{args.aux_log2n} outputs, uniform[0,1) floats",
            "ms_per_step": ms, "value": gbs, "unit": "GB/s", "steps": steps,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak,
                         "traffic": recorded_traffic("window_sum", "w5", n),
                         "peak_source": ("MEASURED_PEAKS.json hbm_gbs" if peaks.get("hbm_gbs")
                                         else "fallback 6.8 TB/s"),
                         "algorithmic": f"4 (n + W - 1) + 4 n = {nbytes} bytes per call"}}


SOFTMAX_COLS = 4096
GRID_ROW_COLS = 65537   # rows this long or longer run softmax_grid_kernel


def _hbm_roofline(gbs, peaks, nbytes, what, traffic=None):
    peak = peaks.get("hbm_gbs") or 6800.0
    return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
            "traffic": traffic,
            "peak_source": ("MEASURED_PEAKS.json hbm_gbs" if peaks.get("hbm_gbs")
                            else "fallback 6.8 TB/s"),
            "algorithmic": f"{what} = {nbytes} bytes per call"}


def reduction_legs(args, flush, stream, peaks) -> dict:
    """sum_f32 over 2^28 floats and softmax_rows_f32 over 65536 rows of 4096 logits (by default)
    ("Tiling Strategies" section 5): HBM-bound, each input read once."""
    import torch
    from tiled_matrix_multiply_gb300 import _abi
    lib = _abi.load()
    steps = max(3, min(args.steps, 100))
    g = torch.Generator(device="cuda").manual_seed(6)
    out = {}

    n = 1 << args.aux_log2n
    x = torch.randn(n, device="cuda", generator=g)
    res = torch.empty(1, device="cuda")
    need = int(lib.sum_f32_workspace_size(n))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def sum_step():
        rc = lib.sum_f32(n, x.data_ptr(), res.data_ptr(), ws.data_ptr(), need,
                         stream.cuda_stream)
        assert rc == _abi.TMM_OK, _abi.last_error()
    ms = statistics.mean(time_device(sum_step, flush, steps, args.warmup, stream, None))
    nbytes = 4 * n
    gbs = nbytes / (ms / 1e3) / 1e9
    out["sum"] = {"workload": f"array sum, n = 2^{args.aux_log2n} standard-normal floats",
                  "ms_per_step": ms,
                  "value": gbs, "unit": "GB/s", "steps": steps, "launches_per_step": 2,
                  "roofline": _hbm_roofline(gbs, peaks, nbytes, "4 n",
                                            recorded_traffic("sum_partials", "normal", n))}
    del x, ws, res
    torch.cuda.empty_cache()

    cols = args.softmax_cols
    rows = max(1, (1 << args.aux_log2n) // cols)
    xs = torch.randn(rows, cols, device="cuda", generator=g) * 4
    ys = torch.empty_like(xs)

    def softmax_step():
        rc = lib.softmax_rows_f32(rows, cols, xs.data_ptr(), cols, ys.data_ptr(), cols,
                                  stream.cuda_stream)
        assert rc == _abi.TMM_OK, _abi.last_error()
    ms = statistics.mean(time_device(softmax_step, flush, steps, args.warmup, stream, None))
    nbytes = 8 * rows * cols
    gbs = nbytes / (ms / 1e3) / 1e9
    out["softmax"] = {"workload": f"row softmax, {rows} rows x {cols} cols, N(0, 16) logits",
                      "ms_per_step": ms, "value": gbs, "unit": "GB/s", "steps": steps,
                      "rows_per_s": rows / (ms / 1e3),
                      "roofline": _hbm_roofline(
                          gbs, peaks, nbytes, "4 rows cols read + 4 rows cols written",
                          recorded_traffic("softmax_grid" if cols >= GRID_ROW_COLS
                                           else "softmax_staged", f"cols{cols}", rows * cols))}
    return out


def contrast_paths(args, w, A, B, C, flush, stream, props, peaks) -> dict:
    """The naive kernel on the same workload (a few steps): the untiled contrast."""
    import torch
    from tiled_matrix_multiply_gb300 import _abi

    def naive():
        _abi.check("gemm_f32_naive", w.M, w.N, w.K, A.data_ptr(), w.K, B.data_ptr(), w.N,
                   C.data_ptr(), w.N, stream.cuda_stream)
    t = time_device(naive, flush, 3, 1, stream, None)
    ms = statistics.mean(t)
    return {"gemm_f32_naive": {"ms_per_step": ms, "value": w.flops / (ms / 1e3) / 1e12,
                               "unit": UNIT,
                               "logical_operand_bytes": 4 * tiling_model.q_naive(w.M, w.N, w.K)}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=inputs.HEADLINE, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="oracle CPU-baseline budget; 0 skips the CPU baseline")
    ap.add_argument("--no-contrast", action="store_true", help="skip the naive-kernel contrast")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-tc3", action="store_true", help="skip the tensor-core (3xTF32) leg")
    ap.add_argument("--no-window", action="store_true", help="skip the window-sum leg")
    ap.add_argument("--no-reduce", action="store_true", help="skip the sum and softmax legs")
    ap.add_argument("--aux-log2n", type=int, default=AUX_LOG2N,
                    help="log2 of the floats each window/sum/softmax call moves (default 28; "
                         "smaller for profiler captures)")
    ap.add_argument("--softmax-cols", type=int, default=SOFTMAX_COLS,
                    help="row length of the softmax leg (default 4096)")
    ap.add_argument("--no-layouts", action="store_true",
                    help="skip the transposed-layout (gemm_f32_ex, gemm_f32_tc3_ex) leg")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the leg that times every product configuration")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)   # at least three untimed warm-up steps, always
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())

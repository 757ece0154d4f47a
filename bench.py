#!/usr/bin/env python
"""Benchmark of the sub-bit weight products on B300. Prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Default workload (the headline metric's configuration): ternary decode
product M=1, K=5120, N=17408 ("batch-1 packed-weight GB/s"). A step is one
pass of the decode kernel over one weight matrix; the timed loop rotates
through enough distinct weight replicas that the working set exceeds L2.
Other workloads (--workload): bin_gemv_1k, sweep_ter, sweep_bin, gemm512_ter,
gemm512_bin, gemm4096_ter, gemm4096_bin, xnor.

Multi-GPU: the path has no exchange step, so N GPUs run N independent
replicas (weak scaling); rank 0 prints the whole-job throughput over the
max-over-ranks time. --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 packed-weight GB/s (% HBM peak); 64-layer tok/s; pp512 TFLOP/s"
L2_BYTES = 126 * 2 ** 20


# ------------------------------------------------------------------ helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"],
                "bf16_sustained": d["bf16_tflops_sustained"], "src": "measured"}
    return {"hbm": 6400.0, "bf16": 1800.0, "bf16_sustained": 1400.0, "src": "fallback"}


class ClockSampler:
    """NVML samples of SM clock and throttle reasons during the timed region."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, index):
        self.samples, self.reasons, self.stop_flag = [], 0, False
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
        except Exception:
            self.nv = None
            self.max_mhz = None

    def _one(self):
        try:
            self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
            self.reasons |= self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
        except Exception:
            pass

    def _run(self):
        while not self.stop_flag:
            self._one()
            time.sleep(0.01)

    def __enter__(self):
        if self.nv:
            self._one()
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *a):
        if self.nv:
            self.stop_flag = True
            self.t.join()
            self._one()

    def report(self):
        if not self.nv or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["nvml unavailable"]}
        names = [v for k, v in self.REASONS.items() if self.reasons & k and k != 0x1]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "samples": len(self.samples), "reasons": names}


def dist_setup(ngpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- workloads
class GemvWorkload:
    """Decode product M=1 over rotating weight replicas."""

    def __init__(self, fmt, n, k, cfg_id, name):
        self.fmt, self.n, self.k, self.cfg_id, self.name = fmt, n, k, cfg_id, name

    def unit_bytes(self):
        import sub_bit_weight_binary_b300 as sb
        rb = sb.bonsai_packed_row_bytes(self.fmt, self.k)
        return self.n * rb + self.n * (self.k // 128) * 2  # packed + scales

    def setup(self):
        import torch
        import sub_bit_weight_binary_b300 as sb
        from sub_bit_weight_binary_b300 import synth, synth_device as sd
        seed = synth.config_seed(self.cfg_id)
        n, k = self.n, self.k
        self.reps = max(1, math.ceil(2 * L2_BYTES / self.unit_bytes()) + 1)
        rb = sb.bonsai_packed_row_bytes(self.fmt, k)
        self.w = []
        codes = torch.empty(n * k, dtype=torch.int8, device="cuda") \
            if self.fmt == sb.BONSAI_FMT_TERNARY else None
        for r in range(self.reps):
            tid = synth.TID_WTER if self.fmt == sb.BONSAI_FMT_TERNARY else synth.TID_WBIN
            packed = torch.empty((n, rb), dtype=torch.uint8, device="cuda")
            if self.fmt == sb.BONSAI_FMT_TERNARY:
                sd.ternary_codes(seed, tid + 64 * r, 0, codes)
                sb.bonsai_pack_ternary(codes.view(n, k), packed)
            else:
                sd.bits32(seed, tid + 64 * r, 0, packed.view(torch.int32))
            scales = torch.empty((n, k // 128), dtype=torch.float16, device="cuda")
            sd.uniform_f16(seed, synth.TID_SCALES + 64 * r, 0, 0.01, 0.05, scales)
            self.w.append(sb.Weights(self.fmt, n, k, packed, scales, sb.BONSAI_WEIGHTS_PREFETCH))
        x = synth.gen_x(seed, 1, k)
        self.x_host = torch.from_numpy(x.view(np.float16)[0]).pin_memory()
        self.x = self.x_host.cuda()
        self.y = torch.empty(n, dtype=torch.float16, device="cuda")
        self.y_host = torch.empty(n, dtype=torch.float16).pin_memory()
        torch.cuda.synchronize()
        sb.check()

    def step(self, i):
        import sub_bit_weight_binary_b300 as sb
        sb.bonsai_gemv(self.w[i % self.reps], self.x, self.y)

    def step_e2e(self, i):
        import sub_bit_weight_binary_b300 as sb
        self.x.copy_(self.x_host, non_blocking=True)
        sb.bonsai_gemv(self.w[i % self.reps], self.x, self.y)
        self.y_host.copy_(self.y, non_blocking=True)

    def io_bytes(self):
        return self.k * 2, self.n * 2

    def launches_per_step(self):
        return 1

    def config(self):
        return {"workload": self.name, "m": 1, "k": self.k, "n": self.n,
                "format": "ternary" if self.fmt == 2 else "binary",
                "weights": "synthetic seeded, resident in HBM",
                "l2": "inputs larger than L2: %d rotating weight replicas, %.0f MB" % (
                    self.reps, self.reps * self.unit_bytes() / 1e6)}

    def metric(self, sec_per_step):
        return self.unit_bytes() / sec_per_step / 1e9, "GB/s"

    def roofline(self, sec_per_step, pk):
        a = self.unit_bytes() / sec_per_step / 1e9
        return {"bound": "hbm", "achieved": round(a, 1), "peak": pk["hbm"], "unit": "GB/s",
                "frac": round(a / pk["hbm"], 4), "traffic": None,
                "peak_src": pk["src"] + " burst copy"}

    # CPU oracle on a bounded sample: whole products, repeated for >= 10 s
    def cpu_sample(self, min_seconds=10.0, max_rows=None):
        import oracle
        from sub_bit_weight_binary_b300 import synth
        seed = synth.config_seed(self.cfg_id)
        n, k = self.n, self.k
        rows = min(n, max_rows or n)
        if self.fmt == 2:
            codes = synth.gen_ternary_codes(seed, rows, k)
            packed = oracle.pack_ternary(codes)
        else:
            packed = synth.gen_binary_words(seed, rows, k).view(np.uint8).reshape(rows, -1)
        scales = synth.gen_scales(seed, rows, k)
        x = synth.gen_x(seed, 1, k)
        t0 = time.perf_counter()
        passes = 0
        while True:
            oracle.linear(self.fmt, packed, scales, x)
            passes += 1
            el = time.perf_counter() - t0
            if el >= min_seconds or el > 30:
                break
        bytes_done = passes * rows * (packed.shape[1] + 2 * (k // 128))
        return bytes_done / el / 1e9, "%d pass(es) over %d of %d rows (%.1f s)" % (
            passes, rows, n, el)


WORKLOADS = {
    "ter_gemv": lambda: GemvWorkload(2, 17408, 5120, 2,
                                     "ternary GEMV M=1 K=5120 N=17408 (decode, config 2)"),
    "bin_gemv_1k": lambda: GemvWorkload(1, 1024, 1024, 1,
                                        "binary GEMV M=1 K=1024 N=1024 (decode, config 1)"),
}


# -------------------------------------------------------------------- runs
def run_ours(args, world, rank, wl):
    import torch
    import sub_bit_weight_binary_b300 as sb
    pk = peaks()
    wl.setup()
    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()
    sb.check()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0.record(stream)
        for i in range(args.steps):
            wl.step(i)
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(world, ms)
    sec = ms / 1e3 / args.steps
    val, unit = wl.metric(sec)
    sb.check()

    # end to end through the C ABI with host buffers (copies in the timed region)
    for i in range(args.warmup):
        wl.step_e2e(i)
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    for i in range(args.steps):
        wl.step_e2e(i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(world, e0.elapsed_time(e1))
    e2e_val, _ = wl.metric(ms_e2e / 1e3 / args.steps)
    bi, bo = wl.io_bytes()
    sb.check()

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(val * world, 2), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded counter-based generator; no trained weights)",
        "config": dict(wl.config(), parallelism="replicas only" if world > 1 else "1 GPU"),
        "roofline": wl.roofline(sec, pk),
        "e2e": {"value": round(e2e_val * world, 2), "unit": unit,
                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
        "gpu_launches": wl.launches_per_step() * args.steps,
        "clocks": clk.report(),
    }
    if not args.no_cpu_baseline and world == 1:
        v, sample = wl.cpu_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": unit, "cores": 1, "kind": "oracle",
                                "sample": sample}
    return line


def run_reference(args, world, rank, wl):
    if rank != 0:
        return None
    # the oracle, as it stands, on the machine's host cores; each step is a
    # bounded sample (a row slice) of the workload
    per_step = []
    rows = max(1, min(wl.n, 2048))
    for i in range(args.warmup + args.steps):
        v, _ = wl.cpu_sample(min_seconds=0.0, max_rows=rows)
        if i >= args.warmup:
            per_step.append(v)
    val = statistics.median(per_step)
    sample = "each step: one oracle pass over %d of %d rows" % (rows, wl.n)
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based generator)", "config": wl.config(),
        "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="ter_gemv")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = WORKLOADS[args.workload]()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        line = run_reference(args, world, rank, wl)
    else:
        from sub_bit_weight_binary_b300 import build
        build.build()
        world, rank, _ = dist_setup(args.gpus)
        line = run_ours(args, world, rank, wl)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line))


if __name__ == "__main__":
    main()

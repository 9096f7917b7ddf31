#!/usr/bin/env python
"""Throughput benchmark of the sm_103a FlashAttention-2 forward kernel.

One step = one call of the public C ABI (fa2_fwd / fa2_fwd_gqa) over the whole
workload batch. Default workload: B=4, H=16, N=4096, d=128, bf16, non-causal,
seeded N(0,1) inputs. Metric: attention-forward TFLOP/s counted as 4*B*H*N^2*d
per step. Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

--impl reference times the fp64 CPU oracle (test infrastructure) on the host
cores over a bounded sample of the same workload: a deliberately slow
baseline, not a GPU implementation.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own copy of the
workload (independent batches, no data-path collective: weak scaling); the
ranks meet only at the timing barriers and the max-over-ranks reduction.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import gen  # noqa: E402

DEFAULT_WORKLOAD = "mha_B4_H16_N4096_d128_bf16"
METRIC = "attention fwd TFLOP/s (4BHN²d) at 1 GB300; % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
KERNEL_SOURCES = [
    os.path.join(ROOT, "attention_fa2_forward_03_gb300", "csrc", "fa2_fwd_sm103.cu"),
    os.path.join(ROOT, "attention_fa2_forward_03_gb300", "csrc", "ptx_sm103.cuh"),
]
REASON_FIELDS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ distributed plumbing

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend: str):
        if self.world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if self.pg is None:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float, device=None) -> float:
        if self.pg is None:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def done(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate_throughput(dist, flops: float, region_ms: float, device=None):
    """Whole-job TFLOP/s: the FLOPs of all ranks over the slowest rank's time."""
    max_ms = dist.max(region_ms, device)
    total = dist.sum(flops, device)
    return total / (max_ms * 1e-3) / 1e12, max_ms


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons (every 100 ms)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = [None, None]

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def mark(self, which: int):
        self.window[which] = time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        t0, t1 = self.window
        inside = [s for (t, s) in self.samples if t0 is not None and t0 <= t <= (t1 or t)]
        if not inside:  # region shorter than the sampling period: nearest sample
            mid = ((t0 or 0) + (t1 or 0)) / 2
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        smax = [num(s[2]) for s in inside if num(s[2]) is not None]
        reasons = set()
        for s in inside:
            for name, val in zip(REASON_FIELDS, s[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max((num(s[3]) or 0.0) for s in inside)}


# ------------------------------------------------------------------ peaks and traffic

def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            peaks = json.load(fh)
        return float(peaks["bf16_tflops"]), "measured (bf16_tflops burst, MEASURED_PEAKS.json)"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback (1.9 PFLOP/s bf16 burst)"


def load_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source for this workload; else None."""
    try:
        with open(TRAFFIC_FILE) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_source_sha") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ CPU oracle timing

def oracle_rows_for(w, seconds: float, q, k, v):
    """Rows per second of the fp64 oracle on this host, then a seeded row
    sample sized to take about `seconds`."""
    import oracle

    rng = np.random.default_rng(w.seed)
    total = w.B * w.Hq * w.N
    calib = rng.integers(0, total, 64)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, w.dtype, rows=calib)
    rate = 64 / max(time.perf_counter() - t0, 1e-6)
    n = int(max(1, min(total, rate * seconds)))
    return rng.integers(0, total, n), oracle.max_threads()


def time_oracle(w, q, k, v, seconds: float):
    import oracle

    rows, cores = oracle_rows_for(w, seconds, q, k, v)
    t0 = time.perf_counter()
    oracle.attention(q, k, v, w.scale, w.dtype, rows=rows)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.N * w.d * len(rows)
    return flops / dt / 1e12, cores, len(rows), dt


# ------------------------------------------------------------------ arms

def run_reference(args, dist, w):
    """fp64 CPU oracle as the reference arm: each step a bounded row sample."""
    if dist.rank != 0:
        return None
    import oracle

    q, k, v = w.inputs()
    total_budget = 120.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    rows, cores = oracle_rows_for(w, per_step, q, k, v)
    for _ in range(args.warmup):
        oracle.attention(q, k, v, w.scale, w.dtype, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention(q, k, v, w.scale, w.dtype, rows=rows)
    dt = time.perf_counter() - t0
    value = 4.0 * w.N * w.d * len(rows) * args.steps / dt / 1e12
    sample = (f"{len(rows)} seeded query rows of the {w.B * w.Hq * w.N}-row workload per step "
              f"(full key length N={w.N}); fp64 C oracle, OpenMP")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config_of(w, n_gpus):
    return {"workload": w.name, "B": w.B, "H_q": w.Hq, "H_kv": w.Hkv, "N": w.N, "d": w.d,
            "dtype": "bf16" if w.dtype == gen.BF16 else "fp16",
            "causal": False, "scale": "1/sqrt(d)", "inputs": f"N(0,1)x{w.amp:g} seed {w.seed}",
            "global_batch": w.B * n_gpus, "seq_len": w.N,
            "parallelism": f"replicas x{n_gpus}" if n_gpus > 1 else "single GPU",
            "l2": l2_note(w)}


def qkv_bytes(w) -> int:
    return 2 * w.d * w.N * w.B * (w.Hq + 2 * w.Hkv)


def l2_note(w) -> str:
    mib = qkv_bytes(w) / 2**20
    if qkv_bytes(w) > L2_BYTES:
        return f"inputs larger than L2: Q+K+V = {mib:.0f} MiB > 129 MiB"
    return f"L2 flushed between timed steps (256 MiB write); Q+K+V = {mib:.1f} MiB"


def run_ours(args, dist, w):
    import torch

    from attention_fa2_forward_03_gb300 import fa2

    fa2.load()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    stream = torch.cuda.current_stream(dev)

    q, k, v = w.inputs()
    tdt = torch.bfloat16 if w.dtype == gen.BF16 else torch.float16

    def up(x):
        return torch.from_numpy(x.view(np.int16)).to(dev).view(tdt)

    tq, tk, tv = up(q), up(k), up(v)
    o = torch.empty_like(tq)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)
    flush = None
    if qkv_bytes(w) <= L2_BYTES:
        flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)

    def step():
        rc = fa2.fa2_fwd_gqa_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.d, w.scale, w.dtype,
                                 stream.cuda_stream)
        if rc != fa2.FA2_OK:
            raise RuntimeError(f"fa2_fwd_gqa: {fa2.status_string(rc)}")

    for _ in range(args.warmup):
        if flush is not None:
            flush.zero_()
        step()
    rc = fa2.fa2_check_status(stream.cuda_stream)
    if rc != fa2.FA2_OK:
        raise RuntimeError(f"kernel status {fa2.status_string(rc)}")

    clocks = ClockSampler(dist.local_rank)
    if dist.rank == 0:
        clocks.start()
        time.sleep(0.3)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)

    dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark(0)
    region0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    region1.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    clocks.mark(1)
    region_ms = region0.elapsed_time(region1)
    kernel_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    rc = fa2.fa2_check_status(stream.cuda_stream)
    if rc != fa2.FA2_OK:
        raise RuntimeError(f"kernel status {fa2.status_string(rc)}")
    if dist.rank == 0:
        time.sleep(0.25)
        clocks.stop()

    value, max_region_ms = aggregate_throughput(dist, float(w.flops) * args.steps, region_ms, dev)

    # end to end through the public binding: pinned host inputs -> device ->
    # kernel -> device -> pinned host outputs, every step
    hq, hk, hv = (torch.from_numpy(x.view(np.int16)).view(tdt).pin_memory() for x in (q, k, v))
    ho = torch.empty(o.shape, dtype=tdt).pin_memory()
    hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step():
        tq.copy_(hq, non_blocking=True)
        tk.copy_(hk, non_blocking=True)
        tv.copy_(hv, non_blocking=True)
        fa2.fa2_fwd_gqa(tq, tk, tv, o, lse, scale=w.scale, stream=stream)
        ho.copy_(o, non_blocking=True)
        hl.copy_(lse, non_blocking=True)

    for _ in range(2):
        e2e_step()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    e2e_value, e2e_ms = aggregate_throughput(dist, float(w.flops) * e2e_steps,
                                             e0.elapsed_time(e1), dev)
    h2d = (hq.numel() + hk.numel() + hv.numel()) * 2
    d2h = ho.numel() * 2 + hl.numel() * 4

    result = None
    if dist.rank == 0:
        peak, peak_src = load_peak()
        achieved = w.flops / (kernel_ms * 1e-3) / 1e12
        traffic = load_traffic(w.name)
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": max_region_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == gen.BF16 else "fp16", "data": "synthetic",
            "config": config_of(w, dist.world),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_src,
                         "kernel": f"fa2_fwd_kernel<{w.d},{'bf16' if w.dtype == gen.BF16 else 'fp16'}>",
                         "kernel_ms": kernel_ms,
                         "alg_flops_per_launch": w.flops, "alg_bytes_per_launch": w.alg_bytes,
                         "hbm_gbs_alg": w.alg_bytes / (kernel_ms * 1e-3) / 1e9},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step": e2e_ms / e2e_steps},
            "gpu_launches": args.steps,
            "clocks": clocks.summary(),
        }
        if dist.world == 1 and not args.no_cpu_baseline:
            cv, cores, nrows, dt = time_oracle(w, q, k, v, args.cpu_seconds)
            result["cpu_baseline"] = {
                "value": cv, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": (f"{nrows} seeded query rows of the {w.B * w.Hq * w.N}-row workload, "
                           f"full key length N={w.N}; fp64 C oracle, OpenMP, {dt:.1f} s")}
    return result


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(gen.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    dist = Dist()
    w = gen.workload(args.workload)
    if args.impl == "reference":
        res = run_reference(args, dist, w)
    else:
        res = run_ours(args, dist, w)
    if res is not None and dist.rank == 0:
        print(json.dumps(res), flush=True)
    dist.done()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Throughput benchmark of the sm_103a FlashAttention-2 forward kernel.

One step = one call of the public C ABI (fa2_fwd / fa2_fwd_gqa) over the whole
workload batch. Default workload: B=4, H=16, N=4096, d=128, bf16, non-causal,
seeded N(0,1) inputs. Metric: attention-forward TFLOP/s counted as 4*B*H*N^2*d
per step. Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--pass fwd|fwd_causal|bwd|bwd_causal]
                    [--impl ours|reference] [--no-cpu-baseline] [--all-configs]

--all-configs runs every forward workload configuration in turn (the tiny
case, the B4 H16 N4096 headline, the twelve sequence-sweep points, the
sharper-softmax d=64 case and the grouped-KV case) and prints one JSON line
for each, then one line per sweep dtype with the harmonic mean of its six
points (the averaging the Ampere series' Performance section uses).

--pass picks what one step runs (default fwd, the line above):
  fwd_causal  fa2_fwd_ex (fa2_fwd_fp8_ex for an FP8 workload) with the
              causal mask; FLOPs counted over the unmasked (query, key)
              pairs only, 4*d*sum_i(i+1) per head
  bwd         fa2_bwd (D = rowsum(dO*O), then dK/dV, then dQ: three
              launches); FLOPs counted as 2.5x the forward's (the five
              GEMMs of the backward), inputs from one forward call
  bwd_causal  the same with the causal mask

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
import re
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
CSRC = os.path.join(ROOT, "attention_fa2_forward_03_gb300", "csrc")
# Device code of each kernel (host planning code is not part of it)
KERNEL_SOURCES = [os.path.join(CSRC, "fa2_fwd_sm103.cuh"), os.path.join(CSRC, "fa2_fwd_d64_sm103.cuh"),
                  os.path.join(CSRC, "ptx_sm103.cuh")]
BWD_SOURCES = KERNEL_SOURCES + [os.path.join(CSRC, "fa2_bwd_sm103.cuh")]
FP8_SOURCES = KERNEL_SOURCES + [os.path.join(CSRC, "fa2_fwd_fp8_sm103.cuh")]
PASSES = ("fwd", "fwd_causal", "bwd", "bwd_causal")
REASON_FIELDS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def strip_comments(src: str) -> str:
    """C++ source without comments and blank runs (string literals in these
    files hold no comment markers), so that a comment edit keeps the hash."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash(which: str = "fwd") -> str:
    """sha256[:16] of the device code a pass runs, comments removed: "fwd"
    (16-bit forward, also fwd_causal), "bwd*" or "fp8"."""
    h = hashlib.sha256()
    files = BWD_SOURCES if which.startswith("bwd") else FP8_SOURCES if which == "fp8" else KERNEL_SOURCES
    for f in files:
        with open(f, encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ distributed plumbing

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend: str):
        if self.world > 1 and self.pg is None:
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

def load_peak(fp8: bool = False):
    """Dense tensor peak for the kernel's operand type: the measured bf16
    burst figure, times the nominal fp8 : bf16 ratio (4.5 : 2.25 PFLOP/s)
    for FP8 operands."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    ratio, tag = (2.0, " x 2 (nominal fp8:bf16 ratio)") if fp8 else (1.0, "")
    try:
        with open(path) as fh:
            peaks = json.load(fh)
        return (float(peaks["bf16_tflops"]) * ratio,
                "measured (bf16_tflops burst, MEASURED_PEAKS.json)" + tag)
    except (OSError, KeyError, ValueError):
        return 1900.0 * ratio, "fallback (1.9 PFLOP/s bf16 burst)" + tag


def load_hbm_peak():
    """Measured HBM copy bandwidth (GB/s), else the stated fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured (hbm_gbs, MEASURED_PEAKS.json)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback (6.8 TB/s)"


def ridge_flop_per_byte(tensor_peak_tflops: float) -> float:
    """FLOP per byte where the tensor and HBM roofs meet."""
    return tensor_peak_tflops * 1e12 / (load_hbm_peak()[0] * 1e9)


def traffic_key(workload: str, which: str) -> str:
    return workload if which == "fwd" else f"{workload}:{which}"


def load_traffic(workload: str, which: str = "fwd"):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source for this workload
    and pass; else None."""
    try:
        with open(TRAFFIC_FILE) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    entry = rec.get(traffic_key(workload, which))
    src = "fp8" if gen.workload(workload).fp8 else which
    if not entry or entry.get("kernel_source_sha") != kernel_source_hash(src):
        return None
    return entry.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ work per pass

def causal_pairs(N: int) -> int:
    """Unmasked (query, key) pairs of one causal head with equal lengths."""
    return N * (N + 1) // 2


def pass_flops(w, which: str) -> float:
    """Algorithmic FLOPs of one step: 4*d per unmasked (query, key) pair for
    the forward, 2.5x that for the backward."""
    pairs = causal_pairs(w.N) if which.endswith("causal") else w.N * w.N
    fwd = 4.0 * w.B * w.Hq * pairs * w.d
    return fwd * (2.5 if which.startswith("bwd") else 1.0)


def pass_bytes(w, which: str) -> int:
    """Algorithmic HBM bytes of one step: every tensor read or written once."""
    if not which.startswith("bwd"):
        return w.alg_bytes
    q = w.B * w.Hq * w.N * w.d * 2
    kv = w.B * w.Hkv * w.N * w.d * 2
    # reads q, k, v, o, dO, lse; writes dq, dk, dv (delta: written and read once)
    return 3 * q + 2 * kv + 4 * w.B * w.Hq * w.N + q + 2 * kv + 8 * w.B * w.Hq * w.N


# ------------------------------------------------------------------ CPU oracle timing

def oracle_forward(w, inputs, rows, causal: bool = False):
    """The oracle's forward on a row sample of this workload."""
    import oracle

    if w.fp8:
        return oracle.attention_fp8(*inputs, w.scale, round_p=False, rows=rows, causal=causal)
    q, k, v = inputs
    if causal:
        return oracle.attention_ex(q, k, v, w.scale, w.dtype, causal=True, rows=rows)
    return oracle.attention(q, k, v, w.scale, w.dtype, rows=rows)


def oracle_rows_for(w, seconds: float, inputs, causal: bool = False):
    """Rows per second of the fp64 oracle on this host, then a seeded row
    sample sized to take about `seconds`."""
    import oracle

    rng = np.random.default_rng(w.seed)
    total = w.B * w.Hq * w.N
    calib = rng.integers(0, total, 64)
    t0 = time.perf_counter()
    oracle_forward(w, inputs, calib, causal)
    rate = 64 / max(time.perf_counter() - t0, 1e-6)
    n = int(max(1, min(total, rate * seconds)))
    return rng.integers(0, total, n), oracle.max_threads()


class OracleSample:
    """A bounded piece of one step's work for the fp64 CPU oracle.

    Forward passes: a seeded sample of query rows (full key length).
    Backward passes: the whole backward of one KV-head group (batch 0, KV
    head 0 and its query heads, full N): dK and dV need every query row.
    """

    def __init__(self, w, which: str, seconds: float, inputs):
        import oracle

        self.oracle, self.w, self.which = oracle, w, which
        self.inputs = inputs
        q, k, v = inputs[:3]
        self.causal = which.endswith("causal")
        self.cores = oracle.max_threads()
        if which.startswith("bwd"):
            G = w.Hq // w.Hkv
            self.q, self.k, self.v = (np.ascontiguousarray(x[:1, :h]) for x, h in
                                      ((q, G), (k, 1), (v, 1)))
            self.do = np.ascontiguousarray(w.grad_output()[:1, :G])
            pairs = causal_pairs(w.N) if self.causal else w.N * w.N
            self.flops = 10.0 * G * pairs * w.d
            self.desc = (f"backward of one KV-head group (b=0, kv head 0, {G} query head(s), "
                         f"N={w.N}) of the {w.B * w.Hkv}-group workload per step; fp64 C oracle, OpenMP")
        else:
            self.rows, _ = oracle_rows_for(w, seconds, inputs, self.causal)
            i = self.rows % w.N
            keys = (i + 1) if self.causal else np.full(self.rows.shape, w.N)
            self.flops = 4.0 * w.d * float(keys.sum())
            self.desc = (f"{len(self.rows)} seeded query rows of the {w.B * w.Hq * w.N}-row "
                         f"workload per step (full key length N={w.N}"
                         f"{', causal' if self.causal else ''}); fp64 C oracle, OpenMP")

    def run(self):
        o, w = self.oracle, self.w
        if self.which.startswith("bwd"):
            o.attention_bwd(self.q, self.k, self.v, self.do, w.scale, w.dtype, causal=self.causal)
        else:
            oracle_forward(w, self.inputs, self.rows, self.causal)


def cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo; Arm hosts may list none)."""
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                key, _, val = line.partition(":")
                if key.strip().lower() in ("model name", "cpu model", "hardware"):
                    return val.strip()
    except OSError:
        pass
    import platform

    return platform.processor() or platform.machine()


def time_oracle(w, which: str, inputs, seconds: float):
    sample = OracleSample(w, which, seconds, inputs)
    t0 = time.perf_counter()
    sample.run()
    dt = time.perf_counter() - t0
    return sample.flops / dt / 1e12, sample.cores, sample.desc, dt


# ------------------------------------------------------------------ arms

def run_reference(args, dist, w):
    """fp64 CPU oracle as the reference arm: each step a bounded sample."""
    if dist.rank != 0:
        return None
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)
    sample = OracleSample(w, args.pass_, per_step, w.inputs())
    for _ in range(args.warmup):
        sample.run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sample.run()
    dt = time.perf_counter() - t0
    value = sample.flops * args.steps / dt / 1e12
    return {
        "impl": "reference",
        "metric": metric_of(args.pass_, w), "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args.gpus, args.pass_),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": sample.cores, "kind": "oracle",
                         "sample": sample.desc, "cpu": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def metric_of(which: str, w=None) -> str:
    if w is not None and w.fp8:
        if which == "fwd_causal":
            return ("attention fwd causal TFLOP/s (4d per unmasked pair) at 1 GB300, FP8 e4m3 inputs; "
                    "% of dense FP8 tensor peak")
        return "attention fwd TFLOP/s (4BHN²d) at 1 GB300, FP8 e4m3 inputs; % of dense FP8 tensor peak"
    if which == "fwd":
        return METRIC
    if which == "fwd_causal":
        return "attention fwd causal TFLOP/s (4d per unmasked pair) at 1 GB300"
    return ("attention bwd TFLOP/s (2.5x forward FLOPs" +
            (", causal" if which == "bwd_causal" else "") + ") at 1 GB300")


def dtype_name(w) -> str:
    return {gen.BF16: "bf16", gen.FP16: "fp16", gen.E4M3: "e4m3"}[w.dtype]


def config_of(w, n_gpus, which: str = "fwd"):
    return {"workload": w.name, "pass": which, "B": w.B, "H_q": w.Hq, "H_kv": w.Hkv, "N": w.N,
            "d": w.d, "dtype": dtype_name(w) + (" in, bf16 out, per-(batch, KV head) descales"
                                                if w.fp8 else ""),
            "causal": which.endswith("causal"), "scale": "1/sqrt(d)",
            "inputs": f"N(0,1)x{w.amp:g} seed {w.seed}"
                      + (f"; dO N(0,1) seed {w.seed + 50000}" if which.startswith("bwd") else ""),
            "global_batch": w.B * n_gpus, "seq_len": w.N,
            "parallelism": f"replicas x{n_gpus}" if n_gpus > 1 else "single GPU",
            "l2": l2_note(w)}


def qkv_bytes(w) -> int:
    return (1 if w.fp8 else 2) * w.d * w.N * w.B * (w.Hq + 2 * w.Hkv)


def l2_note(w) -> str:
    mib = qkv_bytes(w) / 2**20
    if qkv_bytes(w) > L2_BYTES:
        return f"inputs larger than L2: Q+K+V = {mib:.0f} MiB > 129 MiB"
    return f"L2 flushed between timed steps (256 MiB write); Q+K+V = {mib:.1f} MiB"


class Step:
    """Device tensors and the C-ABI call of one step of a pass."""

    def __init__(self, fa2, torch, w, which, dev, stream, inputs):
        self.fa2, self.torch, self.w, self.which, self.stream = fa2, torch, w, which, stream
        self.tdt = torch.bfloat16 if w.dtype in (gen.BF16, gen.E4M3) else torch.float16
        self.causal = which.endswith("causal")
        self.bwd = which.startswith("bwd")
        self.fp8 = w.fp8
        if self.fp8 and self.bwd:
            raise ValueError("FP8 workloads have the forward passes only")

        def up(x):
            if x.dtype == np.uint8 or x.dtype == np.float32:
                return torch.from_numpy(np.ascontiguousarray(x)).to(dev)
            return torch.from_numpy(x.view(np.int16)).to(dev).view(self.tdt)

        self.tq, self.tk, self.tv = (up(x) for x in inputs[:3])
        if self.fp8:
            self.tqd, self.tkd, self.tvd = (up(x) for x in inputs[3:])
        self.o = torch.empty(self.tq.shape, dtype=self.tdt, device=dev)
        self.lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)
        if self.bwd:
            self.tdo = up(w.grad_output())
            fa2.fa2_fwd_ex(self.tq, self.tk, self.tv, self.o, self.lse, scale=w.scale,
                           causal=self.causal, stream=stream)
            self.dq = torch.empty_like(self.tq)
            self.dk = torch.empty_like(self.tk)
            self.dv = torch.empty_like(self.tv)
            self.delta = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)
        # launches of this library's kernels per step
        self.launches = 3 if self.bwd else 1
        if self.bwd:
            self.kernel = "fa2_bwd (delta + dK/dV + dQ kernels)"
        elif self.fp8:
            self.kernel = "fa2_fwd_fp8_kernel" + ("<general>" if self.causal else "")
        elif w.d == 64 and not self.causal and os.environ.get("FA2_TILE_CFG") != "d64=shared":
            self.kernel = f"fa2_fwd_d64_kernel<{'bf16' if w.dtype == gen.BF16 else 'fp16'}>"
        else:
            self.kernel = (f"fa2_fwd_kernel<{w.d},{'bf16' if w.dtype == gen.BF16 else 'fp16'}"
                           f"{',general' if self.causal else ''}>")

    def __call__(self):
        w, f, s = self.w, self.fa2, self.stream.cuda_stream
        if self.bwd:
            rc = f.fa2_bwd_ptr(self.tq.data_ptr(), self.tk.data_ptr(), self.tv.data_ptr(),
                               self.o.data_ptr(), self.lse.data_ptr(), self.tdo.data_ptr(),
                               self.dq.data_ptr(), self.dk.data_ptr(), self.dv.data_ptr(),
                               self.delta.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.d, w.scale,
                               self.causal, w.dtype, s)
            name = "fa2_bwd"
        elif self.fp8 and self.causal:
            rc = f.fa2_fwd_fp8_ex_ptr(self.tq.data_ptr(), self.tk.data_ptr(), self.tv.data_ptr(),
                                      self.tqd.data_ptr(), self.tkd.data_ptr(), self.tvd.data_ptr(),
                                      self.o.data_ptr(), self.lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.N,
                                      w.d, w.scale, True, s)
            name = "fa2_fwd_fp8_ex"
        elif self.fp8:
            rc = f.fa2_fwd_fp8_ptr(self.tq.data_ptr(), self.tk.data_ptr(), self.tv.data_ptr(),
                                   self.tqd.data_ptr(), self.tkd.data_ptr(), self.tvd.data_ptr(),
                                   self.o.data_ptr(), self.lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N, w.d,
                                   w.scale, s)
            name = "fa2_fwd_fp8"
        elif self.causal:
            rc = f.fa2_fwd_ex_ptr(self.tq.data_ptr(), self.tk.data_ptr(), self.tv.data_ptr(),
                                  self.o.data_ptr(), self.lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N,
                                  w.N, w.d, w.scale, True, w.dtype, s)
            name = "fa2_fwd_ex"
        else:
            rc = f.fa2_fwd_gqa_ptr(self.tq.data_ptr(), self.tk.data_ptr(), self.tv.data_ptr(),
                                   self.o.data_ptr(), self.lse.data_ptr(), w.B, w.Hq, w.Hkv, w.N,
                                   w.d, w.scale, w.dtype, s)
            name = "fa2_fwd_gqa"
        if rc != f.FA2_OK:
            raise RuntimeError(f"{name}: {f.status_string(rc)}")

    def _io(self):
        """The device tensors one call reads (inputs) and writes (results)."""
        if self.bwd:
            return [self.tq, self.tk, self.tv, self.o, self.lse, self.tdo], [self.dq, self.dk, self.dv]
        if self.fp8:
            return [self.tq, self.tk, self.tv, self.tqd, self.tkd, self.tvd], [self.o, self.lse]
        return [self.tq, self.tk, self.tv], [self.o, self.lse]

    def _call_public(self, ins, outs, stream):
        """One call through the public torch-level binding."""
        f, w = self.fa2, self.w
        if self.bwd:
            q, k, v, o, lse, do = ins
            dq, dk, dv = outs
            f.fa2_bwd(q, k, v, o, lse, do, scale=w.scale, causal=self.causal, dq=dq, dk=dk, dv=dv,
                      delta=self.delta, stream=stream)
        elif self.fp8 and self.causal:
            q, k, v, qd, kd, vd = ins
            f.fa2_fwd_fp8_ex(q, k, v, qd, kd, vd, outs[0], outs[1], scale=w.scale, causal=True, stream=stream)
        elif self.fp8:
            q, k, v, qd, kd, vd = ins
            f.fa2_fwd_fp8(q, k, v, qd, kd, vd, outs[0], outs[1], scale=w.scale, stream=stream)
        elif self.causal:
            f.fa2_fwd_ex(*ins, outs[0], outs[1], scale=w.scale, causal=True, stream=stream)
        else:
            f.fa2_fwd_gqa(*ins, outs[0], outs[1], scale=w.scale, stream=stream)

    def e2e_run(self, host, warm, steps):
        """End to end through the public binding: every step copies its
        inputs from pinned host memory to the device, calls the library, and
        copies its results back to pinned host memory. The steps are pipelined
        the way a serving loop streams batches: two device buffer sets, the
        upload of step i+1 and the download of step i-1 overlapping the
        kernels of step i on their own streams (events order each buffer's
        reuse). Returns the milliseconds from before the first timed upload
        to after the last timed download."""
        torch = self.torch
        ins_h, outs_h = host
        first = self._io()
        slots = [first, ([torch.empty_like(t) for t in first[0]], [torch.empty_like(t) for t in first[1]])]
        comp = self.stream
        up = torch.cuda.Stream(device=comp.device)
        down = torch.cuda.Stream(device=comp.device)
        up_done = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        down_done = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def one(i):
            s = i % 2
            ins, outs = slots[s]
            with torch.cuda.stream(up):
                if used[s]:
                    up.wait_event(comp_done[s])      # the kernel two steps back read these
                for d_, h_ in zip(ins, ins_h):
                    d_.copy_(h_, non_blocking=True)
                up_done[s].record(up)
            comp.wait_event(up_done[s])
            if used[s]:
                comp.wait_event(down_done[s])        # the download two steps back read these
            self._call_public(ins, outs, comp)
            comp_done[s].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(comp_done[s])
                for h_, d_ in zip(outs_h, outs):
                    h_.copy_(d_, non_blocking=True)
                down_done[s].record(down)
            used[s] = True

        for i in range(warm):
            one(i)
        torch.cuda.synchronize(comp.device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(up)
        for i in range(warm, warm + steps):
            one(i)
        e1.record(down)
        torch.cuda.synchronize(comp.device)
        return e0.elapsed_time(e1)

    def host_buffers(self):
        """Pinned host copies of the step's inputs and room for its results."""
        def pin(t):
            return t.detach().cpu().pin_memory()

        if self.bwd:
            ins = tuple(pin(t) for t in (self.tq, self.tk, self.tv, self.o, self.lse, self.tdo))
            outs = tuple(self.torch.empty(t.shape, dtype=t.dtype).pin_memory()
                         for t in (self.dq, self.dk, self.dv))
        else:
            dev_in = (self.tq, self.tk, self.tv) + ((self.tqd, self.tkd, self.tvd) if self.fp8 else ())
            ins = tuple(pin(t) for t in dev_in)
            outs = tuple(self.torch.empty(t.shape, dtype=t.dtype).pin_memory()
                         for t in (self.o, self.lse))
        nbytes = [sum(t.numel() * t.element_size() for t in x) for x in (ins, outs)]
        return (ins, outs), nbytes[0], nbytes[1]


ALL_CONFIGS = (["tiny_B1_H1_N128_d128_bf16", "mha_B4_H16_N4096_d128_bf16"]
               + [f"sweep_N{n}_{t}" for t in ("bf16", "fp16") for n in (512, 1024, 2048, 4096, 8192, 16384)]
               + ["sharp_B8_H32_N2048_d64_bf16_x3", "gqa_B2_Hq32_Hkv8_N8192_d128_bf16"])


def harmonic_mean_line(lines, tag, n_gpus):
    """One line for the harmonic mean over the sweep points of one dtype."""
    pts = [ln for ln in lines if ln["config"]["workload"].startswith("sweep_") and
           ln["config"]["workload"].endswith(tag)]
    if not pts:
        return None
    hm = len(pts) / sum(1.0 / ln["value"] for ln in pts)
    # per-launch kernel TFLOP/s of each point (points left of the ridge
    # report GB/s as `achieved` and keep their TFLOP/s under `tflops`)
    rate = lambda r: r["tflops"] if r["bound"] == "hbm" else r["achieved"]
    hk = len(pts) / sum(1.0 / rate(ln["roofline"]) for ln in pts)
    peak, peak_src = load_peak()
    return {"metric": METRIC + "; harmonic mean over N in {512..16384}", "value": hm, "unit": UNIT,
            "n_gpus": n_gpus, "steps": pts[0]["steps"], "warmup": pts[0]["warmup"],
            "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": tag, "data": "synthetic",
            "config": {"workload": f"sweep_{tag}_harmonic_mean", "points": {
                ln["config"]["workload"]: round(ln["value"], 1) for ln in pts},
                "B*N": 16384, "H": 16, "d": 128},
            "roofline": {"bound": "tensor", "achieved": hk, "peak": peak, "unit": UNIT, "frac": hk / peak,
                         "traffic": None, "peak_source": peak_src,
                         "kernel": pts[0]["roofline"]["kernel"],
                         "note": "harmonic mean of the points' per-launch kernel rates"}}


def run_ours(args, dist, w):
    import torch

    from attention_fa2_forward_03_gb300 import fa2

    fa2.load()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    stream = torch.cuda.current_stream(dev)

    inputs = w.inputs()
    step = Step(fa2, torch, w, args.pass_, dev, stream, inputs)
    flops = pass_flops(w, args.pass_)
    flush = None
    if qkv_bytes(w) <= L2_BYTES:
        flush = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)

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
    # With an L2 flush between steps the flush is not part of the work: the
    # timed span is then the sum of the steps' own intervals.
    timed_ms = kernel_ms * args.steps if flush is not None else region_ms
    rc = fa2.fa2_check_status(stream.cuda_stream)
    if rc != fa2.FA2_OK:
        raise RuntimeError(f"kernel status {fa2.status_string(rc)}")
    if dist.rank == 0:
        time.sleep(0.25)
        clocks.stop()

    value, max_region_ms = aggregate_throughput(dist, flops * args.steps, timed_ms, dev)

    # end to end through the public binding, every step: pinned host inputs
    # -> device -> kernels -> device -> pinned host results (pipelined)
    host, h2d, d2h = step.host_buffers()
    e2e_steps = max(3, min(args.steps, 50))
    dist.barrier()
    e2e_region = step.e2e_run(host, 2, e2e_steps)
    dist.barrier()
    e2e_value, e2e_ms = aggregate_throughput(dist, flops * e2e_steps, e2e_region, dev)

    result = None
    if dist.rank == 0:
        peak, peak_src = load_peak(w.fp8)
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        nbytes = pass_bytes(w, args.pass_)
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "traffic": load_traffic(w.name, args.pass_),
                "peak_source": peak_src, "kernel": step.kernel, "kernel_ms": kernel_ms,
                "alg_flops_per_launch": flops, "alg_bytes_per_launch": nbytes,
                "hbm_gbs_alg": nbytes / (kernel_ms * 1e-3) / 1e9}
        if flops / nbytes < ridge_flop_per_byte(peak):
            # left of the ridge (the one-tile case, N = 512): judged by bytes moved
            hbm, hbm_src = load_hbm_peak()
            roof.update({"bound": "hbm", "achieved": roof["hbm_gbs_alg"], "peak": hbm, "unit": "GB/s",
                         "frac": roof["hbm_gbs_alg"] / hbm, "peak_source": hbm_src,
                         "tflops": achieved})
        result = {
            "metric": metric_of(args.pass_, w), "value": value, "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": max_region_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": dtype_name(w), "data": "synthetic",
            "config": config_of(w, dist.world, args.pass_),
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step": e2e_ms / e2e_steps,
                    "note": "public binding; upload of step i+1 and download of step i-1 overlap step i"},
            "gpu_launches": args.steps * step.launches,
            "clocks": clocks.summary(),
        }
        if dist.world == 1 and not args.no_cpu_baseline:
            cv, cores, desc, dt = time_oracle(w, args.pass_, inputs, args.cpu_seconds)
            result["cpu_baseline"] = {"value": cv, "unit": UNIT, "cores": cores, "kind": "oracle",
                                      "sample": f"{desc}, {dt:.1f} s", "cpu": cpu_model()}
    return result


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(gen.WORKLOADS))
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=PASSES)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="oracle time budget of a whole --impl reference run (warm-up + timed steps)")
    ap.add_argument("--all-configs", action="store_true",
                    help="one line per forward workload configuration plus the sweep's harmonic means")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.all_configs and args.pass_ != "fwd":
        ap.error("--all-configs runs the forward pass")
    dist = Dist()
    names = ALL_CONFIGS if args.all_configs else [args.workload]
    if args.all_configs and args.cpu_seconds == ap.get_default("cpu_seconds"):
        args.cpu_seconds = 3.0        # 16 configurations: keep the oracle legs short
    lines = []
    for name in names:
        w = gen.workload(name)
        if args.impl == "reference":
            res = run_reference(args, dist, w)
        else:
            res = run_ours(args, dist, w)
        if res is not None and dist.rank == 0:
            print(json.dumps(res), flush=True)
            lines.append(res)
        if args.impl != "reference" and args.all_configs:
            import torch

            torch.cuda.empty_cache()
    if args.all_configs and args.impl != "reference" and dist.rank == 0:
        for tag in ("bf16", "fp16"):
            hm = harmonic_mean_line(lines, tag, dist.world)
            if hm is not None:
                print(json.dumps(hm), flush=True)
    dist.done()


if __name__ == "__main__":
    main()

"""bench.py's host side on the CPU: the reference arm (the fp64 oracle timed
on a bounded sample) for every pass and for an FP8 workload, the JSON line's
keys, and the FLOP and byte counts of each pass."""
import json
import os
import subprocess
import sys

import pytest

import bench
import gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3", "--ref-seconds", "4", *args],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("pass_", ["fwd", "fwd_causal", "bwd", "bwd_causal"])
def test_reference_arm_every_pass(pass_):
    d = run_reference("--workload", "tiny_B1_H1_N128_d128_bf16", "--pass", pass_)
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["config"]["pass"] == pass_ and d["config"]["causal"] == pass_.endswith("causal")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["cpu"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_fp8_workload():
    d = run_reference("--workload", "fp8_mha_B4_H16_N4096_d128_e4m3")
    assert d["value"] > 0 and d["config"]["dtype"].startswith("e4m3")
    assert "FP8" in d["metric"]


def test_reference_arm_fp8_causal_workload():
    d = run_reference("--workload", "fp8_mha_B4_H16_N4096_d128_e4m3", "--pass", "fwd_causal")
    assert d["value"] > 0 and d["config"]["causal"] is True
    assert "FP8" in d["metric"] and "causal" in d["metric"]


def test_pass_flop_and_byte_counts():
    w = gen.workload("mha_B4_H16_N4096_d128_bf16")
    assert bench.pass_flops(w, "fwd") == 4.0 * 4 * 16 * 4096 * 4096 * 128
    assert bench.pass_flops(w, "fwd_causal") == 4.0 * 4 * 16 * (4096 * 4097 // 2) * 128
    assert bench.pass_flops(w, "bwd") == 2.5 * bench.pass_flops(w, "fwd")
    assert bench.pass_flops(w, "bwd_causal") == 2.5 * bench.pass_flops(w, "fwd_causal")
    assert bench.pass_bytes(w, "fwd") == w.alg_bytes == 269484032
    q = 4 * 16 * 4096 * 128 * 2
    # reads q, k, v, o, dO (5 tensors) + lse; writes dq, dk, dv; delta written and read
    assert bench.pass_bytes(w, "bwd") == 8 * q + 4 * 4 * 16 * 4096 + 8 * 4 * 16 * 4096
    f = gen.workload("fp8_mha_B4_H16_N4096_d128_e4m3")
    # Q, K, V one byte each, O bf16, LSE fp32, 3 descales per KV head
    assert f.alg_bytes == 3 * q // 2 + q + 4 * 4 * 16 * 4096 + 12 * 4 * 16


def test_fp8_peak_is_twice_the_bf16_peak():
    bf, _ = bench.load_peak(False)
    f8, src = bench.load_peak(True)
    assert f8 == 2 * bf and "x 2" in src


def test_traffic_record_in_bytes_and_only_current_entries_reported():
    # Each entry of the committed DRAM-traffic record names the kernel source
    # hash it was captured on. An entry whose hash matches the current
    # sources is what bench.py reports as `traffic`: bytes per launch, read
    # + write, of the order of the algorithmic bytes (never MB); a stale one
    # is reported as null.
    import json

    with open(bench.TRAFFIC_FILE) as fh:
        rec = json.load(fh)
    assert rec
    for key, entry in rec.items():
        name, _, pass_ = key.partition(":")
        pass_ = pass_ or "fwd"
        w = gen.workload(name)
        assert entry["dram_bytes_per_launch"] == entry["dram_bytes_read"] + entry["dram_bytes_write"]
        assert 0.5 * bench.pass_bytes(w, pass_) < entry["dram_bytes_per_launch"] < 10 * bench.pass_bytes(w, pass_)
        src = "fp8" if w.fp8 else pass_
        current = entry["kernel_source_sha"] == bench.kernel_source_hash(src)
        expect = entry["dram_bytes_per_launch"] if current else None
        assert bench.load_traffic(name, pass_) == expect, key


def test_traffic_is_null_for_uncaptured_passes():
    assert bench.load_traffic("mha_B4_H16_N4096_d128_bf16", "bwd") is None
    assert bench.load_traffic("tiny_B1_H1_N128_d128_bf16", "fwd") is None


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    # The driver launches both arms the same way for N > 1: one process per
    # rank under torchrun. For the reference arm rank 0 alone works and
    # prints; the other ranks exit 0 without output.
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                          "--master-addr", "127.0.0.1", "--master-port", str(port),
                          os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "3", "--ref-seconds", "4"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_all_configs_cover_every_forward_configuration():
    names = bench.ALL_CONFIGS
    assert len(names) == len(set(names)) == 16
    ws = [gen.workload(n) for n in names]
    assert not any(w.fp8 for w in ws)
    sweep = [w for w in ws if w.name.startswith("sweep_")]
    assert sorted({w.N for w in sweep}) == [512, 1024, 2048, 4096, 8192, 16384]
    assert all(w.B * w.N == 16384 and w.Hq == 16 and w.d == 128 for w in sweep)
    assert {w.dtype for w in sweep} == {gen.BF16, gen.FP16}


def test_harmonic_mean_line():
    def line(name, v, a, hbm=False):
        roof = {"bound": "tensor", "achieved": a, "peak": 2000.0, "peak_source": "x", "kernel": "k"}
        if hbm:   # left of the ridge: GB/s as achieved, TFLOP/s kept aside
            roof.update({"bound": "hbm", "achieved": 3800.0, "unit": "GB/s", "tflops": a})
        return {"value": v, "steps": 10, "warmup": 3, "config": {"workload": name}, "roofline": roof}
    lines = [line("sweep_N512_bf16", 1000.0, 1100.0, hbm=True), line("sweep_N1024_bf16", 2000.0, 2200.0),
             line("sweep_N512_fp16", 5.0, 5.0), line("mha_B4_H16_N4096_d128_bf16", 7.0, 7.0)]
    hm = bench.harmonic_mean_line(lines, "bf16", 1)
    assert abs(hm["value"] - 2 / (1 / 1000 + 1 / 2000)) < 1e-9
    assert abs(hm["roofline"]["achieved"] - 2 / (1 / 1100 + 1 / 2200)) < 1e-9
    peak, _ = bench.load_peak()
    assert abs(hm["roofline"]["frac"] - hm["roofline"]["achieved"] / peak) < 1e-12
    assert hm["roofline"]["unit"] == "TFLOP/s"
    assert set(hm["config"]["points"]) == {"sweep_N512_bf16", "sweep_N1024_bf16"}
    assert bench.harmonic_mean_line(lines, "e4m3", 1) is None


def test_left_of_the_ridge_are_the_one_tile_case_and_the_shortest_sweep_point():
    # 64 and 255 FLOP/B against a ridge of ~281 (1901.5 TFLOP/s / 6759 GB/s)
    peak, _ = bench.load_peak()
    ridge = bench.ridge_flop_per_byte(peak)
    left_names = {"tiny_B1_H1_N128_d128_bf16", "sweep_N512_bf16", "sweep_N512_fp16"}
    for name in bench.ALL_CONFIGS:
        w = gen.workload(name)
        left = bench.pass_flops(w, "fwd") / bench.pass_bytes(w, "fwd") < ridge
        assert left == (name in left_names), name

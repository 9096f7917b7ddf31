"""Parity of the backward (fa2_bwd, through the C ABI) with the fp64 oracle.

Tolerance, derived from the arithmetic (the workload definition gives none
for gradients): P and dS are rounded to the 16-bit input type before their
GEMMs (relative 2^-8 for bf16, 2^-11 for fp16, per element), D = rowsum(dO o O)
uses the 16-bit forward output, and the gradients are rounded once more at
the end. Per tensor this gives normwise bounds, checked for dQ, dK and dV:
    max|G - G_ref| <= 2^-6 * max|G_ref|,  ||G - G_ref||_F <= 2^-7 * ||G_ref||_F
for bf16 (2^-8 and 2^-9 for fp16). The forward output O and LSE fed to the
backward come from the GPU forward, as in training.
"""
import math

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


def to_dev(x, dtype):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to("cuda")
    return t.view(torch.bfloat16 if dtype == gen.BF16 else torch.float16)


def check(name, g, ref, dtype, floor=0.0):
    """floor: an absolute error allowance for gradients that are exactly zero
    (a single key: dS = dP - D = 0), where the relative bounds are void."""
    g = np.asarray(g, dtype=np.float64)
    tmax, tfro = (2.0 ** -6, 2.0 ** -7) if dtype == gen.BF16 else (2.0 ** -8, 2.0 ** -9)
    err = np.abs(g - ref)
    scale = np.max(np.abs(ref))
    assert np.isfinite(g).all(), name
    assert err.max() <= max(tmax * scale, floor), f"{name}: max err {err.max():.4g} vs {tmax * scale:.4g}"
    if scale > 0:
        fro = np.linalg.norm(g - ref) / np.linalg.norm(ref)
        assert fro <= tfro, f"{name}: relative Frobenius error {fro:.4g}"
    else:
        fro = 0.0
    return err.max() / max(scale, 1e-300), fro


CASES = [
    # B, Hq, Hkv, N, d, dtype, causal
    (1, 1, 1, 128, 128, gen.BF16, False),
    (1, 2, 2, 256, 128, gen.BF16, False),
    (1, 2, 2, 384, 128, gen.BF16, True),
    (2, 2, 2, 256, 64, gen.FP16, False),
    (1, 4, 2, 256, 128, gen.BF16, False),   # grouped heads: dK, dV summed over 2 query heads
    (1, 4, 1, 384, 64, gen.BF16, True),
    (1, 2, 2, 512, 128, gen.FP16, True),
    (1, 2, 2, 2048, 128, gen.BF16, False),  # 16 steps: every ring wraps several times
    (1, 4, 2, 2048, 128, gen.BF16, True),   # grouped heads, causal, up to 32 dK/dV steps
    # ragged lengths (N not a multiple of 128): rows past N are zero-filled
    # by the tensor maps, masked and not stored
    (1, 2, 2, 200, 128, gen.BF16, False),
    (2, 2, 1, 129, 128, gen.BF16, True),
    (1, 4, 2, 300, 64, gen.FP16, True),
    (1, 1, 1, 1, 128, gen.BF16, False),     # a single row
    (1, 2, 2, 1000, 128, gen.BF16, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,causal", CASES)
def test_backward_matches_oracle(gpu_lib, B, Hq, Hkv, N, d, dtype, causal):
    import torch

    q, k, v = gen.make_qkv(4000 + N + d + Hq, B, Hq, Hkv, N, d, dtype)
    do, _, _ = gen.make_qkv(4100 + N + d + Hq, B, Hq, Hkv, N, d, dtype)
    scale = 1 / math.sqrt(d)
    tq, tk, tv, tdo = (to_dev(x, dtype) for x in (q, k, v, do))
    o, lse = gpu_lib.fa2_fwd_ex(tq, tk, tv, scale=scale, causal=causal)
    dq, dk, dv = gpu_lib.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=scale, causal=causal)
    assert gpu_lib.fa2_check_status(torch.cuda.current_stream().cuda_stream) == gpu_lib.FA2_OK
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, scale, dtype, causal=causal)
    # fp32 accumulation error of dP and D over d terms, carried into dQ and dK
    mx = lambda x: float(np.max(np.abs(gen.bits_to_float32(x, dtype))))
    floor = d * 2.0 ** -20 * mx(do) * mx(v) * mx(k) * scale
    res = [check(n, g.float().cpu().numpy(), r, dtype, floor)
           for n, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv))]
    print("max/fro errors (relative):", res)


def test_backward_zero_upstream_gradient(gpu_lib):
    import torch

    q, k, v = gen.make_qkv(4200, 1, 2, 2, 256, 128, gen.BF16)
    tq, tk, tv = (to_dev(x, gen.BF16) for x in (q, k, v))
    o, lse = gpu_lib.fa2_fwd_gqa(tq, tk, tv)
    dq, dk, dv = gpu_lib.fa2_bwd(tq, tk, tv, o, lse, torch.zeros_like(tq))
    assert not bool(dq.any()) and not bool(dk.any()) and not bool(dv.any())


def test_backward_key_gradient_sums_to_zero(gpu_lib):
    """sum_j dK_j = 0 for every (batch, KV head): each row of dS sums to 0."""
    import torch

    q, k, v = gen.make_qkv(4300, 2, 4, 2, 512, 128, gen.BF16)
    do, _, _ = gen.make_qkv(4301, 2, 4, 2, 512, 128, gen.BF16)
    tq, tk, tv, tdo = (to_dev(x, gen.BF16) for x in (q, k, v, do))
    o, lse = gpu_lib.fa2_fwd_gqa(tq, tk, tv)
    dq, dk, dv = gpu_lib.fa2_bwd(tq, tk, tv, o, lse, tdo)
    s = dk.double().sum(dim=2)
    assert float(s.abs().max()) <= 2.0 ** -6 * float(dk.double().abs().sum(dim=2).max())


def test_backward_full_size_bench_workload_slices(gpu_lib):
    """The backward bench workload (B4 H16 N4096 d128 bf16, dO from the
    workload's generator), in the bench's launch configuration; two (batch,
    head) slices are checked against the oracle run on that slice alone (with
    equal head counts a head's gradients depend on its own Q, K, V, dO only)."""
    import torch

    w = gen.workload("mha_B4_H16_N4096_d128_bf16")
    q, k, v = w.inputs()
    do = w.grad_output()
    tq, tk, tv, tdo = (to_dev(x, w.dtype) for x in (q, k, v, do))
    o, lse = gpu_lib.fa2_fwd_gqa(tq, tk, tv, scale=w.scale)
    dq, dk, dv = gpu_lib.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=w.scale)
    assert gpu_lib.fa2_check_status(torch.cuda.current_stream().cuda_stream) == gpu_lib.FA2_OK
    for b, h in ((0, 0), (3, 15)):
        sl = lambda x: np.ascontiguousarray(x[b:b + 1, h:h + 1])
        rq, rk, rv = oracle.attention_bwd(sl(q), sl(k), sl(v), sl(do), w.scale, w.dtype)
        for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            check(f"{name}[{b},{h}]", g[b:b + 1, h:h + 1].float().cpu().numpy(), r, w.dtype)

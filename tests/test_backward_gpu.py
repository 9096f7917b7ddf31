"""Parity of the backward (fa2_bwd, through the C ABI) with the fp64 oracle,
element by element.

Tolerance, derived from the arithmetic (the workload definition gives none
for gradients). With u the unit roundoff of the 16-bit type (2^-8 bf16,
2^-11 fp16), the kernels
  * round P to 16 bits before dV = P^T dO, and dS = P o (dP - D) to 16 bits
    before dK = scale dS^T Q and dQ = scale dS K (relative u per element,
    or 2^-25 absolutely below fp16's normal range);
  * take D = rowsum(dO o O) from the 16-bit forward output O, whose error is
    at most u (|O| + a) per element (a = sum_j P_ij |V_j|: the forward's own
    rounding of P), and the forward's fp32 LSE;
  * accumulate every product in fp32 (at most n 2^-24 of the sum of |terms|
    over n terms), and round each gradient to 16 bits at the end (u |G|, or
    eta absolutely below the normal range).
Summed over a row or column this bounds every element:
    |dV - ref| <= (2u + N 2^-24) A_V + eta C_V + u |ref| + eta
    |dK - ref| <= (2u + N 2^-24) A_K + 2u BE_K + d 2^-24 BF_K + eta C_K + u |ref| + eta
    |dQ - ref| <= (2u + N 2^-24) A_Q + 2u BE_Q + d 2^-24 BF_Q + eta C_Q + u |ref| + eta
with the oracle's absolute sums A = sum |dS| |K or Q| * scale (A_V =
sum_i P_ij |dO_i|), BE = scale sum P E_i |K or Q| (E_i = sum_t |dO_it|
(|O_it| + a_it): D's error), BF = scale sum P F_ij |K or Q| (F_ij =
sum_t |dO_it| |V_jt|: dP's fp32 error), C = the same sums with the weight
|dS| or P replaced by 1 (the subnormal floor; eta = 2^-25 for fp16, 2^-126
for bf16, whose subnormal P and dS flush to zero), and a margin of 1.25 over the whole. u covers the roundings; the
factor 2 on them absorbs the fp32 exponentials, the forward's LSE error and
the product of two roundings. The forward output O and LSE fed to the
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


def _allowed_sums(x, n_other, causal, keys):
    """sum over the allowed partners of |x| along the row axis: for keys=True
    x is [.., N_q, d] summed over the query rows i that may attend key j
    (i >= j when causal), else x is [.., N_k, d] summed over keys j <= i."""
    ax = np.abs(x)
    if not causal:
        return np.broadcast_to(ax.sum(axis=-2, keepdims=True), ax.shape[:-2] + (n_other, ax.shape[-1]))
    if keys:  # suffix sums: rows i >= j
        return np.flip(np.cumsum(np.flip(ax, -2), axis=-2), -2)
    return np.cumsum(ax, axis=-2)  # prefix sums: keys j <= i


def bwd_bounds(q, k, do, bnd, scale, dtype, causal):
    """Elementwise bounds for dq, dk, dv from the oracle's absolute sums."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    u = 2.0 ** -8 if dtype == gen.BF16 else 2.0 ** -11
    eta = 2.0 ** -126 if dtype == gen.BF16 else 2.0 ** -25
    gam_n, gam_d = N * 2.0 ** -24, d * 2.0 ** -24
    Q, K, dO = (oracle.decode16(x, dtype) for x in (q, k, do))
    kv = lambda x: x.reshape(B, Hkv, G, N, d).sum(axis=2)
    c_q = scale * _allowed_sums(np.repeat(K, G, axis=1), N, causal, keys=False)
    c_k = scale * kv(_allowed_sums(Q, N, causal, keys=True))
    c_v = kv(_allowed_sums(dO, N, causal, keys=True))
    aq, beq, bfq = bnd["q"]
    ak, bek, bfk = bnd["k"]
    return ((2 * u + gam_n) * aq + 2 * u * beq + gam_d * bfq + eta * c_q,
            (2 * u + gam_n) * ak + 2 * u * bek + gam_d * bfk + eta * c_k,
            (2 * u + gam_n) * bnd["v"] + eta * c_v), u, eta


def check(name, g, ref, bound, u, eta):
    g = np.asarray(g, dtype=np.float64)
    assert np.isfinite(g).all(), name
    err = np.abs(g - ref)
    lim = 1.25 * (bound + u * np.abs(ref) + eta)
    bad = err > lim
    worst = float(np.max(err / np.maximum(lim, 1e-300))) if err.size else 0.0
    assert not bad.any(), (f"{name}: {int(bad.sum())}/{bad.size} elements beyond the bound, worst "
                           f"{worst:.3g} of it at {np.unravel_index(np.argmax(err - lim), err.shape)}")
    return worst


def check_all(dq, dk, dv, q, k, v, do, scale, dtype, causal, what=""):
    rq, rk, rv, bnd = oracle.attention_bwd(q, k, v, do, scale, dtype, causal=causal, bounds=True)
    (bq, bk, bv), u, eta = bwd_bounds(q, k, do, bnd, scale, dtype, causal)
    return [check(f"{what}{n}", g, r, b, u, eta)
            for n, g, r, b in (("dq", dq, rq, bq), ("dk", dk, rk, bk), ("dv", dv, rv, bv))]


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
    # more tiles than the 152 SMs: the persistent CTAs take several tiles each
    # (160 key / query tiles); causal with 5 tiles a head: pairs (0, 4),
    # (1, 3) and the middle tile alone, 192 units
    (1, 40, 40, 512, 64, gen.BF16, False),
    (1, 64, 64, 640, 64, gen.FP16, True),
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
    res = check_all(*(g.float().cpu().numpy() for g in (dq, dk, dv)), q, k, v, do, scale, dtype, causal)
    print("worst error / bound (dq, dk, dv):", res)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_watchdog_reports_timeout_and_context_survives(gpu_lib, causal):
    """The dK/dV kernel with its query-tile loads skipped (test hook): its
    bounded waits run out, the status word reports FA2_ERR_TIMEOUT, every
    persistent CTA returns, and the next backward on the same context is
    correct."""
    import torch

    B, Hq, Hkv, N, d, dtype = 1, 2, 2, 384, 128, gen.BF16
    q, k, v = gen.make_qkv(4200, B, Hq, Hkv, N, d, dtype)
    do, _, _ = gen.make_qkv(4201, B, Hq, Hkv, N, d, dtype)
    scale = 1 / math.sqrt(d)
    tq, tk, tv, tdo = (to_dev(x, dtype) for x in (q, k, v, do))
    o, lse = gpu_lib.fa2_fwd_ex(tq, tk, tv, scale=scale, causal=causal)
    assert gpu_lib.fa2_check_status(torch.cuda.current_stream().cuda_stream) == gpu_lib.FA2_OK
    old_limit = gpu_lib.fa2_set_wait_limit_ns(20_000_000)  # 20 ms
    old_flags = gpu_lib.fa2_set_debug_flags(1)
    try:
        gpu_lib.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=scale, causal=causal)
        rc = gpu_lib.fa2_check_status(torch.cuda.current_stream().cuda_stream)
    finally:
        gpu_lib.fa2_set_debug_flags(old_flags)
        gpu_lib.fa2_set_wait_limit_ns(old_limit)
    assert rc == gpu_lib.FA2_ERR_TIMEOUT
    assert gpu_lib.fa2_check_status(0) == gpu_lib.FA2_OK  # the word was cleared
    dq, dk, dv = gpu_lib.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=scale, causal=causal)
    assert gpu_lib.fa2_check_status(torch.cuda.current_stream().cuda_stream) == gpu_lib.FA2_OK
    check_all(*(g.float().cpu().numpy() for g in (dq, dk, dv)), q, k, v, do, scale, dtype, causal, "after watchdog")


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
    workload's generator), in the bench's launch configuration; four (batch,
    head) slices are checked against the oracle run on that slice alone (with
    equal head counts a head's gradients depend on its own Q, K, V, dO only),
    every element of those slices against the elementwise bound."""
    import torch

    w = gen.workload("mha_B4_H16_N4096_d128_bf16")
    q, k, v = w.inputs()
    do = w.grad_output()
    tq, tk, tv, tdo = (to_dev(x, w.dtype) for x in (q, k, v, do))
    o, lse = gpu_lib.fa2_fwd_gqa(tq, tk, tv, scale=w.scale)
    dq, dk, dv = gpu_lib.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=w.scale)
    assert gpu_lib.fa2_check_status(torch.cuda.current_stream().cuda_stream) == gpu_lib.FA2_OK
    for b, h in ((0, 0), (1, 7), (2, 9), (3, 15)):
        sl = lambda x: np.ascontiguousarray(x[b:b + 1, h:h + 1])
        gs = [g[b:b + 1, h:h + 1].float().cpu().numpy() for g in (dq, dk, dv)]
        check_all(*gs, sl(q), sl(k), sl(v), sl(do), w.scale, w.dtype, False, what=f"[{b},{h}] ")

"""Parity of the FP8 (e4m3) forward (fa2_fwd_fp8, fa2_fwd_fp8_ex) with the fp64 oracle,
through the C ABI.

Tolerance, derived from the method's arithmetic (no tolerance is given for
FP8 inputs). The kernel computes S = Q K^T exactly in fp32 from the e4m3
codes, then P' = 2^8 p in fp32 and rounds P' to e4m3 before P.V; l sums the
unrounded P'. Rounding to e4m3 moves each weight by at most 2^-4 p_j (normal
range) or 2^-10 / 2^8 absolutely (subnormal range), so against attention on
the dequantised inputs (the oracle with round_p=False):
    |O - O_plain| <= 2^-4 a + 2^-18 b + 2^-8 |O_plain| + 2^-12 a
elementwise, with a = sum_j p_j |v_j| / l and b = sum_j |v_j| / l from the
oracle; 2^-8 |O| is the bf16 rounding of O and 2^-12 a covers the fp32
arithmetic (exponentials, sums). The bound holds whatever running max each
weight is rounded against, so it does not depend on the kernel's tiling:
the GPU is judged against the plain definition only. The LSE carries no
rounding of P: |LSE - LSE_ref| <= 1e-3 (the 16-bit path's bound).
"""
import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


def run_fp8(fa2, q, k, v, qd, kd, vd, scale):
    import torch

    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda")
    o, lse = fa2.fa2_fwd_fp8(dev(q), dev(k), dev(v), dev(qd), dev(kd), dev(vd), scale=scale)
    assert fa2.fa2_check_status(torch.cuda.current_stream().cuda_stream) == fa2.FA2_OK
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def run_fp8_ex(fa2, q, k, v, qd, kd, vd, scale, causal):
    import torch

    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to("cuda")
    o, lse = fa2.fa2_fwd_fp8_ex(dev(q), dev(k), dev(v), dev(qd), dev(kd), dev(vd), scale=scale, causal=causal)
    assert fa2.fa2_check_status(torch.cuda.current_stream().cuda_stream) == fa2.FA2_OK
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def assert_fp8_parity(o, lse, q, k, v, qd, kd, vd, scale, rows=None, what="", causal=False):
    op, lp, a, b = oracle.attention_fp8(q, k, v, qd, kd, vd, scale, round_p=False, rows=rows, causal=causal)
    d = q.shape[-1]
    if rows is not None:
        o = o.reshape(-1, d)[rows]
        lse = lse.reshape(-1)[rows]
    o, op, a, b = (x.reshape(-1, d) for x in (o, op, a, b))
    assert np.isfinite(o).all(), what
    bound = 2.0 ** -4 * a + 2.0 ** -18 * b + 2.0 ** -8 * np.abs(op) + 2.0 ** -12 * a + 1e-7
    err = np.abs(o - op)
    bad = err > bound
    worst = float((err / bound).max()) if err.size else 0.0
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond the rounding bound, worst ratio {worst:.3g}"
    lse, lp = lse.reshape(-1), lp.reshape(-1)
    empty = np.isneginf(lp)                 # rows that see no key: o = 0, lse = -inf
    assert np.array_equal(np.isneginf(lse), empty), what
    assert not o[empty].any(), what
    assert np.max(np.abs(lse[~empty] - lp[~empty]), initial=0.0) <= 1e-3, what
    return worst


CASES = [
    # B, Hq, Hkv, N, amp
    (1, 1, 1, 128, 1.0),      # one tile, one KV tile
    (1, 2, 1, 256, 1.0),      # grouped heads, two KV tiles
    (1, 1, 1, 384, 1.0),      # three query tiles: an item with one tile
    (2, 4, 2, 1024, 1.0),     # grouped heads, eight KV tiles
    (1, 4, 4, 1024, 3.0),     # sharp softmax: many rescales, large logits
    (2, 16, 16, 1024, 1.0),   # 256 items on 152 SMs: CTAs take several items
]


@pytest.mark.parametrize("B,Hq,Hkv,N,amp", CASES)
def test_fp8_matches_oracle(gpu_lib, B, Hq, Hkv, N, amp):
    q, k, v, qd, kd, vd = gen.make_qkv_fp8(7000 + N + Hq + int(amp), B, Hq, Hkv, N, 128, amp)
    scale = 128 ** -0.5
    o, lse = run_fp8(gpu_lib, q, k, v, qd, kd, vd, scale)
    assert_fp8_parity(o, lse, q, k, v, qd, kd, vd, scale, what=f"B{B} Hq{Hq} Hkv{Hkv} N{N} x{amp}")


@pytest.mark.parametrize("log2_step,causal", [(0.5, False), (1.0, False), (3.0, False), (1.0, True)])
def test_fp8_running_max_grows_in_steps(gpu_lib, log2_step, causal):
    """Row maxima growing by about 0.5 (1, 3) log2 units per KV tile: every
    tile's weights are rounded to e4m3 against a new running max and O is
    rescaled, also in the general (causal) mode; the step is checked on the
    decoded inputs."""
    B, Hq, Hkv, N, d = 1, 2, 2, 1280, 128
    rng = np.random.default_rng(int(log2_step * 100))
    scale = d ** -0.5
    qf = 0.5 + 0.02 * rng.standard_normal((B, Hq, N, d))
    tile = (np.arange(N) // 128).astype(np.float64)
    kf = (tile * log2_step / np.log2(np.e) / (scale * 0.5 * d))[None, None, :, None] + 0.02 * rng.standard_normal((B, Hkv, N, d))
    vf = rng.standard_normal((B, Hkv, N, d))
    ones = np.ones(B * Hkv, dtype=np.float32)
    q, k, v = gen.e4m3_encode(qf), gen.e4m3_encode(kf), gen.e4m3_encode(vf)
    dec = lambda c: np.where(c & 0x80, -1.0, 1.0) * gen._E4M3[np.minimum(c & 0x7F, 126)]
    s = dec(q[0, 0]) @ dec(k[0, 0]).T * scale * np.log2(np.e)
    steps = np.diff(s.reshape(N, N // 128, 128).max(axis=2), axis=1)
    assert abs(float(np.median(steps)) - log2_step) < 0.25 * log2_step + 0.1, float(np.median(steps))
    if causal:
        o, lse = run_fp8_ex(gpu_lib, q, k, v, ones, ones, ones, scale, True)
    else:
        o, lse = run_fp8(gpu_lib, q, k, v, ones, ones, ones, scale)
    assert_fp8_parity(o, lse, q, k, v, ones, ones, ones, scale, what=f"running max +{log2_step} a tile",
                      causal=causal)


def test_fp8_descales_are_applied(gpu_lib):
    # A descale changes only its own group, by its own factor: a power of two
    # on v's descale scales that group's O exactly and leaves its LSE alone.
    B, Hq, Hkv, N = 2, 2, 1, 256                         # two groups: batch 0 and batch 1
    q, k, v, qd, kd, vd = gen.make_qkv_fp8(7101, B, Hq, Hkv, N, 128)
    vd2 = vd * np.array([1.0, 4.0], dtype=np.float32)
    o1, l1 = run_fp8(gpu_lib, q, k, v, qd, kd, vd, 0.09)
    o2, l2 = run_fp8(gpu_lib, q, k, v, qd, kd, vd2, 0.09)
    assert np.array_equal(o1[0], o2[0]) and np.array_equal(l1, l2)
    assert np.array_equal(o1[1] * 4.0, o2[1])          # power-of-two factor: exact in bf16
    assert_fp8_parity(o2, l2, q, k, v, qd, kd, vd2, 0.09, what="vd x4")
    kd2 = kd * np.float32(2.0)
    o3, l3 = run_fp8(gpu_lib, q, k, v, qd, kd2, vd, 0.09)
    assert_fp8_parity(o3, l3, q, k, v, qd, kd2, vd, 0.09, what="kd x2")


def test_fp8_constant_values(gpu_lib):
    # V = 2 everywhere: the plain result is exactly 2; the method's is within
    # 2^-4 of it (P rounding) -- and every row's weights still sum to l.
    B, Hq, Hkv, N = 1, 2, 1, 512
    q, k, _, qd, kd, _ = gen.make_qkv_fp8(7102, B, Hq, Hkv, N, 128)
    v = np.full((B, Hkv, N, 128), 0x40, dtype=np.uint8)
    vd = np.ones(B * Hkv, dtype=np.float32)
    o, lse = run_fp8(gpu_lib, q, k, v, qd, kd, vd, 0.1)
    assert np.max(np.abs(o - 2.0)) <= 2.0 ** -4 * 2.0 + 2.0 ** -7
    assert_fp8_parity(o, lse, q, k, v, qd, kd, vd, 0.1, what="V = 2")


def test_fp8_accepts_torch_float8_tensors(gpu_lib):
    import torch

    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    q, k, v, qd, kd, vd = gen.make_qkv_fp8(7103, 1, 2, 2, 256, 128)
    t = lambda x: torch.from_numpy(x).to("cuda").view(torch.float8_e4m3fn)
    f = lambda x: torch.from_numpy(x).to("cuda")
    o, lse = gpu_lib.fa2_fwd_fp8(t(q), t(k), t(v), f(qd), f(kd), f(vd), scale=0.1)
    o2, lse2 = run_fp8(gpu_lib, q, k, v, qd, kd, vd, 0.1)
    assert np.array_equal(o.float().cpu().numpy(), o2) and np.array_equal(lse.cpu().numpy(), lse2)


def test_fp8_full_size_bench_workload(gpu_lib):
    # The workload bench.py times for FP8, in the same launch configuration:
    # every element against the oracle's plain definition.
    w = gen.workload("fp8_mha_B4_H16_N4096_d128_e4m3")
    q, k, v, qd, kd, vd = w.inputs()
    o, lse = run_fp8(gpu_lib, q, k, v, qd, kd, vd, w.scale)
    assert_fp8_parity(o, lse, q, k, v, qd, kd, vd, w.scale, what=w.name)


def test_fp8_rejects_unsupported_head_dim(gpu_lib):
    import torch

    q = torch.zeros((1, 1, 128, 64), dtype=torch.uint8, device="cuda")
    ds = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(gpu_lib.FA2Error):
        gpu_lib.fa2_fwd_fp8(q, q, q, ds, ds, ds)


# ------------------------------------------------------------ general mode

def fp8_general_inputs(seed, B, Hq, Hkv, nq, nk, amp=1.0):
    q, _, _, qd, _, _ = gen.make_qkv_fp8(seed, B, Hq, Hkv, nq, 128, amp)
    _, k, v, _, kd, vd = gen.make_qkv_fp8(seed + 1, B, Hq, Hkv, nk, 128, amp)
    return q, k, v, qd, kd, vd


GEN_CASES = [
    # B, Hq, Hkv, Nq, Nk, causal
    (1, 2, 1, 128, 128, True),      # one tile: the diagonal tile only
    (1, 2, 2, 200, 200, True),      # ragged, causal, two query tiles in one item
    (2, 4, 2, 300, 500, False),     # unequal lengths, ragged key tail
    (1, 2, 1, 500, 300, True),      # Nq > Nk: the first 200 rows see no key
    (1, 1, 1, 1, 1, False),         # one query, one key
    (1, 2, 1, 1, 700, True),        # one query row (decode) over 700 keys
    (1, 4, 1, 1000, 1000, True),    # causal over eight key tiles, grouped heads
    (2, 2, 1, 129, 129, False),     # one row past a tile
    (1, 2, 1, 640, 384, True),      # items with different KV tile counts per tile
    (2, 8, 8, 1024, 1024, True),    # 64 items of unequal work on the persistent grid
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,causal", GEN_CASES)
def test_fp8_general_matches_oracle(gpu_lib, B, Hq, Hkv, Nq, Nk, causal):
    q, k, v, qd, kd, vd = fp8_general_inputs(7200 + Nq + 3 * Nk + Hq, B, Hq, Hkv, Nq, Nk)
    scale = 128 ** -0.5
    o, lse = run_fp8_ex(gpu_lib, q, k, v, qd, kd, vd, scale, causal)
    assert o.shape == (B, Hq, Nq, 128) and lse.shape == (B, Hq, Nq)
    assert_fp8_parity(o, lse, q, k, v, qd, kd, vd, scale, causal=causal,
                      what=f"B{B} Hq{Hq} Hkv{Hkv} Nq{Nq} Nk{Nk} causal{causal}")


def test_fp8_general_sharp_softmax_and_zero_descale(gpu_lib):
    # amp 3: large logits and many rescales under the mask; then a zero k
    # descale: every score is 0, so each row averages its visible values.
    q, k, v, qd, kd, vd = fp8_general_inputs(7301, 1, 2, 1, 384, 384, amp=3.0)
    o, lse = run_fp8_ex(gpu_lib, q, k, v, qd, kd, vd, 0.09, True)
    assert_fp8_parity(o, lse, q, k, v, qd, kd, vd, 0.09, causal=True, what="causal x3")
    kd0 = np.zeros_like(kd)
    o, lse = run_fp8_ex(gpu_lib, q, k, v, qd, kd0, vd, 0.09, True)
    assert_fp8_parity(o, lse, q, k, v, qd, kd0, vd, 0.09, causal=True, what="k descale 0")
    assert np.allclose(lse[0, 0], np.log(np.arange(1, 385)), atol=1e-3)


def test_fp8_general_equal_lengths_route_to_the_packed_kernel(gpu_lib):
    # Non-causal, N_q == N_k, N % 128 == 0: fa2_fwd_fp8_ex gives fa2_fwd_fp8's
    # result bit for bit.
    q, k, v, qd, kd, vd = gen.make_qkv_fp8(7302, 1, 4, 2, 256, 128)
    o1, l1 = run_fp8(gpu_lib, q, k, v, qd, kd, vd, 0.1)
    o2, l2 = run_fp8_ex(gpu_lib, q, k, v, qd, kd, vd, 0.1, False)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_fp8_general_causal_full_size(gpu_lib):
    # The FP8 bench workload (B 4, H 16, N 4096) with the causal mask: every
    # element against the oracle's plain definition.
    w = gen.workload("fp8_mha_B4_H16_N4096_d128_e4m3")
    q, k, v, qd, kd, vd = w.inputs()
    o, lse = run_fp8_ex(gpu_lib, q, k, v, qd, kd, vd, w.scale, True)
    assert_fp8_parity(o, lse, q, k, v, qd, kd, vd, w.scale, causal=True, what=w.name + " causal")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_many_short_items_per_cta(gpu_lib, causal):
    # 512 short items (one or two KV tiles) on at most 152 CTAs: several items
    # per CTA, so the epilogue's statistics slots alternate every item. Five
    # launches agree bit for bit and with the oracle.
    B, Hq, Hkv, N = (4, 128, 128, 256) if causal else (4, 256, 128, 128)
    q, k, v, qd, kd, vd = gen.make_qkv_fp8(7400 + int(causal), B, Hq, Hkv, N, 128)
    scale = 128 ** -0.5
    o, lse = run_fp8_ex(gpu_lib, q, k, v, qd, kd, vd, scale, causal)
    assert_fp8_parity(o, lse, q, k, v, qd, kd, vd, scale, causal=causal, what=f"512 short items causal={causal}")
    for _ in range(4):
        o2, l2 = run_fp8_ex(gpu_lib, q, k, v, qd, kd, vd, scale, causal)
        assert np.array_equal(o2, o) and np.array_equal(l2, lse)

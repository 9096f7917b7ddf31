"""Parity of the general entry point (fa2_fwd_ex: unequal and ragged lengths,
causal mask) with the fp64 oracle, through the C ABI.

Same tolerances as the plain path: |O_gpu - O_ref| <= 1e-2 + 1e-2*|O_ref|
(bf16) or 5e-3 + 5e-3*|O_ref| (fp16), |LSE_gpu - LSE_ref| <= 1e-3; rows with
no allowed key must give exactly O = 0 and LSE = -inf.
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


def inputs(seed, B, Hq, Hkv, Nq, Nk, d, dtype, amp=1.0):
    q, _, _ = gen.make_qkv(seed, B, Hq, Hkv, Nq, d, dtype, amp)
    _, k, v = gen.make_qkv(seed + 1, B, Hq, Hkv, Nk, d, dtype, amp)
    return q, k, v


def run_ex(fa2, q, k, v, dtype, scale, causal):
    import torch

    o, lse = fa2.fa2_fwd_ex(to_dev(q, dtype), to_dev(k, dtype), to_dev(v, dtype), scale=scale, causal=causal)
    assert fa2.fa2_check_status(torch.cuda.current_stream().cuda_stream) == fa2.FA2_OK
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def assert_parity(o, lse, o_ref, lse_ref, dtype, what):
    t = 1e-2 if dtype == gen.BF16 else 5e-3
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf rows differ"
    assert np.all(o[empty] == 0.0), f"{what}: empty rows must be 0"
    full = ~empty
    err = np.abs(o[full] - o_ref[full])
    bad = err > t + t * np.abs(o_ref[full])
    assert not bad.any(), f"{what}: {int(bad.sum())} O elements out of tolerance, worst {err.max():.4g}"
    if full.any():
        assert np.max(np.abs(lse[full] - lse_ref[full])) <= 1e-3, what
    assert np.isfinite(o).all()


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, dtype, causal, amp
    (1, 1, 1, 128, 128, 128, gen.BF16, True, 1.0),
    (1, 2, 2, 512, 512, 128, gen.BF16, True, 1.0),
    (2, 4, 2, 384, 384, 64, gen.FP16, True, 1.0),     # odd tile count per head
    (1, 2, 2, 200, 200, 128, gen.BF16, False, 1.0),   # ragged, non-causal
    (1, 2, 1, 200, 200, 128, gen.BF16, True, 1.0),    # ragged, causal, grouped heads
    (1, 2, 2, 100, 300, 128, gen.BF16, False, 1.0),   # Nq < Nk
    (1, 2, 2, 100, 300, 64, gen.BF16, True, 1.0),     # causal, Nq < Nk
    (1, 2, 2, 300, 100, 128, gen.BF16, True, 1.0),    # causal, Nq > Nk: empty rows
    (1, 1, 1, 1, 1, 128, gen.BF16, False, 1.0),
    (1, 1, 1, 1, 1000, 64, gen.BF16, True, 1.0),
    (1, 1, 1, 1000, 1, 64, gen.BF16, True, 1.0),      # only the last row attends
    (1, 2, 2, 1000, 1000, 128, gen.BF16, True, 3.0),  # sharp softmax, causal
    (2, 4, 4, 129, 257, 128, gen.FP16, False, 1.0),
    (1, 8, 2, 640, 640, 128, gen.BF16, True, 1.0),    # grouped heads, causal
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,dtype,causal,amp", CASES)
def test_general_every_element(gpu_lib, B, Hq, Hkv, Nq, Nk, d, dtype, causal, amp):
    q, k, v = inputs(3000 + Nq + 7 * Nk + d, B, Hq, Hkv, Nq, Nk, d, dtype, amp)
    scale = 1 / math.sqrt(d)
    o, lse = run_ex(gpu_lib, q, k, v, dtype, scale, causal)
    o_ref, lse_ref = oracle.attention_ex(q, k, v, scale, dtype, causal=causal)
    assert_parity(o, lse, o_ref, lse_ref, dtype, f"B{B} Hq{Hq} Hkv{Hkv} Nq{Nq} Nk{Nk} d{d} causal{causal}")


@pytest.mark.parametrize("log2_step", [4.0, 12.0])
def test_causal_running_max_grows_in_steps(gpu_lib, log2_step):
    """Causal and ragged (N = 1000), row maxima growing by about 4 (12) log2
    units per KV tile: the general mode rescales O on every tile, with
    masked keys in the diagonal tiles."""
    N, d = 1000, 128
    rng = np.random.default_rng(int(log2_step))
    scale = d ** -0.5
    qv = np.full((1, 2, N, d), 0.5) + 0.02 * rng.standard_normal((1, 2, N, d))
    tile = (np.arange(N) // 128).astype(np.float64)
    kv = (tile * log2_step / np.log2(np.e) / (scale * 0.5 * d))[None, None, :, None] + 0.02 * rng.standard_normal((1, 2, N, d))
    q, k = gen.round_to_16bit(qv, gen.BF16), gen.round_to_16bit(kv, gen.BF16)
    v = gen.round_to_16bit(rng.standard_normal((1, 2, N, d)), gen.BF16)
    o, lse = run_ex(gpu_lib, q, k, v, gen.BF16, scale, True)
    o_ref, lse_ref = oracle.attention_ex(q, k, v, scale, gen.BF16, causal=True)
    assert_parity(o, lse, o_ref, lse_ref, gen.BF16, f"causal running max +{log2_step} a tile")


def test_causal_zero_queries_give_prefix_means(gpu_lib):
    Nq = Nk = 384
    _, k, v = inputs(3100, 1, 2, 2, Nq, Nk, 128, gen.BF16)
    q = np.zeros((1, 2, Nq, 128), np.uint16)
    o, lse = run_ex(gpu_lib, q, k, v, gen.BF16, 128 ** -0.5, True)
    vd = oracle.decode16(v, gen.BF16)
    ref = np.cumsum(vd, axis=2) / np.arange(1, Nk + 1)[None, None, :, None]
    assert_parity(o, lse, ref, np.broadcast_to(np.log(np.arange(1, Nq + 1)), lse.shape), gen.BF16,
                  "causal Q=0")


def test_plain_case_matches_fast_entry_bitwise(gpu_lib):
    import torch

    q, k, v = gen.make_qkv(3200, 1, 4, 2, 256, 128, gen.BF16)
    tq, tk, tv = (to_dev(x, gen.BF16) for x in (q, k, v))
    o1, l1 = gpu_lib.fa2_fwd_gqa(tq, tk, tv, scale=0.1)
    o2, l2 = gpu_lib.fa2_fwd_ex(tq, tk, tv, scale=0.1, causal=False)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_general_path_on_multiple_of_128_agrees_with_fast_path(gpu_lib):
    """Causal=False with unequal multiples of 128 runs the general kernel."""
    q, k, v = inputs(3300, 1, 2, 2, 256, 384, 128, gen.BF16)
    o, lse = run_ex(gpu_lib, q, k, v, gen.BF16, 0.09, False)
    o_ref, lse_ref = oracle.attention_ex(q, k, v, 0.09, gen.BF16, causal=False)
    assert_parity(o, lse, o_ref, lse_ref, gen.BF16, "general 256x384")


def test_causal_full_size(gpu_lib):
    """B=4, H=16, N=4096, d=128, causal (the causal benchmark's workload and
    launch): every element against the oracle."""
    import torch

    w = gen.workload("mha_B4_H16_N4096_d128_bf16")
    q, k, v = w.inputs()
    o, lse = gpu_lib.fa2_fwd_ex(to_dev(q, w.dtype), to_dev(k, w.dtype), to_dev(v, w.dtype),
                                scale=w.scale, causal=True)
    assert gpu_lib.fa2_check_status(torch.cuda.current_stream().cuda_stream) == gpu_lib.FA2_OK
    o_ref, lse_ref = oracle.attention_ex(q, k, v, w.scale, w.dtype, causal=True)
    assert_parity(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                  o_ref, lse_ref, w.dtype, "causal B4 H16 N4096")
    assert bool(torch.isfinite(o.float()).all())


def test_causal_many_short_items_per_cta(gpu_lib):
    # Causal, N = 256: 512 items whose first tile has one KV tile and the
    # second two, several per CTA (the epilogue's statistics slots alternate
    # every item). Five launches agree bit for bit and with the oracle.
    B, H, N, d = 4, 128, 256, 128
    q, k, v = inputs(1402, B, H, H, N, N, d, gen.BF16)
    scale = d ** -0.5
    o, lse = run_ex(gpu_lib, q, k, v, gen.BF16, scale, True)
    o_ref, lse_ref = oracle.attention_ex(q, k, v, scale, gen.BF16, causal=True)
    assert_parity(o, lse, o_ref, lse_ref, gen.BF16, "causal N=256 x 512 heads")
    for _ in range(4):
        o2, l2 = run_ex(gpu_lib, q, k, v, gen.BF16, scale, True)
        assert np.array_equal(o2, o) and np.array_equal(l2, lse)

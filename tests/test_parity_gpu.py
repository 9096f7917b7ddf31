"""Parity of the sm_103a kernel (through the C ABI) with the fp64 oracle.

Tolerances (fixed by the workload definition): |O_gpu - O_ref| <= 1e-2 +
1e-2*|O_ref| for bf16 and 5e-3 + 5e-3*|O_ref| for fp16, elementwise, and
|LSE_gpu - LSE_ref| <= 1e-3. O_ref is the unrounded fp64 result.
"""
import math

import numpy as np
import pytest

import gen
import oracle

pytestmark = pytest.mark.gpu


def _torch():
    import torch

    return torch


def to_dev(x, dtype):
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to("cuda")
    return t.view(torch.bfloat16 if dtype == gen.BF16 else torch.float16)


def run_gpu(fa2, q, k, v, dtype, scale, stream=None):
    torch = _torch()
    tq, tk, tv = (to_dev(x, dtype) for x in (q, k, v))
    o, lse = fa2.fa2_fwd_gqa(tq, tk, tv, scale=scale, stream=stream)
    s = stream if stream is not None else torch.cuda.current_stream()
    assert fa2.fa2_check_status(s.cuda_stream) == fa2.FA2_OK
    return o, lse


def tol(dtype):
    return 1e-2 if dtype == gen.BF16 else 5e-3


def assert_parity(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    t = tol(dtype)
    err = np.abs(o_gpu - o_ref)
    bound = t + t * np.abs(o_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} O elements out of tolerance; "
                           f"worst |dO|={err.max():.4g} at {np.unravel_index(err.argmax(), err.shape)}")
    lerr = np.abs(lse_gpu - lse_ref)
    assert lerr.max() <= 1e-3, f"{what}: max |dLSE|={lerr.max():.4g}"
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all()


def full_check(fa2, q, k, v, dtype, scale, what=""):
    o, lse = run_gpu(fa2, q, k, v, dtype, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, dtype)
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, dtype, what)
    return o, lse


# ------------------------------------------------------------------ small shapes, every element

SMALL = [
    # B, Hq, Hkv, N, d, dtype, amp
    (1, 1, 1, 128, 128, gen.BF16, 1.0),
    (1, 1, 1, 128, 64, gen.FP16, 1.0),
    (2, 3, 3, 256, 128, gen.BF16, 1.0),
    (1, 2, 2, 384, 64, gen.BF16, 1.0),
    (1, 3, 1, 384, 128, gen.FP16, 1.0),    # 9 packed query tiles: last CTA has one tile
    (2, 4, 2, 640, 128, gen.BF16, 3.0),
    (1, 2, 2, 1024, 64, gen.BF16, 3.0),
    (1, 1, 1, 2048, 128, gen.FP16, 1.0),
    (1, 2, 2, 512, 128, gen.BF16, 6.0),    # very sharp softmax
    (1, 8, 2, 256, 64, gen.FP16, 3.0),
    # d = 64 runs four query tiles per item: items of 2, of 4 + 1, of 4 + 3
    (2, 3, 3, 256, 64, gen.BF16, 1.0),
    (1, 5, 1, 256, 64, gen.FP16, 1.0),
    (1, 7, 7, 768, 64, gen.BF16, 3.0),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,amp", SMALL)
def test_small_shapes_every_element(gpu_lib, B, Hq, Hkv, N, d, dtype, amp):
    q, k, v = gen.make_qkv(2000 + N + d + Hq, B, Hq, Hkv, N, d, dtype, amp)
    full_check(gpu_lib, q, k, v, dtype, 1 / math.sqrt(d), f"B{B} Hq{Hq} Hkv{Hkv} N{N} d{d}")


# ------------------------------------------------------------------ the planner's other d = 64 kernel

@pytest.mark.parametrize("B,Hq,Hkv,N,dtype,amp", [
    (1, 2, 2, 384, gen.BF16, 1.0),     # one item of three tiles
    (1, 8, 2, 256, gen.FP16, 3.0),
    (2, 3, 3, 1024, gen.BF16, 3.0),    # the d = 64 workload's input scale
])
def test_d64_shared_kernel_every_element(gpu_lib, B, Hq, Hkv, N, dtype, amp):
    """d = 64 with equal lengths on the 16-bit kernel's d = 64 path (P over S),
    selected through the planner hook instead of the default d = 64 kernel."""
    q, k, v = gen.make_qkv(4000 + N + Hq, B, Hq, Hkv, N, 64, dtype, amp)
    old = gpu_lib.fa2_set_tile_config(gpu_lib.TILE_CFG_D64_SHARED)
    try:
        full_check(gpu_lib, q, k, v, dtype, 1 / 8, f"shared d64 B{B} Hq{Hq} Hkv{Hkv} N{N}")
    finally:
        gpu_lib.fa2_set_tile_config(old)


# ------------------------------------------------------------------ degenerate and adversarial inputs

@pytest.mark.parametrize("d", [64, 128])
def test_zero_queries_give_mean_of_values(gpu_lib, d):
    _, k, v = gen.make_qkv(31, 1, 2, 2, 384, d, gen.BF16)
    q = np.zeros((1, 2, 384, d), np.uint16)
    o, lse = run_gpu(gpu_lib, q, k, v, gen.BF16, d ** -0.5)
    vd = oracle.decode16(v, gen.BF16)
    mean = np.broadcast_to(vd.mean(axis=2, keepdims=True), (1, 2, 384, d))
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), mean,
                  np.full((1, 2, 384), math.log(384)), gen.BF16, "Q=0")


def test_constant_values_give_constant_output(gpu_lib):
    q, k, _ = gen.make_qkv(32, 2, 2, 2, 256, 128, gen.FP16, 3.0)
    v = np.full(k.shape, 0x3C00, np.uint16)  # fp16 1.0
    o, _ = run_gpu(gpu_lib, q, k, v, gen.FP16, 128 ** -0.5)
    np.testing.assert_allclose(o.float().cpu().numpy(), 1.0, rtol=0, atol=5e-3)


@pytest.mark.parametrize("increasing", [True, False])
def test_running_max_moves_every_tile(gpu_lib, increasing):
    """Scores grow (or shrink) by about 8 log2 units per KV tile, so the
    running-max rescale of O runs on every tile (or never after the first)."""
    N, d = 1024, 128
    rng = np.random.default_rng(5)
    q = gen.round_to_16bit(np.abs(rng.standard_normal((1, 2, N, d))) * 0.5 + 0.25, gen.BF16)
    step = (np.arange(N) // 128).astype(np.float64)
    if not increasing:
        step = step[::-1]
    kv = step[None, None, :, None] * 0.7 + 0.05 * rng.standard_normal((1, 2, N, d))
    k = gen.round_to_16bit(kv, gen.BF16)
    v = gen.round_to_16bit(rng.standard_normal((1, 2, N, d)), gen.BF16)
    full_check(gpu_lib, q, k, v, gen.BF16, d ** -0.5, f"monotone max increasing={increasing}")


@pytest.mark.parametrize("log2_step,dtype", [(4.0, gen.BF16), (12.0, gen.FP16), (7.5, gen.BF16)])
def test_running_max_grows_in_steps(gpu_lib, log2_step, dtype):
    """Scores whose row max grows by about 4 (12, 7.5) log2 units per KV
    tile: a rescale of O on every tile by a factor of 2^-4 (2^-12, 2^-7.5),
    with the weights of the earlier tiles fading; the step is checked on the
    inputs."""
    N, d = 1536, 128
    rng = np.random.default_rng(int(log2_step * 10))
    qv = np.full((1, 2, N, d), 0.5) + 0.02 * rng.standard_normal((1, 2, N, d))
    tile = (np.arange(N) // 128).astype(np.float64)
    scale = d ** -0.5
    # s = scale * q.k: a per-tile offset of log2_step / log2(e) natural units
    kv = (tile * log2_step / np.log2(np.e) / (scale * 0.5 * d))[None, None, :, None] + 0.02 * rng.standard_normal((1, 2, N, d))
    q, k = gen.round_to_16bit(qv, dtype), gen.round_to_16bit(kv, dtype)
    v = gen.round_to_16bit(rng.standard_normal((1, 2, N, d)), dtype)
    s = gen.bits_to_float32(q, dtype)[0, 0].astype(np.float64) @ gen.bits_to_float32(k, dtype)[0, 0].astype(np.float64).T
    tile_max = (s * scale * np.log2(np.e)).reshape(N, N // 128, 128).max(axis=2)
    steps = np.diff(tile_max, axis=1)
    assert abs(float(np.median(steps)) - log2_step) < 0.5, float(np.median(steps))
    full_check(gpu_lib, q, k, v, dtype, scale, f"running max +{log2_step} log2 units a tile")


def test_one_dominant_key_per_row(gpu_lib):
    N, d = 512, 64
    rng = np.random.default_rng(6)
    qv = rng.standard_normal((1, 1, N, d))
    kv = rng.standard_normal((1, 1, N, d)) * 0.1
    # key j = 5*i mod N aligns strongly with query i for a few queries
    for i in range(0, N, 7):
        kv[0, 0, (5 * i) % N] = 4.0 * qv[0, 0, i]
    q, k = gen.round_to_16bit(qv, gen.BF16), gen.round_to_16bit(kv, gen.BF16)
    v = gen.round_to_16bit(rng.standard_normal((1, 1, N, d)), gen.BF16)
    full_check(gpu_lib, q, k, v, gen.BF16, d ** -0.5, "dominant keys")


def test_key_shift_leaves_output_unchanged(gpu_lib):
    N, d = 256, 128
    rng = np.random.default_rng(7)
    q = gen.round_to_16bit(rng.integers(-2, 3, (1, 2, N, d)).astype(float) * 0.25, gen.BF16)
    kint = rng.integers(-2, 3, (1, 2, N, d)).astype(float) * 0.25
    c = rng.integers(-2, 3, d).astype(float) * 0.25
    k1 = gen.round_to_16bit(kint, gen.BF16)
    k2 = gen.round_to_16bit(kint + c, gen.BF16)
    v = gen.round_to_16bit(rng.standard_normal((1, 2, N, d)), gen.BF16)
    o1, l1 = run_gpu(gpu_lib, q, k1, v, gen.BF16, d ** -0.5)
    o2, l2 = run_gpu(gpu_lib, q, k2, v, gen.BF16, d ** -0.5)
    o_ref, lse_ref = oracle.attention(q, k1, v, d ** -0.5, gen.BF16)
    assert_parity(o1.float().cpu().numpy(), l1.cpu().numpy(), o_ref, lse_ref, gen.BF16, "unshifted")
    qd = oracle.decode16(q, gen.BF16)
    shift = (qd @ c) * d ** -0.5
    assert_parity(o2.float().cpu().numpy(), l2.cpu().numpy(), o_ref, lse_ref + shift, gen.BF16,
                  "shifted keys")


def test_joint_permutation_of_keys_and_values(gpu_lib):
    q, k, v = gen.make_qkv(33, 1, 2, 2, 512, 128, gen.BF16)
    perm = np.random.default_rng(8).permutation(512)
    o1, l1 = run_gpu(gpu_lib, q, k, v, gen.BF16, 128 ** -0.5)
    o2, l2 = run_gpu(gpu_lib, q, k[:, :, perm].copy(), v[:, :, perm].copy(), gen.BF16, 128 ** -0.5)
    np.testing.assert_allclose(o1.float().cpu().numpy(), o2.float().cpu().numpy(), rtol=1e-2, atol=1e-2)
    np.testing.assert_allclose(l1.cpu().numpy(), l2.cpu().numpy(), rtol=0, atol=1e-3)


def test_grouped_heads_match_repeated_heads(gpu_lib):
    torch = _torch()
    q, k, v = gen.make_qkv(34, 2, 8, 2, 256, 128, gen.BF16)
    o1, l1 = run_gpu(gpu_lib, q, k, v, gen.BF16, 128 ** -0.5)
    kr, vr = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
    o2, l2 = run_gpu(gpu_lib, q, kr, vr, gen.BF16, 128 ** -0.5)
    # same query rows against the same keys in the same order: bitwise equal
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_batch_and_head_independence(gpu_lib):
    torch = _torch()
    q, k, v = gen.make_qkv(35, 2, 3, 3, 256, 64, gen.FP16)
    o, lse = run_gpu(gpu_lib, q, k, v, gen.FP16, 0.125)
    for b, h in ((0, 0), (1, 2), (0, 1)):
        o1, l1 = run_gpu(gpu_lib, q[b:b + 1, h:h + 1].copy(), k[b:b + 1, h:h + 1].copy(),
                         v[b:b + 1, h:h + 1].copy(), gen.FP16, 0.125)
        assert torch.equal(o1[0, 0], o[b, h]) and torch.equal(l1[0, 0], lse[b, h])


def test_side_stream_and_preallocated_outputs(gpu_lib):
    torch = _torch()
    q, k, v = gen.make_qkv(36, 1, 2, 2, 256, 128, gen.BF16)
    tq, tk, tv = (to_dev(x, gen.BF16) for x in (q, k, v))
    o = torch.full_like(tq, 7.0)
    lse = torch.full((1, 2, 256), 7.0, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gpu_lib.fa2_fwd(tq, tk, tv, o, lse, scale=128 ** -0.5, stream=s)
    assert gpu_lib.fa2_check_status(s.cuda_stream) == gpu_lib.FA2_OK
    o_ref, lse_ref = oracle.attention(q, k, v, 128 ** -0.5, gen.BF16)
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, gen.BF16, "side stream")


def test_invalid_arguments_launch_nothing(gpu_lib):
    torch = _torch()
    q, k, v = gen.make_qkv(37, 1, 1, 1, 128, 128, gen.BF16)
    tq, tk, tv = (to_dev(x, gen.BF16) for x in (q, k, v))
    o = torch.full_like(tq, 3.0)
    lse = torch.full((1, 1, 128), 3.0, device="cuda")
    f = gpu_lib.fa2_fwd_ptr
    args = [tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr()]
    assert f(*args, 1, 1, 128, 128, -1.0, 0) == gpu_lib.FA2_ERR_INVALID_ARG
    assert f(*args, 1, 1, 128, 96, 0.1, 0) == gpu_lib.FA2_ERR_UNSUPPORTED
    assert f(*args, 1, 1, 100, 128, 0.1, 0) == gpu_lib.FA2_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((o == 3.0).all()) and bool((lse == 3.0).all())
    assert gpu_lib.fa2_check_status(0) == gpu_lib.FA2_OK


def test_long_sequence_single_head(gpu_lib):
    """N = 32768 (256 KV tiles): sampled rows against the oracle."""
    N, d = 32768, 128
    q, k, v = gen.make_qkv(38, 1, 2, 1, N, d, gen.BF16)
    o, lse = run_gpu(gpu_lib, q, k, v, gen.BF16, d ** -0.5)
    rows = sample_rows(1, 2, N, 48, seed=1)
    check_rows(o, lse, q, k, v, gen.BF16, d ** -0.5, rows, "N=32768")


# ------------------------------------------------------------------ watchdog

@pytest.mark.parametrize("d", [128, 64])   # d = 64: the kernel with two MMA warps
def test_watchdog_reports_timeout_and_context_survives(gpu_lib, d):
    torch = _torch()
    q, k, v = gen.make_qkv(39, 1, 1, 1, 256, d, gen.BF16)
    tq, tk, tv = (to_dev(x, gen.BF16) for x in (q, k, v))
    old_limit = gpu_lib.fa2_set_wait_limit_ns(20_000_000)  # 20 ms
    old_flags = gpu_lib.fa2_set_debug_flags(1)              # skip the query-tile loads
    try:
        gpu_lib.fa2_fwd(tq, tk, tv, scale=d ** -0.5)
        rc = gpu_lib.fa2_check_status(torch.cuda.current_stream().cuda_stream)
    finally:
        gpu_lib.fa2_set_debug_flags(old_flags)
        gpu_lib.fa2_set_wait_limit_ns(old_limit)
    assert rc == gpu_lib.FA2_ERR_TIMEOUT
    assert gpu_lib.fa2_check_status(0) == gpu_lib.FA2_OK  # the word was cleared
    full_check(gpu_lib, q, k, v, gen.BF16, d ** -0.5, "after watchdog")


def test_check_status_reads_the_streams_device_word(gpu_lib):
    """fa2_check_status(stream) reports a timeout of a kernel queued on a side
    stream (the status word of that stream's device), clears it, and leaves
    the current device as it found it; the word is shared by the device's
    streams, so a later check on the default stream sees it cleared."""
    torch = _torch()
    q, k, v = gen.make_qkv(40, 1, 1, 1, 256, 128, gen.BF16)
    tq, tk, tv = (to_dev(x, gen.BF16) for x in (q, k, v))
    side = torch.cuda.Stream()
    dev_before = torch.cuda.current_device()
    old_limit = gpu_lib.fa2_set_wait_limit_ns(20_000_000)
    old_flags = gpu_lib.fa2_set_debug_flags(1)
    try:
        with torch.cuda.stream(side):
            gpu_lib.fa2_fwd(tq, tk, tv, scale=128 ** -0.5, stream=side)
        rc = gpu_lib.fa2_check_status(side.cuda_stream)
    finally:
        gpu_lib.fa2_set_debug_flags(old_flags)
        gpu_lib.fa2_set_wait_limit_ns(old_limit)
    assert rc == gpu_lib.FA2_ERR_TIMEOUT
    assert torch.cuda.current_device() == dev_before
    assert gpu_lib.fa2_check_status(side.cuda_stream) == gpu_lib.FA2_OK
    assert gpu_lib.fa2_check_status(0) == gpu_lib.FA2_OK
    full_check(gpu_lib, q, k, v, gen.BF16, 128 ** -0.5, "after a side-stream timeout")


# ------------------------------------------------------------------ full-size workloads

def sample_rows(B, Hq, N, n_random, seed):
    """First/last rows of the first, second and last query tiles of a few
    heads, plus seeded random rows."""
    rng = np.random.default_rng(seed)
    heads = sorted({0, B * Hq - 1, (B * Hq) // 2})
    rows = []
    for bh in heads:
        for i in (0, 127, 128, 255, N - 128, N - 1):
            if 0 <= i < N:
                rows.append(bh * N + i)
    rows.extend(rng.integers(0, B * Hq * N, n_random).tolist())
    return np.unique(np.array(rows, dtype=np.int64))


def check_rows(o, lse, q, k, v, dtype, scale, rows, what):
    torch = _torch()
    d = q.shape[-1]
    idx = torch.from_numpy(rows).to(o.device)
    o_s = o.reshape(-1, d).index_select(0, idx).float().cpu().numpy()
    l_s = lse.reshape(-1).index_select(0, idx).cpu().numpy()
    o_ref, lse_ref = oracle.attention(q, k, v, scale, dtype, rows=rows)
    assert_parity(o_s, l_s, o_ref, lse_ref, dtype, what)


def check_convex_hull(o, v, Hq):
    """Every output element lies between the min and max of its value column."""
    torch = _torch()
    G = Hq // v.shape[1]
    vt = to_dev(v, gen.BF16 if o.dtype == torch.bfloat16 else gen.FP16).float()
    lo = vt.amin(dim=2).repeat_interleave(G, dim=1)[:, :, None, :]
    hi = vt.amax(dim=2).repeat_interleave(G, dim=1)[:, :, None, :]
    of = o.float()
    slack = 1e-2 * (1 + torch.maximum(lo.abs(), hi.abs()))
    assert bool(((of >= lo - slack) & (of <= hi + slack)).all())
    assert bool(torch.isfinite(of).all())


FULL = [w for w in gen.WORKLOADS.values() if not w.fp8]   # FP8 workloads: tests/test_fp8_gpu.py


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_full_size_workloads(gpu_lib, w):
    """Every workload at full size, in the launch configuration the benchmark
    times: every element of O and LSE against the oracle."""
    q, k, v = w.inputs()
    o, lse = run_gpu(gpu_lib, q, k, v, w.dtype, w.scale)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.dtype)
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, w.dtype, w.name)
    check_convex_hull(o, v, w.Hq)


def test_many_single_tile_items_per_cta(gpu_lib):
    # 512 items of one KV tile each (two packed query tiles per item) on at
    # most 152 CTAs: every CTA runs several items back to back, so the
    # per-row statistics handed to the epilogue alternate between their two
    # slots every item. Five launches must agree bit for bit and with the
    # oracle.
    B, Hq, Hkv, N, d = 4, 256, 128, 128, 128
    q, k, v = gen.make_qkv(1401, B, Hq, Hkv, N, d, gen.BF16)
    scale = d ** -0.5
    o, lse = full_check(gpu_lib, q, k, v, gen.BF16, scale, what="512 one-tile items")
    o0, l0 = o.float().cpu().numpy(), lse.cpu().numpy()
    for _ in range(4):
        o, lse = run_gpu(gpu_lib, q, k, v, gen.BF16, scale)
        assert np.array_equal(o.float().cpu().numpy(), o0) and np.array_equal(lse.cpu().numpy(), l0)

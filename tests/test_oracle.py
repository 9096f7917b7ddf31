"""Pins for the fp64 oracle and the seeded input generator (CPU only).

Each check ties the oracle to something other than itself: values worked by
hand (tests/golden), closed forms of attention (zero queries, constant values,
one key), exact invariances (joint key/value permutation, key shift, batch and
head independence, grouped heads as repeated heads), the logsumexp identity,
and an independent library computation (torch CPU softmax in float64).
"""
import json
import math
import os

import numpy as np
import pytest

import gen
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(values):
    return gen.round_to_16bit(np.asarray(values, dtype=np.float64), gen.BF16)


def exact_bf16(values):
    bits = bf16_bits(values)
    assert np.array_equal(oracle.decode16(bits, gen.BF16), np.asarray(values, dtype=np.float64))
    return bits


def rand_inputs(seed, B, Hq, Hkv, N, d, dtype=gen.BF16, amp=1.0):
    return gen.make_qkv(seed, B, Hq, Hkv, N, d, dtype, amp)


# ---------------------------------------------------------------- generator

def test_splitmix64_published_vectors():
    # Reference outputs of SplitMix64 for seed 1234567 (Vigna's reference
    # implementation) and the first output for seed 0.
    z = gen.splitmix64(1234567, 0, 3)
    assert [int(x) for x in z] == [6457827717110365317, 3203168211198807973,
                                   9817491932198370423]
    assert int(gen.splitmix64(0, 0, 1)[0]) == 0xE220A8397B1DCDAF


def test_generator_is_deterministic_and_chunk_free():
    a = gen.normals(7, 0, 10)
    b = gen.normals(7, 4, 6)
    assert np.array_equal(a[4:], b)
    q1, k1, v1 = rand_inputs(11, 1, 2, 1, 128, 64)
    q2, k2, v2 = rand_inputs(11, 1, 2, 1, 128, 64)
    assert np.array_equal(q1, q2) and np.array_equal(k1, k2) and np.array_equal(v1, v2)
    assert q1.shape == (1, 2, 128, 64) and k1.shape == (1, 1, 128, 64)


def test_generator_moments():
    x = gen.normals(99, 0, 1 << 20)
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    # fraction within one standard deviation of a normal: erf(1/sqrt 2)
    assert abs(np.mean(np.abs(x) < 1.0) - math.erf(1 / math.sqrt(2))) < 3e-3


def test_bf16_rounding_nearest_even():
    one = 1.0
    cases = {
        one + 2.0 ** -8: 0x3F80,             # halfway, ties to even (1.0)
        one + 3 * 2.0 ** -8: 0x3F82,         # halfway, ties to even (1 + 2^-6)
        one + 2.0 ** -8 + 2.0 ** -30: 0x3F81,  # just above halfway rounds up
        -2.0: 0xC000,
        0.0: 0x0000,
        3.0e38: 0x7F62,
    }
    for x, bits in cases.items():
        assert int(bf16_bits([x])[0]) == bits, (x, hex(int(bf16_bits([x])[0])))


def test_fp16_rounding_nearest_even():
    got = gen.round_to_16bit(np.array([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 65504.0, 2.0 ** -24]),
                             gen.FP16)
    assert [int(b) for b in got] == [0x3C00, 0x3C02, 0x7BFF, 0x0001]


# ---------------------------------------------------------------- decoding

def test_decode_fixed_patterns():
    bf = oracle.decode16(np.array([0x3F80, 0xC000, 0x0001, 0x7F80, 0x4049], np.uint16), gen.BF16)
    assert bf[0] == 1.0 and bf[1] == -2.0 and bf[2] == 2.0 ** -133 and math.isinf(bf[3])
    assert bf[4] == 3.140625
    hf = oracle.decode16(np.array([0x3C00, 0x0001, 0x7BFF, 0xFC00, 0x3555], np.uint16), gen.FP16)
    assert hf[0] == 1.0 and hf[1] == 2.0 ** -24 and hf[2] == 65504.0 and hf[3] == -math.inf
    assert hf[4] == 0.333251953125


def test_decode_fp16_all_patterns_match_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode16(bits, gen.FP16)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


# ---------------------------------------------------------------- hand-worked cases

def test_hand_case_n2_d1():
    g = json.load(open(os.path.join(GOLDEN, "hand_n2_d1.json")))
    q = exact_bf16(g["q"]).reshape(1, 1, 1, 1)
    q = np.repeat(q, 2, axis=2)  # N = 2 query rows, both q = 1
    k = exact_bf16(g["k"]).reshape(1, 1, 2, 1)
    v = exact_bf16(g["v"]).reshape(1, 1, 2, 1)
    o, lse = oracle.attention(q, k, v, math.log(3) / 2, gen.BF16)
    assert abs(o[0, 0, 0, 0] - g["o"][0]) < 1e-13
    assert abs(lse[0, 0, 0] - math.log(4)) < 1e-13


def test_hand_case_n3_d2():
    g = json.load(open(os.path.join(GOLDEN, "hand_n3_d2.json")))
    q = exact_bf16(g["q"]).reshape(1, 1, 3, 2)
    k = exact_bf16(g["k"]).reshape(1, 1, 3, 2)
    v = exact_bf16(g["v"]).reshape(1, 1, 3, 2)
    o, lse = oracle.attention(q, k, v, math.log(2), gen.BF16)
    np.testing.assert_allclose(o[0, 0, :2], np.array(g["o_rows_0_1"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0, :2], [math.log(7), math.log(4.5)], rtol=0, atol=1e-13)
    np.testing.assert_allclose(o[0, 0, 2], [7 / 3, -7 / 3], rtol=0, atol=1e-13)
    assert abs(lse[0, 0, 2] - math.log(3)) < 1e-13


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dtype", [gen.BF16, gen.FP16])
def test_zero_queries_give_column_mean(dtype):
    _, k, v = rand_inputs(3, 2, 2, 2, 96, 32, dtype)
    q = np.zeros((2, 2, 96, 32), np.uint16)
    o, lse = oracle.attention(q, k, v, 1 / math.sqrt(32), dtype)
    vd = oracle.decode16(v, dtype)
    np.testing.assert_allclose(o, np.broadcast_to(vd.mean(axis=2, keepdims=True), o.shape),
                               rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(96), rtol=0, atol=1e-13)


def test_constant_values_give_constant_output():
    q, k, _ = rand_inputs(5, 1, 3, 3, 80, 16, amp=3.0)
    v = np.full(k.shape, 0x3F80, np.uint16)  # bf16 1.0
    o, _ = oracle.attention(q, k, v, 0.25, gen.BF16)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-12)


def test_single_key():
    q, k, v = rand_inputs(6, 2, 2, 2, 1, 8)
    o, lse = oracle.attention(q, k, v, 0.3, gen.BF16)
    qd, kd, vd = (oracle.decode16(x, gen.BF16) for x in (q, k, v))
    np.testing.assert_array_equal(o, vd)
    np.testing.assert_allclose(lse[..., 0], 0.3 * np.sum(qd[:, :, 0] * kd[:, :, 0], -1),
                               rtol=0, atol=1e-12)


def test_rows_of_p_sum_to_one():
    q, k, _ = rand_inputs(8, 1, 2, 1, 200, 64, amp=3.0)
    for row in (0, 57, 399):
        p = oracle.softmax_row(q, k, 0.125, gen.BF16, row)
        assert abs(p.sum() - 1.0) <= 1e-12
        assert np.all(p > 0)


def test_dominant_key():
    rng = np.random.default_rng(0)
    N, d = 64, 16
    q = exact_bf16(np.ones(d))
    k = bf16_bits(rng.integers(-1, 2, size=(N, d)).astype(np.float64))
    k[17] = bf16_bits(np.full(d, 8.0))   # score gap at least 8*16*0.5 - 16*0.5 = 56
    v = bf16_bits(rng.standard_normal((N, d)))
    o, _ = oracle.attention(q.reshape(1, 1, 1, d).repeat(N, 2), k.reshape(1, 1, N, d),
                            v.reshape(1, 1, N, d), 0.5, gen.BF16)
    vd = oracle.decode16(v, gen.BF16)
    np.testing.assert_allclose(o[0, 0, 0], vd[17], rtol=0, atol=1e-20 + N * math.exp(-50) * 5)


# ---------------------------------------------------------------- invariances

def test_joint_permutation_of_keys_and_values():
    q, k, v = rand_inputs(9, 1, 2, 2, 160, 32)
    perm = np.random.default_rng(1).permutation(160)
    o1, l1 = oracle.attention(q, k, v, 0.2, gen.BF16)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.2, gen.BF16)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)
    # permuting keys without the values must change the output
    o3, _ = oracle.attention(q, k[:, :, perm], v, 0.2, gen.BF16)
    assert np.max(np.abs(o3 - o1)) > 1e-3


def test_key_shift_invariance():
    rng = np.random.default_rng(2)
    N, d = 48, 8
    qv = rng.integers(-3, 4, size=(1, 1, N, d)).astype(np.float64)
    kv = rng.integers(-3, 4, size=(1, 1, N, d)).astype(np.float64)
    c = rng.integers(-2, 3, size=d).astype(np.float64)
    q, k = exact_bf16(qv), exact_bf16(kv)
    k2 = exact_bf16(kv + c)
    v = bf16_bits(rng.standard_normal((1, 1, N, d)))
    o1, l1 = oracle.attention(q, k, v, 0.15, gen.BF16)
    o2, l2 = oracle.attention(q, k2, v, 0.15, gen.BF16)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 0.15 * (qv @ c), rtol=0, atol=1e-12)


def test_batch_and_head_independence():
    q, k, v = rand_inputs(10, 2, 3, 3, 64, 16)
    o, lse = oracle.attention(q, k, v, 0.25, gen.BF16)
    for b in range(2):
        for h in range(3):
            o1, l1 = oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                      v[b:b + 1, h:h + 1], 0.25, gen.BF16)
            np.testing.assert_array_equal(o1[0, 0], o[b, h])
            np.testing.assert_array_equal(l1[0, 0], lse[b, h])


def test_grouped_heads_equal_repeated_heads():
    q, k, v = rand_inputs(12, 2, 8, 2, 64, 16)
    o, lse = oracle.attention(q, k, v, 0.25, gen.BF16)
    kr, vr = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
    o2, l2 = oracle.attention(q, kr, vr, 0.25, gen.BF16)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, l2)
    # a wrong head mapping (h % Hkv) must give a different result
    wrong_k = np.tile(k, (1, 4, 1, 1))
    wrong_v = np.tile(v, (1, 4, 1, 1))
    o3, _ = oracle.attention(q, wrong_k, wrong_v, 0.25, gen.BF16)
    assert np.max(np.abs(o3 - o)) > 1e-3


def test_row_subset_matches_full():
    q, k, v = rand_inputs(13, 2, 2, 1, 96, 32)
    o, lse = oracle.attention(q, k, v, 0.2, gen.BF16)
    rows = np.array([0, 5, 95, 96, 250, 383])
    os_, ls_ = oracle.attention(q, k, v, 0.2, gen.BF16, rows=rows)
    np.testing.assert_array_equal(os_, o.reshape(-1, 32)[rows])
    np.testing.assert_array_equal(ls_, lse.reshape(-1)[rows])


# ---------------------------------------------------------------- identities and library

@pytest.mark.parametrize("dtype,amp", [(gen.BF16, 1.0), (gen.FP16, 1.0), (gen.BF16, 3.0)])
def test_lse_identity_and_library_crosscheck(dtype, amp):
    torch = pytest.importorskip("torch")
    q, k, v = rand_inputs(14, 1, 2, 1, 192, 64, dtype, amp)
    scale = 1 / 8
    o, lse = oracle.attention(q, k, v, scale, dtype)
    qd, kd, vd = (torch.from_numpy(oracle.decode16(x, dtype)) for x in (q, k, v))
    kd = kd.repeat_interleave(2, dim=1)
    vd = vd.repeat_interleave(2, dim=1)
    s = scale * torch.einsum("bhid,bhjd->bhij", qd, kd)
    ref_o = torch.softmax(s, dim=-1) @ vd
    ref_lse = torch.logsumexp(s, dim=-1)
    np.testing.assert_allclose(o, ref_o.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)
    # O = sum_j exp(s_j - LSE) v_j
    o_from_lse = torch.exp(s - torch.from_numpy(lse)[..., None]) @ vd
    np.testing.assert_allclose(o, o_from_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_oracle_rejects_bad_sizes():
    q, k, v = rand_inputs(15, 1, 3, 2, 16, 8)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, 0.1, gen.BF16)  # 3 query heads over 2 KV heads


# ---------------------------------------------------------------- generalised form: ragged, unequal, causal

def kend(i, nq, nk, causal):
    return min(nk, i + 1 + nk - nq) if causal else nk


def test_hand_causal_case():
    g = json.load(open(os.path.join(GOLDEN, "hand_causal_n2_d1.json")))
    q = exact_bf16(g["q"]).reshape(1, 1, 2, 1)
    k = exact_bf16(g["k"]).reshape(1, 1, 2, 1)
    v = exact_bf16(g["v"]).reshape(1, 1, 2, 1)
    o, lse = oracle.attention_ex(q, k, v, math.log(3) / 2, gen.BF16, causal=True)
    np.testing.assert_allclose(o[0, 0, :, 0], g["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], [0.0, math.log(4)], rtol=0, atol=1e-13)


@pytest.mark.parametrize("nq,nk", [(5, 5), (7, 12), (12, 7), (130, 130), (1, 9)])
def test_causal_zero_queries_give_prefix_means(nq, nk):
    _, k, v = rand_inputs(40, 1, 2, 1, nk, 8)
    q = np.zeros((1, 2, nq, 8), np.uint16)
    o, lse = oracle.attention_ex(q, k, v, 0.3, gen.BF16, causal=True)
    vd = oracle.decode16(v, gen.BF16)[0, 0]
    for i in range(nq):
        e = kend(i, nq, nk, True)
        if e <= 0:
            assert np.all(o[0, :, i] == 0.0) and np.all(np.isneginf(lse[0, :, i]))
        else:
            np.testing.assert_allclose(o[0, 0, i], vd[:e].mean(axis=0), rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[0, :, i], math.log(e), rtol=0, atol=1e-13)


@pytest.mark.parametrize("nq,nk", [(3, 10), (10, 3), (77, 200)])
def test_unequal_lengths_zero_queries_give_mean(nq, nk):
    _, k, v = rand_inputs(41, 2, 2, 2, nk, 16)
    q = np.zeros((2, 2, nq, 16), np.uint16)
    o, lse = oracle.attention_ex(q, k, v, 0.3, gen.BF16, causal=False)
    vd = oracle.decode16(v, gen.BF16)
    np.testing.assert_allclose(o, np.broadcast_to(vd.mean(axis=2, keepdims=True), o.shape), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(nk), rtol=0, atol=1e-13)


def test_causal_first_row_is_first_value():
    q, k, v = rand_inputs(42, 2, 3, 3, 40, 8)
    o, lse = oracle.attention_ex(q, k, v, 0.2, gen.BF16, causal=True)
    qd, kd, vd = (oracle.decode16(x, gen.BF16) for x in (q, k, v))
    np.testing.assert_array_equal(o[:, :, 0], vd[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], 0.2 * np.sum(qd[:, :, 0] * kd[:, :, 0], -1), rtol=0, atol=1e-12)


def test_causal_ignores_keys_past_the_mask():
    q, k, v = rand_inputs(43, 1, 2, 2, 64, 16)
    o1, l1 = oracle.attention_ex(q, k, v, 0.25, gen.BF16, causal=True)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 40:] = bf16_bits(np.full((1, 2, 24, 16), 3.0))
    v2[:, :, 40:] = bf16_bits(np.full((1, 2, 24, 16), -7.0))
    o2, l2 = oracle.attention_ex(q, k2, v2, 0.25, gen.BF16, causal=True)
    np.testing.assert_array_equal(o1[:, :, :40], o2[:, :, :40])
    np.testing.assert_array_equal(l1[:, :, :40], l2[:, :, :40])
    assert np.max(np.abs(o1[:, :, 40:] - o2[:, :, 40:])) > 1e-3


def test_non_causal_equal_lengths_reduces_to_attention():
    q, k, v = rand_inputs(44, 1, 4, 2, 96, 32)
    o1, l1 = oracle.attention(q, k, v, 0.2, gen.BF16)
    o2, l2 = oracle.attention_ex(q, k, v, 0.2, gen.BF16, causal=False)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("nq,nk,causal", [(70, 70, True), (50, 90, True), (90, 50, True), (33, 100, False)])
def test_generalised_library_crosscheck(nq, nk, causal):
    torch = pytest.importorskip("torch")
    q, _, _ = rand_inputs(45, 1, 4, 2, nq, 32)
    _, k, v = rand_inputs(46, 1, 4, 2, nk, 32)
    o, lse = oracle.attention_ex(q, k, v, 0.15, gen.BF16, causal=causal)
    qd, kd, vd = (torch.from_numpy(oracle.decode16(x, gen.BF16)) for x in (q, k, v))
    kd, vd = kd.repeat_interleave(2, dim=1), vd.repeat_interleave(2, dim=1)
    s = 0.15 * torch.einsum("bhid,bhjd->bhij", qd, kd)
    if causal:
        i = torch.arange(nq)[:, None]
        j = torch.arange(nk)[None, :]
        s = s.masked_fill(j > i + (nk - nq), float("-inf"))
    ref_lse = torch.logsumexp(s, dim=-1)
    ref_o = torch.nan_to_num(torch.softmax(s, dim=-1)) @ vd
    np.testing.assert_allclose(o, ref_o.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- backward

def bwd_inputs(seed, B, Hq, Hkv, N, d, dtype=gen.BF16):
    q, k, v = rand_inputs(seed, B, Hq, Hkv, N, d, dtype)
    do, _, _ = rand_inputs(seed + 1, B, Hq, Hkv, N, d, dtype)
    return q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    B, Hq, Hkv, N, d, scale = 1, 2, 1, 12, 8, 0.35
    q, k, v, do = bwd_inputs(50, B, Hq, Hkv, N, d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, gen.BF16, causal=causal)
    qd, kd, vd, dod = (oracle.decode16(x, gen.BF16) for x in (q, k, v, do))

    def loss(qq, kk, vv):
        return float(np.sum(dod * oracle.attention_f64(qq, kk, vv, scale, causal)))

    rng = np.random.default_rng(1)
    eps = 1e-6
    for name, x, g in (("q", qd, dq), ("k", kd, dk), ("v", vd, dv)):
        for _ in range(6):
            idx = tuple(rng.integers(0, s) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, kd, vd), "k": (qd, xp, vd), "v": (qd, kd, xp)}[name]
            args_m = {"q": (xm, kd, vd), "k": (qd, xm, vd), "v": (qd, kd, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-6 * (1 + abs(fd)), (name, idx, fd, g[idx])


@pytest.mark.parametrize("causal,Hq,Hkv", [(False, 2, 2), (True, 4, 2), (True, 2, 1)])
def test_backward_library_crosscheck(causal, Hq, Hkv):
    torch = pytest.importorskip("torch")
    B, N, d, scale = 2, 40, 16, 0.25
    q, k, v, do = bwd_inputs(51, B, Hq, Hkv, N, d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, gen.BF16, causal=causal)
    qt, kt, vt = (torch.from_numpy(oracle.decode16(x, gen.BF16)).requires_grad_() for x in (q, k, v))
    dot = torch.from_numpy(oracle.decode16(do, gen.BF16))
    G = Hq // Hkv
    s = scale * torch.einsum("bhid,bhjd->bhij", qt, kt.repeat_interleave(G, 1))
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, -1) @ vt.repeat_interleave(G, 1)
    o.backward(dot)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_closed_forms():
    B, Hq, Hkv, N, d = 1, 2, 2, 30, 8
    q, k, _, do = bwd_inputs(52, B, Hq, Hkv, N, d)
    # constant values: O = v for every row, dP_ij = dO_i . v = D_i, so dS = 0
    v = np.full((B, Hkv, N, d), 0x3FC0, np.uint16)  # bf16 1.5
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.3, gen.BF16)
    assert np.max(np.abs(dq)) < 1e-12 and np.max(np.abs(dk)) < 1e-12
    # each row of dS sums to zero, so sum_j dK_j = scale * sum_i q_i * 0 = 0
    _, _, v2 = rand_inputs(53, B, Hq, Hkv, N, d)
    for causal in (False, True):
        _, dk2, dv2 = oracle.attention_bwd(q, k, v2, do, 0.3, gen.BF16, causal=causal)
        np.testing.assert_allclose(dk2.sum(axis=2), 0.0, atol=1e-12)
        # sum_j dV_j = sum_i dO_i (rows of P sum to one)
        np.testing.assert_allclose(dv2.sum(axis=2), oracle.decode16(do, gen.BF16).sum(axis=2), atol=1e-11)
    # zero upstream gradient: zero gradients
    dq0, dk0, dv0 = oracle.attention_bwd(q, k, v2, np.zeros_like(do), 0.3, gen.BF16)
    assert not dq0.any() and not dk0.any() and not dv0.any()


@pytest.mark.parametrize("causal,Hq,Hkv", [(False, 2, 2), (True, 4, 2)])
def test_backward_bound_sums_follow_their_definitions(causal, Hq, Hkv):
    """The absolute sums the GPU backward's elementwise bound is built from,
    recomputed here with dense float64 numpy arrays from their definitions
    (P, dS, O, a, E and F as matrices; grouped heads by repetition)."""
    B, N, d, scale = 2, 33, 8, 0.3
    q, k, v, do = bwd_inputs(54, B, Hq, Hkv, N, d)
    dq, dk, dv, bnd = oracle.attention_bwd(q, k, v, do, scale, gen.BF16, causal=causal, bounds=True)
    G = Hq // Hkv
    Q, dO = (oracle.decode16(x, gen.BF16) for x in (q, do))
    K, V = (np.repeat(oracle.decode16(x, gen.BF16), G, axis=1) for x in (k, v))
    s = scale * np.einsum("bhid,bhjd->bhij", Q, K)
    if causal:
        s = np.where(np.triu(np.ones((N, N), bool), 1), -np.inf, s)
    P = np.exp(s - s.max(-1, keepdims=True))
    P /= P.sum(-1, keepdims=True)
    O = P @ V
    a = P @ np.abs(V)
    E = np.sum(np.abs(dO) * (np.abs(O) + a), -1)                       # [b,h,i]
    F = np.einsum("bhid,bhjd->bhij", np.abs(dO), np.abs(V))           # [b,h,i,j]
    dS = P * (dO @ np.swapaxes(V, -1, -2) - np.sum(dO * O, -1)[..., None])
    np.testing.assert_allclose(dq, scale * dS @ K, rtol=1e-10, atol=1e-12)
    want_q = [scale * np.abs(dS) @ np.abs(K), scale * E[..., None] * (P @ np.abs(K)),
              scale * (P * F) @ np.abs(K)]
    kv = lambda x: x.reshape(B, Hkv, G, N, d).sum(axis=2)              # sum over a KV head's query heads
    tr = lambda x: np.swapaxes(x, -1, -2)
    want_k = [kv(scale * tr(np.abs(dS)) @ np.abs(Q)), kv(scale * tr(P * E[..., None]) @ np.abs(Q)),
              kv(scale * tr(P * F) @ np.abs(Q))]
    for got, want in zip(bnd["q"], want_q):
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-13)
    for got, want in zip(bnd["k"], want_k):
        np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(bnd["v"], kv(tr(P) @ np.abs(dO)), rtol=1e-10, atol=1e-13)
    # the bound sums dominate the gradients they bound
    assert np.all(np.abs(dq) <= bnd["q"][0] * (1 + 1e-12) + 1e-15)
    assert np.all(np.abs(dk) <= bnd["k"][0] * (1 + 1e-12) + 1e-15)
    assert np.all(np.abs(dv) <= bnd["v"] * (1 + 1e-12) + 1e-15)


# ---------------------------------------------------------------- FP8 (e4m3) inputs

def _torch_e4m3():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    return torch


def test_e4m3_decode_matches_torch_on_every_code():
    torch = _torch_e4m3()
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2   # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_rounding_matches_torch_and_the_generator():
    torch = _torch_e4m3()
    rng = np.random.default_rng(5)
    vals = oracle.decode_e4m3(np.arange(127, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2                    # exact ties: go to the even code
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.uniform(-2.0 ** -5, 2.0 ** -5, 20000),
                        mids, -mids, vals, rng.normal(0, 3, 5000)])
    ours = oracle.round_e4m3(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
    assert np.array_equal(ours, oracle.decode_e4m3(gen.e4m3_encode(x)))
    # ties to even: 17 lies between 16 (code 0x58) and 18 (0x59)
    assert oracle.round_e4m3(np.array([17.0, 2.0 ** -10, 1.5 * 2.0 ** -9]))[0] == 16.0
    # saturation above the largest finite value (the GPU conversion is .satfinite)
    assert oracle.round_e4m3(np.array([460.0, 1e6]))[1] == 448.0


def test_fp8_hand_case():
    with open(os.path.join(GOLDEN, "hand_fp8_n2_d1.json")) as fh:
        g = json.load(fh)
    scale = math.log(3.0) / 2.0
    for case in g["cases"]:
        q = np.array(case["q_codes"], dtype=np.uint8).reshape(1, 1, 1, 1)
        k = np.array(case["k_codes"], dtype=np.uint8).reshape(1, 1, 2, 1)
        v = np.array(case["v_codes"], dtype=np.uint8).reshape(1, 1, 2, 1)
        # query row 0 only has N = 2 keys: make a 2-row problem with the same query twice
        q2 = np.concatenate([q, q], axis=2)
        qd, kd, vd = ([x] for x in case["descales"])
        o, lse, a, b = oracle.attention_fp8(q2, k, v, qd, kd, vd, scale, round_p=True, bc=g["bc_for_o_method"])
        assert o[0, 0, 0, 0] == pytest.approx(g["o_method"], abs=1e-14)
        o1, _, _, _ = oracle.attention_fp8(q2, k, v, qd, kd, vd, scale, round_p=True, bc=1)
        assert o1[0, 0, 0, 0] == pytest.approx(g["o_method_bc1"], abs=1e-14)
        assert lse[0, 0, 0] == pytest.approx(math.log(4.0), abs=1e-14)
        assert a[0, 0, 0, 0] == pytest.approx(g["a"], abs=1e-14)
        assert b[0, 0, 0, 0] == pytest.approx(g["b"], abs=1e-14)
        o, lse, _, _ = oracle.attention_fp8(q2, k, v, qd, kd, vd, scale, round_p=False)
        assert o[0, 0, 0, 0] == pytest.approx(g["o_plain"], abs=1e-14)


def _fp8_inputs(seed, B=1, Hq=2, Hkv=1, N=64, d=32, amp=1.0):
    return gen.make_qkv_fp8(seed, B, Hq, Hkv, N, d, amp)


def _dequant(codes, descale, heads_per_group):
    B, H = codes.shape[:2]
    x = oracle.decode_e4m3(codes)
    ds = np.asarray(descale, dtype=np.float64).reshape(B, -1)
    return x * np.repeat(ds, heads_per_group, axis=1)[:, :, None, None]


def test_fp8_plain_mode_is_attention_on_dequantised_inputs():
    torch = pytest.importorskip("torch")
    B, Hq, Hkv, N, d = 2, 4, 2, 96, 32
    q, k, v, qd, kd, vd = _fp8_inputs(21, B, Hq, Hkv, N, d)
    scale = 0.3
    o, lse, _, _ = oracle.attention_fp8(q, k, v, qd, kd, vd, scale, round_p=False)
    G = Hq // Hkv
    qx, kx, vx = _dequant(q, qd, G), _dequant(k, kd, 1), _dequant(v, vd, 1)
    ref = oracle.attention_f64(qx, kx, vx, scale)
    assert np.max(np.abs(o - ref)) < 1e-12
    # and an independent library computation of the same thing
    kr = torch.from_numpy(np.repeat(kx, G, axis=1))
    vr = torch.from_numpy(np.repeat(vx, G, axis=1))
    s = torch.from_numpy(qx) @ kr.transpose(-1, -2) * scale
    lib = (torch.softmax(s, -1) @ vr).numpy()
    assert np.max(np.abs(o - lib)) < 1e-12
    assert np.max(np.abs(lse - torch.logsumexp(s, -1).numpy())) < 1e-12


def test_fp8_method_equals_plain_when_weights_are_e4m3_exact():
    # scores (0, -ln 2, -2 ln 2, -3 ln 2) give 256 p = 256, 128, 64, 32: exact in e4m3
    scale = math.log(2.0)
    q = np.full((1, 1, 4, 1), 0x38, dtype=np.uint8)            # q = 1
    kvals = np.array([0.0, -1.0, -2.0, -3.0])
    k = gen.e4m3_encode(kvals).reshape(1, 1, 4, 1)
    assert np.array_equal(oracle.decode_e4m3(k).ravel(), kvals)
    v = gen.e4m3_encode(np.array([1.0, -2.0, 3.0, 0.5])).reshape(1, 1, 4, 1)
    one = [1.0]
    om, lm, _, _ = oracle.attention_fp8(q, k, v, one, one, one, scale, round_p=True)
    op, lp, _, _ = oracle.attention_fp8(q, k, v, one, one, one, scale, round_p=False)
    assert np.array_equal(om, op) and np.array_equal(lm, lp)
    assert om[0, 0, 0, 0] == pytest.approx((1 - 1.0 + 0.75 + 0.0625) / 1.875, abs=1e-15)


def test_fp8_rounding_error_within_its_bound():
    # |o_method - o_plain| <= 2^-4 a + 2^-18 b elementwise (relative rounding
    # error 2^-4 of e4m3 normals, absolute 2^-10 / 2^8 below 2^-6 * 2^8)
    q, k, v, qd, kd, vd = _fp8_inputs(22, 1, 2, 1, 512, 64, amp=2.0)
    om, lm, a, b = oracle.attention_fp8(q, k, v, qd, kd, vd, 0.125, round_p=True)
    op, lp, _, _ = oracle.attention_fp8(q, k, v, qd, kd, vd, 0.125, round_p=False)
    err = np.abs(om - op)
    assert np.all(err <= 2.0 ** -4 * a + 2.0 ** -18 * b + 1e-15)
    assert err.max() > 0                     # rounding does change the result
    assert np.array_equal(lm, lp)            # l uses the unrounded weights
    # V = constant c: the plain output is c, the method's stays within 2^-4 c
    vc = np.full_like(v, 0x40)                # 2.0
    om, _, _, _ = oracle.attention_fp8(q, k, vc, qd, kd, [1.0], 0.125, round_p=True)
    op, _, _, _ = oracle.attention_fp8(q, k, vc, qd, kd, [1.0], 0.125, round_p=False)
    assert np.max(np.abs(op - 2.0)) < 1e-12
    assert np.max(np.abs(om - 2.0)) <= 2.0 ** -4 * 2.0


def test_fp8_grouped_heads_equal_repeated_heads():
    B, Hq, Hkv, N, d = 2, 4, 2, 64, 32
    q, k, v, qd, kd, vd = _fp8_inputs(23, B, Hq, Hkv, N, d)
    G = Hq // Hkv
    og, lg, _, _ = oracle.attention_fp8(q, k, v, qd, kd, vd, 0.2)
    # MHA on repeated K/V: each query head becomes its own group with the
    # descales of its KV head
    rep = lambda x: np.repeat(x, G, axis=1)
    repd = lambda s: np.repeat(np.asarray(s).reshape(B, Hkv), G, axis=1).ravel()
    om, lm, _, _ = oracle.attention_fp8(q, rep(k), rep(v), repd(qd), repd(kd), repd(vd), 0.2)
    assert np.array_equal(og, om) and np.array_equal(lg, lm)


def test_fp8_generator_quantisation():
    B, Hq, Hkv, N, d = 2, 4, 2, 64, 32
    q, k, v, qd, kd, vd = gen.make_qkv_fp8(31, B, Hq, Hkv, N, d)
    assert q.dtype == np.uint8 and qd.dtype == np.float32 and qd.shape == (B * Hkv,)
    x = gen.normals(31, 0, q.size).reshape(q.shape)
    G = Hq // Hkv
    for t, ds, heads in ((q, qd, G), (k, kd, 1), (v, vd, 1)):
        deq = _dequant(t, ds, heads)
        groups = np.abs(t.reshape(B * Hkv, -1) & 0x7F).max(axis=1)
        assert np.all(groups == 0x7E)                      # every group reaches 448
    deq = _dequant(q, qd, G)
    rel = np.abs(deq - x) / np.maximum(np.abs(x), 2.0 ** -6 * np.repeat(qd.reshape(B, Hkv), G, 1)[:, :, None, None])
    assert rel.max() <= 2.0 ** -4 + 1e-6


def test_fp8_tiling_changes_nothing_when_the_max_comes_first():
    # Online softmax over key tiles: if every row's largest score sits in the
    # first tile, the running max is final from the first tile on, so each
    # weight is rounded exactly as without tiling (bc >= N).
    N, d = 300, 16
    q, k, v, qd, kd, vd = gen.make_qkv_fp8(41, 1, 1, 1, N, d)
    q = q[:, :, :1].copy()
    k = k.copy()
    k[0, 0, 0] = q[0, 0, 0]                 # key 0 parallel to the query
    one = [1.0]
    qx = oracle.decode_e4m3(q).reshape(d)
    kx = oracle.decode_e4m3(k).reshape(N, d)
    assert np.argmax(kx @ qx) == 0          # the premise: key 0 has the top score
    qq = np.concatenate([q] * N, axis=2)    # N query rows so that q is [1, 1, N, d]
    o_all, _, _, _ = oracle.attention_fp8(qq, k, v, one, one, one, 0.7, bc=N)
    for bc in (1, 7, 128, 299, 1000):
        o_bc, _, _, _ = oracle.attention_fp8(qq, k, v, one, one, one, 0.7, bc=bc)
        assert np.array_equal(o_bc[0, 0, 0], o_all[0, 0, 0])


def test_fp8_tiled_method_stays_within_the_rounding_bound():
    q, k, v, qd, kd, vd = _fp8_inputs(42, 1, 2, 1, 700, 32, amp=2.0)
    for bc in (1, 64, 128, 700):
        om, op, lp, a, b = oracle.attention_fp8_both(q, k, v, qd, kd, vd, 0.2, bc=bc)
        assert np.all(np.abs(om - op) <= 2.0 ** -4 * a + 2.0 ** -18 * b + 1e-15)


def _fp8_general_inputs(seed, B, Hq, Hkv, nq, nk, d, amp=1.0):
    q, _, _, qd, _, _ = gen.make_qkv_fp8(seed, B, Hq, Hkv, nq, d, amp)
    _, k, v, _, kd, vd = gen.make_qkv_fp8(seed + 1, B, Hq, Hkv, nk, d, amp)
    return q, k, v, qd, kd, vd


@pytest.mark.parametrize("nq,nk,causal", [(70, 70, True), (50, 90, True), (90, 50, True), (33, 100, False),
                                          (100, 33, False)])
def test_fp8_general_plain_mode_library_crosscheck(nq, nk, causal):
    # Plain mode with unequal lengths and the bottom-right causal mask is
    # masked softmax attention on the dequantised inputs; rows that see no key
    # (causal, nq > nk) give o = 0 and lse = -inf.
    torch = pytest.importorskip("torch")
    B, Hq, Hkv, d = 2, 4, 2, 32
    q, k, v, qd, kd, vd = _fp8_general_inputs(51, B, Hq, Hkv, nq, nk, d)
    o, lse, _, _ = oracle.attention_fp8(q, k, v, qd, kd, vd, 0.25, round_p=False, causal=causal)
    G = Hq // Hkv
    qx = torch.from_numpy(_dequant(q, qd, G))
    kx = torch.from_numpy(np.repeat(_dequant(k, kd, 1), G, axis=1))
    vx = torch.from_numpy(np.repeat(_dequant(v, vd, 1), G, axis=1))
    s = 0.25 * qx @ kx.transpose(-1, -2)
    if causal:
        i = torch.arange(nq)[:, None]
        j = torch.arange(nk)[None, :]
        s = s.masked_fill(j > i + (nk - nq), float("-inf"))
    ref_o = torch.nan_to_num(torch.softmax(s, dim=-1)) @ vx
    np.testing.assert_allclose(o, ref_o.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)
    if causal and nq > nk:
        assert np.all(np.isneginf(lse[:, :, : nq - nk])) and np.all(o[:, :, : nq - nk] == 0)
        assert np.all(np.isfinite(lse[:, :, nq - nk:]))


def test_fp8_causal_first_row_is_its_first_value():
    # Equal lengths, causal: row 0 sees key 0 alone, so p = 1, 2^8 p = 256 is
    # exact in e4m3 and both modes return v_0 dequantised, exactly.
    q, k, v, qd, kd, vd = _fp8_inputs(52, 1, 2, 1, 64, 32)
    for round_p in (True, False):
        o, lse, _, _ = oracle.attention_fp8(q, k, v, qd, kd, vd, 0.3, round_p=round_p, causal=True)
        v0 = oracle.decode_e4m3(v[0, 0, 0]) * np.float64(vd[0])
        for h in range(2):
            assert np.array_equal(o[0, h, 0], v0)
            s0 = 0.3 * np.dot(oracle.decode_e4m3(q[0, h, 0]) * np.float64(qd[0]),
                              oracle.decode_e4m3(k[0, 0, 0]) * np.float64(kd[0]))
            assert lse[0, h, 0] == pytest.approx(s0, abs=1e-12)


@pytest.mark.parametrize("nq,nk", [(40, 40), (30, 75), (75, 30)])
def test_fp8_causal_method_equals_the_method_on_the_visible_keys(nq, nk):
    # The mask only removes keys: with key tiles starting at key 0, causal row
    # i is the non-causal method on keys [0, kend(i)) -- for every tile width,
    # so the rounding against the running max is the same too.
    q, k, v, qd, kd, vd = _fp8_general_inputs(53, 1, 1, 1, nq, nk, 16, amp=2.0)
    for bc in (1, 8, 128):
        o, lse, a, b = oracle.attention_fp8(q, k, v, qd, kd, vd, 0.4, causal=True, bc=bc)
        for i in range(nq):
            kend = min(nk, i + 1 + nk - nq)
            if kend <= 0:
                assert np.isneginf(lse[0, 0, i]) and not o[0, 0, i].any()
                continue
            oi, li, ai, bi = oracle.attention_fp8(q[:, :, i:i + 1], k[:, :, :kend], v[:, :, :kend], qd, kd, vd,
                                                  0.4, bc=bc)
            assert np.array_equal(o[0, 0, i], oi[0, 0, 0]) and lse[0, 0, i] == li[0, 0, 0]
            assert np.array_equal(a[0, 0, i], ai[0, 0, 0]) and np.array_equal(b[0, 0, i], bi[0, 0, 0])


def test_fp8_general_method_stays_within_the_rounding_bound():
    q, k, v, qd, kd, vd = _fp8_general_inputs(54, 1, 2, 1, 300, 500, 32, amp=2.0)
    for causal in (False, True):
        om, op, lp, a, b = oracle.attention_fp8_both(q, k, v, qd, kd, vd, 0.2, causal=causal)
        assert np.all(np.abs(om - op) <= 2.0 ** -4 * a + 2.0 ** -18 * b + 1e-15)


def test_results_do_not_depend_on_the_thread_count():
    # Query rows are independent, so the OpenMP thread count must not change
    # a single bit of the forward oracles' results.
    q, k, v = rand_inputs(61, 1, 4, 2, 192, 32)
    o1, l1 = oracle.attention(q, k, v, 0.2, gen.BF16, threads=1)
    o4, l4 = oracle.attention(q, k, v, 0.2, gen.BF16, threads=4)
    assert np.array_equal(o1, o4) and np.array_equal(l1, l4)
    e1 = oracle.attention_ex(q[:, :, :150], k, v, 0.2, gen.BF16, causal=True, threads=1)
    e4 = oracle.attention_ex(q[:, :, :150], k, v, 0.2, gen.BF16, causal=True, threads=3)
    assert all(np.array_equal(a, b) for a, b in zip(e1, e4))
    q8, k8, v8, qd, kd, vd = gen.make_qkv_fp8(62, 1, 2, 1, 200, 32)
    f1 = oracle.attention_fp8_both(q8, k8, v8, qd, kd, vd, 0.3, threads=1, causal=True)
    f4 = oracle.attention_fp8_both(q8, k8, v8, qd, kd, vd, 0.3, threads=4, causal=True)
    assert all(np.array_equal(a, b) for a, b in zip(f1, f4))

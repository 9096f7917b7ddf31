"""The FMA-pipe exp2 used for one softmax pair in eight (CPU).

The kernel header evaluates exp2(x), x <= 0, by Cody-Waite range reduction
(x = n + f, n nearest integer via the 1.5 * 2^23 rounding constant, |f| <= 1/2),
a degree-3 polynomial with constant term 1 for 2^f, and an integer add of n into
the exponent field. This test reads the polynomial coefficients out of the
header, replays the same float32 operation sequence with numpy, and checks it
against 2^x in float64: relative error <= 1.1e-4 over [-125, 0], exactly 1 at
x = 0, exact powers of two at the integers, and the clamp below -125.
"""
import os
import re

import numpy as np

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "attention_fa2_forward_03_gb300", "csrc", "ptx_sm103.cuh")
f32 = np.float32


def header_coefficients():
    src = open(HEADER).read()
    body = src[src.index("uint64_t ex2_poly_f2("):]
    body = body[:body.index("return f2_pack(")]
    clamp = [float(c) for c in re.findall(r"fmaxf\(x0, ([-0-9.e]+)f\)", body)]
    consts = [float(c) for c in re.findall(r"f2_pack\(([-0-9.e]+)f,", body)]
    # clamp, then +magic, -magic, -1, c3, c2, c1, 1 in source order
    return clamp + consts


def emulate(x, c):
    clamp, magic, nmagic, neg1, c3, c2, c1, one = (f32(v) for v in c[:8])
    x = np.maximum(np.asarray(x, dtype=f32), clamp)
    t = (x + magic).astype(f32)
    r = (t + nmagic).astype(f32)
    f = (r * neg1 + x).astype(f32)
    p = (c3 * f + c2).astype(f32)
    p = (p * f + c1).astype(f32)
    p = (p * f + one).astype(f32)
    bits = (t.view(np.uint32).astype(np.uint64) * 8388608 + p.view(np.uint32).astype(np.uint64)) % (1 << 32)
    return bits.astype(np.uint32).view(f32)


def test_coefficients_are_read_from_the_header():
    c = header_coefficients()
    assert len(c) == 8, c
    assert c[0] == -125.0
    assert c[1] == 12582912.0 and c[2] == -12582912.0 and c[3] == -1.0 and c[7] == 1.0


def test_relative_error_bound_and_exact_one():
    c = header_coefficients()
    rng = np.random.default_rng(0)
    x = np.concatenate([-rng.random(1 << 20) * 125.0, -np.arange(0, 125, 0.125),
                        [0.0, -0.5, -1e-7, -0.4999999, -124.9]]).astype(f32)
    y = emulate(x, c).astype(np.float64)
    ref = 2.0 ** x.astype(np.float64)
    assert np.max(np.abs(y / ref - 1.0)) <= 1.1e-4
    assert emulate(np.array([0.0], f32), c)[0] == 1.0
    n = np.arange(-125, 1).astype(f32)
    assert np.array_equal(emulate(n, c).astype(np.float64), 2.0 ** n.astype(np.float64))


def test_clamp_keeps_tiny_results_normal_and_positive():
    c = header_coefficients()
    y = emulate(np.array([-126.0, -200.0, -1e30], f32), c)
    assert np.all(y > 0) and np.all(np.isfinite(y))
    assert np.all(y >= np.finfo(np.float32).tiny)
    assert np.all(y <= 2.0 ** -124)

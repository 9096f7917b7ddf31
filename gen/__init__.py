"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the fp64 oracle's tests and by the GPU path's tests
and benchmark. It produces the *bit patterns* of the 16-bit Q, K and V tensors
and nothing else: it holds none of the attention arithmetic.

Recipe (one portable stream per workload):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) in its counter form: the i-th output (i = 1, 2, ...)
  is the SplitMix64 finaliser applied to ``seed + i * 0x9E3779B97F4A7C15``
  (mod 2**64).
* Each output becomes a uniform in (0, 1]: ``((z >> 11) + 1) * 2**-53``.
* Box-Muller in double precision turns the uniforms u(2k), u(2k+1) into two
  standard normals ``r*cos(2*pi*u2)`` and ``r*sin(2*pi*u2)`` with
  ``r = sqrt(-2*ln(u1))``.
* The normals are multiplied by ``amp`` (1 for most workloads, 3 for the
  sharper-softmax workload) and rounded once, from double, to bf16 or fp16 with
  round-to-nearest-even.
* Q, K and V are drawn in that order from one stream: Q takes the first |Q|
  normals, K the next |K|, V the next |V|.
* FP8 workloads (e4m3 inputs) draw the same normals and quantise each tensor
  per (batch, KV head) group -- for Q the group is the query heads that share
  that KV head: descale = max|x| / 448 over the group (1 if the group is all
  zero), code = e4m3(x / descale) rounded to nearest-even from double,
  saturating at the largest finite e4m3 value 448. The dequantised input is
  code * descale.

Everything is vectorised with numpy and processed in bounded chunks, so the
largest workloads (about 10**8 values) need a few hundred MB of host memory.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = [
    "BF16",
    "FP16",
    "Workload",
    "splitmix64",
    "normals",
    "round_to_16bit",
    "bits_to_float32",
    "make_qkv",
    "E4M3",
    "e4m3_encode",
    "make_qkv_fp8",
    "WORKLOADS",
    "workload",
]

BF16 = 0
FP16 = 1
E4M3 = 2        # 8-bit float, 4 exponent bits (bias 7), 3 mantissa bits, no infinities
E4M3_MAX = 448.0

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start+1 .. start+count of the SplitMix64 stream of ``seed``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _uniform(z: np.ndarray) -> np.ndarray:
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normals(seed: int, start: int, count: int) -> np.ndarray:
    """Standard normals start .. start+count-1 of the stream (``start`` even)."""
    if start % 2:
        raise ValueError("normals are produced in Box-Muller pairs; start must be even")
    out = np.empty(count, dtype=np.float64)
    done = 0
    while done < count:
        n = min(_CHUNK, count - done)
        pairs = (n + 1) // 2
        z = splitmix64(seed, start + done, 2 * pairs)
        u1 = _uniform(z[0::2])
        u2 = _uniform(z[1::2])
        r = np.sqrt(-2.0 * np.log(u1))
        t = (2.0 * math.pi) * u2
        pair = np.empty(2 * pairs, dtype=np.float64)
        pair[0::2] = r * np.cos(t)
        pair[1::2] = r * np.sin(t)
        out[done:done + n] = pair[:n]
        done += n
    return out


def round_to_16bit(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round doubles once to bf16 or fp16 (nearest-even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    if dtype == FP16:
        return x.astype(np.float16).view(np.uint16)
    if dtype != BF16:
        raise ValueError(f"unknown dtype {dtype}")
    # bf16 keeps the top 8 significand bits; round the double's 52-bit fraction
    # at bit 45 to nearest-even, then the value is exact in float32 and bf16.
    bits = x.view(np.uint64)
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    with np.errstate(over="ignore"):
        bits = bits + np.uint64((1 << 44) - 1) + lsb
    bits = bits & ~np.uint64((1 << 45) - 1)
    f32 = bits.view(np.float64).astype(np.float32)
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bits_to_float32(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact widening of 16-bit patterns to float32 (for inspection only)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == FP16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_qkv(seed: int, B: int, Hq: int, Hkv: int, N: int, d: int,
             dtype: int = BF16, amp: float = 1.0):
    """Q [B,Hq,N,d], K and V [B,Hkv,N,d] as uint16 bit patterns."""
    nq = B * Hq * N * d
    nkv = B * Hkv * N * d
    out = []
    start = 0
    for count, shape in ((nq, (B, Hq, N, d)), (nkv, (B, Hkv, N, d)), (nkv, (B, Hkv, N, d))):
        vals = normals(seed, start, count)
        if amp != 1.0:
            vals *= amp
        out.append(round_to_16bit(vals, dtype).reshape(shape))
        start += count + (count % 2)
    return tuple(out)


def make_tensor(seed: int, shape, dtype: int = BF16, amp: float = 1.0) -> np.ndarray:
    """One tensor of iid N(0, amp^2) values rounded to 16 bits (uint16 bits),
    from the start of the stream of ``seed``."""
    count = int(np.prod(shape))
    vals = normals(seed, 0, count)
    if amp != 1.0:
        vals *= amp
    return round_to_16bit(vals, dtype).reshape(shape)


def _e4m3_table() -> np.ndarray:
    """Values of the 127 non-negative finite e4m3 codes 0x00..0x7E, in code
    order (which is value order): subnormals m/8 * 2**-6 for exponent field 0,
    (1 + m/8) * 2**(e - 7) otherwise."""
    codes = np.arange(127)
    e, m = codes >> 3, codes & 7
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))


_E4M3 = _e4m3_table()


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """e4m3 codes (uint8) of doubles: nearest value, ties to the even code,
    magnitudes above 448 saturate to 448 (input quantisation only)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_E4M3, a, side="left"), 1, 126)
    lo = hi - 1
    dlo, dhi = a - _E4M3[lo], _E4M3[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == 0.0, 0, code).astype(np.uint8)
    return code | np.where(x < 0, 0x80, 0).astype(np.uint8)


def make_qkv_fp8(seed: int, B: int, Hq: int, Hkv: int, N: int, d: int, amp: float = 1.0):
    """FP8 inputs: (q, k, v, q_descale, k_descale, v_descale). q [B,Hq,N,d],
    k and v [B,Hkv,N,d] as e4m3 codes (uint8); descales float32 [B*Hkv],
    exactly representable in fp32 (they are rounded to fp32 before the
    codes are computed)."""
    nq = B * Hq * N * d
    nkv = B * Hkv * N * d
    out, scales = [], []
    start = 0
    for count, shape in ((nq, (B, Hq, N, d)), (nkv, (B, Hkv, N, d)), (nkv, (B, Hkv, N, d))):
        vals = normals(seed, start, count).reshape(shape)
        if amp != 1.0:
            vals *= amp
        g = vals.reshape(B * Hkv, -1)
        amax = np.abs(g).max(axis=1)
        descale = np.where(amax > 0, amax / E4M3_MAX, 1.0).astype(np.float32).astype(np.float64)
        out.append(e4m3_encode(g / descale[:, None]).reshape(shape))
        scales.append(descale.astype(np.float32))
        start += count + (count % 2)
    return (*out, *scales)


@dataclass(frozen=True)
class Workload:
    """One attention-forward workload: shapes, dtype, scale and input recipe."""

    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    dtype: int
    seed: int
    amp: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> int:
        return 4 * self.B * self.Hq * self.N * self.N * self.d

    @property
    def alg_bytes(self) -> int:
        """Q, K, V read once, O (16-bit) and LSE written once; FP8 inputs are
        one byte per element (plus 12 bytes of descales per KV head)."""
        es = 1 if self.fp8 else 2
        q = self.B * self.Hq * self.N * self.d
        kv = self.B * self.Hkv * self.N * self.d
        extra = 12 * self.B * self.Hkv if self.fp8 else 0
        return es * q + 2 * es * kv + 2 * q + 4 * self.B * self.Hq * self.N + extra

    @property
    def fp8(self) -> bool:
        return self.dtype == E4M3

    def inputs(self):
        """16-bit workloads: (q, k, v) bit patterns. FP8 workloads:
        (q, k, v, q_descale, k_descale, v_descale)."""
        if self.fp8:
            return make_qkv_fp8(self.seed, self.B, self.Hq, self.Hkv, self.N, self.d, self.amp)
        return make_qkv(self.seed, self.B, self.Hq, self.Hkv, self.N, self.d,
                        self.dtype, self.amp)

    def grad_output(self):
        """The upstream gradient dO [B,Hq,N,d] for backward runs: N(0,1)
        from seed + 50000 (independent of Q, K and V)."""
        return make_tensor(self.seed + 50000, (self.B, self.Hq, self.N, self.d), self.dtype)


def _sweep():
    out = []
    for n in (512, 1024, 2048, 4096, 8192, 16384):
        for dt, tag in ((FP16, "fp16"), (BF16, "bf16")):
            out.append(Workload(f"sweep_N{n}_{tag}", 16384 // n, 16, 16, n, 128, dt,
                                1002 + n))
    return out


WORKLOADS = {w.name: w for w in [
    Workload("tiny_B1_H1_N128_d128_bf16", 1, 1, 1, 128, 128, BF16, 1000),
    Workload("mha_B4_H16_N4096_d128_bf16", 4, 16, 16, 4096, 128, BF16, 1001),
    *_sweep(),
    Workload("sharp_B8_H32_N2048_d64_bf16_x3", 8, 32, 32, 2048, 64, BF16, 1003, 3.0),
    Workload("gqa_B2_Hq32_Hkv8_N8192_d128_bf16", 2, 32, 8, 8192, 128, BF16, 1004),
    Workload("fp8_mha_B4_H16_N4096_d128_e4m3", 4, 16, 16, 4096, 128, E4M3, 1101),
    Workload("fp8_gqa_B2_Hq32_Hkv8_N8192_d128_e4m3", 2, 32, 8, 8192, 128, E4M3, 1104),
    Workload("fp8_sweep_N16384_d128_e4m3", 1, 16, 16, 16384, 128, E4M3, 1102 + 16384),
]}


def workload(name: str) -> Workload:
    return WORKLOADS[name]

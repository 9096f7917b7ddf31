"""fp64 CPU oracle for the FlashAttention-2 forward pass (test infrastructure).

Only the tests, the package's ``smoke()`` check and the benchmark's CPU
baseline may import this module. The GPU library and its Python binding never
do. The arithmetic lives in ``oracle.c`` (the plain definition of attention in
double precision, the full score row materialised); this wrapper only builds
that file with gcc and marshals numpy arrays to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP16 = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP) if it is missing or stale."""
    with _lock:
        stale = (not os.path.exists(_LIB)
                 or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
                   "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64 = ctypes.c_int64
        p = ctypes.c_void_p
        lib.oracle_attention_rows.argtypes = [p, p, p, ctypes.c_int, i64, i64, i64, i64, i64,
                                              ctypes.c_double, p, i64, p, p, ctypes.c_int]
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_softmax_row.argtypes = [p, p, ctypes.c_int, i64, i64, i64, i64, i64,
                                           ctypes.c_double, i64, p]
        lib.oracle_softmax_row.restype = ctypes.c_int
        lib.oracle_decode16.argtypes = [p, i64, ctypes.c_int, p]
        lib.oracle_decode16.restype = None
        lib.oracle_attention_ex_rows.argtypes = [p, p, p, ctypes.c_int, i64, i64, i64, i64, i64, i64,
                                                 ctypes.c_double, ctypes.c_int, p, i64, p, p,
                                                 ctypes.c_int]
        lib.oracle_attention_ex_rows.restype = ctypes.c_int
        lib.oracle_attention_bwd.argtypes = [p, p, p, p, ctypes.c_int, i64, i64, i64, i64, i64,
                                             ctypes.c_double, ctypes.c_int, p, p, p, p, p, p]
        lib.oracle_attention_bwd.restype = ctypes.c_int
        lib.oracle_attention_f64.argtypes = [p, p, p, i64, i64, i64, i64, i64, ctypes.c_double,
                                             ctypes.c_int, p]
        lib.oracle_attention_f64.restype = ctypes.c_int
        lib.oracle_decode_e4m3.argtypes = [p, i64, p]
        lib.oracle_decode_e4m3.restype = None
        lib.oracle_round_e4m3.argtypes = [p, i64, p]
        lib.oracle_round_e4m3.restype = None
        lib.oracle_attention_fp8_rows.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64, i64,
                                                  ctypes.c_double, ctypes.c_int, i64, p, i64, p, p, p, p, p,
                                                  ctypes.c_int]
        lib.oracle_attention_fp8_rows.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are 16-bit bit patterns (uint16)")
    return a


def decode16(bits, dtype: int) -> np.ndarray:
    """Exact double values of bf16 (dtype 0) or fp16 (dtype 1) bit patterns."""
    bits = _u16(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_decode16(bits.ctypes.data, bits.size, dtype, out.ctypes.data)
    return out


def attention(q, k, v, scale: float, dtype: int, rows=None, threads: int = 0):
    """Exact attention forward in fp64.

    q: uint16 [B, Hq, N, d]; k, v: uint16 [B, Hkv, N, d].
    rows: optional flat query-row indices (b*Hq + h)*N + i.
    Returns (o, lse): o float64 [B, Hq, N, d] (or [len(rows), d]) and
    lse float64 [B, Hq, N] (or [len(rows)]).
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, N, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if (Bk, Nk, dk) != (B, N, d) or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k and v")
    if rows is None:
        nrows = B * Hq * N
        rows_arr = None
        rptr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
        rptr = rows_arr.ctypes.data
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty(nrows, dtype=np.float64)
    rc = _load().oracle_attention_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dtype,
                                       B, Hq, Hkv, N, d, float(scale), rptr, nrows,
                                       o.ctypes.data, lse.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    if rows is None:
        return o.reshape(B, Hq, N, d), lse.reshape(B, Hq, N)
    return o, lse


def attention_ex(q, k, v, scale: float, dtype: int, causal: bool = False, rows=None,
                 threads: int = 0):
    """Attention forward with independent query/key lengths and an optional
    causal mask (key j allowed for query i iff j < min(Nk, i + 1 + Nk - Nq)).

    q: uint16 [B, Hq, Nq, d]; k, v: uint16 [B, Hkv, Nk, d]. Rows with no
    allowed key give o = 0 and lse = -inf. Returns (o, lse) shaped like
    :func:`attention` (rows index [B, Hq, Nq]).
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if (Bk, dk) != (B, d) or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k and v")
    if rows is None:
        nrows = B * Hq * Nq
        rptr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
        rptr = rows_arr.ctypes.data
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty(nrows, dtype=np.float64)
    rc = _load().oracle_attention_ex_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, dtype,
                                          B, Hq, Hkv, Nq, Nk, d, float(scale), int(bool(causal)),
                                          rptr, nrows, o.ctypes.data, lse.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    if rows is None:
        return o.reshape(B, Hq, Nq, d), lse.reshape(B, Hq, Nq)
    return o, lse


def attention_bwd(q, k, v, dout, scale: float, dtype: int, causal: bool = False, bounds: bool = False):
    """Gradients (dq, dk, dv) of attention for upstream gradient dout, fp64.

    q, dout: uint16 [B, Hq, N, d]; k, v: uint16 [B, Hkv, N, d]. With grouped
    heads dk and dv sum over the query heads of each KV head.

    bounds=True also returns a dict of the absolute sums that bound the
    error of a computation rounding P, dS and O to 16 bits (see oracle.c):
    ``q`` and ``k`` are [3, ...] arrays (A, BE, BF) shaped like dq and dk,
    ``v`` is A shaped like dv.
    """
    q, k, v, dout = _u16(q), _u16(k), _u16(v), _u16(dout)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape or dout.shape != q.shape:
        raise ValueError("shape mismatch")
    dq = np.empty(q.shape, dtype=np.float64)
    dk = np.empty(k.shape, dtype=np.float64)
    dv = np.empty(v.shape, dtype=np.float64)
    bq = np.empty((3,) + q.shape, dtype=np.float64) if bounds else None
    bk = np.empty((3,) + k.shape, dtype=np.float64) if bounds else None
    bv = np.empty(v.shape, dtype=np.float64) if bounds else None
    ptr = lambda a: None if a is None else a.ctypes.data
    rc = _load().oracle_attention_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data,
                                      dtype, B, Hq, Hkv, N, d, float(scale), int(bool(causal)),
                                      dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
                                      ptr(bq), ptr(bk), ptr(bv))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    if bounds:
        return dq, dk, dv, {"q": bq, "k": bk, "v": bv}
    return dq, dk, dv


def attention_f64(q, k, v, scale: float, causal: bool = False) -> np.ndarray:
    """Forward on float64 inputs (q [B,Hq,N,d], k/v [B,Hkv,N,d]); returns o."""
    q, k, v = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v))
    B, Hq, N, d = q.shape
    o = np.empty(q.shape, dtype=np.float64)
    rc = _load().oracle_attention_f64(q.ctypes.data, k.ctypes.data, v.ctypes.data, B, Hq, k.shape[1], N,
                                      d, float(scale), int(bool(causal)), o.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    return o


def decode_e4m3(codes) -> np.ndarray:
    """Exact double values of e4m3 codes (uint8)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_decode_e4m3(c.ctypes.data, c.size, out.ctypes.data)
    return out


def round_e4m3(x) -> np.ndarray:
    """Doubles rounded to the nearest e4m3 value (ties to even, saturating at 448)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    _load().oracle_round_e4m3(x.ctypes.data, x.size, out.ctypes.data)
    return out


def attention_fp8_both(q, k, v, q_descale, k_descale, v_descale, scale: float, rows=None,
                       threads: int = 0, bc: int = 128, causal: bool = False, method: bool = True):
    """Attention forward on e4m3 inputs with per-(batch, KV head) descales,
    in one pass: returns (o_method, o_plain, lse, a, b).

    q: uint8 [B, Hq, Nq, d]; k, v: uint8 [B, Hkv, Nk, d]; descales: [B*Hkv].
    causal: query row i sees keys j < min(Nk, i + 1 + Nk - Nq) (rows that
    see none: o = 0, lse = -inf). o_method follows the FP8 method: the
    online softmax over key tiles of bc keys (from key 0), with each tile's
    weights scaled by 2^8 and rounded to e4m3 (against the tile's running
    max) before the P.V product; o_plain is the plain definition on the
    dequantised inputs. o_*, a, b: [B, Hq, Nq, d] (or [len(rows), d]); lse:
    [B, Hq, N] (or [len(rows)]); a = sum_j p_j |v_j| / l and
    b = sum_j |v_j| / l elementwise. method=False skips the method (o_method
    is then None).
    """
    q, k, v = (np.ascontiguousarray(x, dtype=np.uint8) for x in (q, k, v))
    B, Hq, N, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape != (B, Hkv, Nk, d) or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k and v")
    qd, kd, vd = (np.ascontiguousarray(x, dtype=np.float64).reshape(-1) for x in
                  (q_descale, k_descale, v_descale))
    if not (qd.size == kd.size == vd.size == B * Hkv):
        raise ValueError("descales must have B*Hkv entries")
    if rows is None:
        nrows, rptr = B * Hq * N, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rptr = rows_arr.size, rows_arr.ctypes.data
    om = np.empty((nrows, d), dtype=np.float64) if method else None
    op, a, b = (np.empty((nrows, d), dtype=np.float64) for _ in range(3))
    lse = np.empty(nrows, dtype=np.float64)
    rc = _load().oracle_attention_fp8_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, qd.ctypes.data,
                                           kd.ctypes.data, vd.ctypes.data, B, Hq, Hkv, N, Nk, d, float(scale),
                                           int(bool(causal)), int(bc), rptr, nrows,
                                           None if om is None else om.ctypes.data, op.ctypes.data,
                                           lse.ctypes.data, a.ctypes.data, b.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    if rows is None:
        shp = (B, Hq, N, d)
        return (None if om is None else om.reshape(shp)), op.reshape(shp), lse.reshape(B, Hq, N), \
            a.reshape(shp), b.reshape(shp)
    return om, op, lse, a, b


def attention_fp8(q, k, v, q_descale, k_descale, v_descale, scale: float, round_p: bool = True,
                  rows=None, threads: int = 0, bc: int = 128, causal: bool = False):
    """(o, lse, a, b) of :func:`attention_fp8_both`, with o the method's
    output (round_p=True) or the plain definition's (round_p=False)."""
    om, op, lse, a, b = attention_fp8_both(q, k, v, q_descale, k_descale, v_descale, scale, rows, threads, bc,
                                           causal, method=round_p)
    return (om if round_p else op), lse, a, b


def softmax_row(q, k, scale: float, dtype: int, row: int) -> np.ndarray:
    """The normalised softmax weights of one query row (flat index), fp64 [N]."""
    q, k = _u16(q), _u16(k)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    p = np.empty(N, dtype=np.float64)
    rc = _load().oracle_softmax_row(q.ctypes.data, k.ctypes.data, dtype, B, Hq, Hkv, N, d,
                                    float(scale), int(row), p.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    return p


def max_threads() -> int:
    return _load().oracle_max_threads()

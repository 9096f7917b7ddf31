"""Python binding of the C ABI in include/fa2.h (argument marshalling only).

Every entry point forwards raw device pointers, sizes and the CUDA stream
handle to ``libfa2.so``; all compute runs in the library's sm_103a kernel.
If the library cannot be loaded the call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa2.so")

FA2_BF16 = 0
FA2_FP16 = 1

FA2_OK = 0
FA2_ERR_INVALID_ARG = 1
FA2_ERR_UNSUPPORTED = 2
FA2_ERR_CUDA = 3
FA2_ERR_TIMEOUT = 4
FA2_ERR_BOUNDS = 5   # debug builds only: a device-side bounds check failed

# symbols declared in include/fa2.h
EXPORTS = ("fa2_fwd", "fa2_fwd_gqa", "fa2_fwd_ex", "fa2_fwd_fp8", "fa2_fwd_fp8_ex", "fa2_bwd", "fa2_bwd_noalloc", "fa2_check_status",
           "fa2_status_string",
           "fa2_set_wait_limit_ns", "fa2_set_debug_flags", "fa2_set_tile_config", "fa2_version")

_lib = None


class FA2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed: {status_string(status)}")


def load(path: str = LIB_PATH):
    """Load libfa2.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"CUDA library {path} is missing: run __graft_entry__.build() "
                          "(python -m attention_fa2_forward_03_gb300.build)")
    lib = ctypes.CDLL(path)
    p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa2_fwd.argtypes = [p, p, p, p, p, i, i, i, i, f, i, p]
    lib.fa2_fwd.restype = i
    lib.fa2_fwd_gqa.argtypes = [p, p, p, p, p, i, i, i, i, i, f, i, p]
    lib.fa2_fwd_gqa.restype = i
    lib.fa2_fwd_ex.argtypes = [p, p, p, p, p, i, i, i, i, i, i, f, i, i, p]
    lib.fa2_fwd_ex.restype = i
    lib.fa2_fwd_fp8.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, f, p]
    lib.fa2_fwd_fp8.restype = i
    lib.fa2_fwd_fp8_ex.argtypes = [p, p, p, p, p, p, p, p, i, i, i, i, i, i, f, i, p]
    lib.fa2_fwd_fp8_ex.restype = i
    lib.fa2_bwd.argtypes = [p, p, p, p, p, p, p, p, p, p, i, i, i, i, i, f, i, i, p]
    lib.fa2_bwd.restype = i
    lib.fa2_bwd_noalloc.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, f, i, i, p]
    lib.fa2_bwd_noalloc.restype = i
    lib.fa2_check_status.argtypes = [p]
    lib.fa2_check_status.restype = i
    lib.fa2_status_string.argtypes = [i]
    lib.fa2_status_string.restype = ctypes.c_char_p
    lib.fa2_set_wait_limit_ns.argtypes = [ctypes.c_int64]
    lib.fa2_set_wait_limit_ns.restype = ctypes.c_int64
    lib.fa2_set_debug_flags.argtypes = [i]
    lib.fa2_set_debug_flags.restype = i
    lib.fa2_set_tile_config.argtypes = [i]
    lib.fa2_set_tile_config.restype = i
    lib.fa2_version.argtypes = []
    lib.fa2_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().fa2_status_string(int(status)).decode()


# ------------------------------------------------------------------ raw pointer API

def fa2_fwd_gqa_ptr(q, k, v, o, lse, B, H_q, H_kv, N, d, scale, dtype, stream=0) -> int:
    """fa2_fwd_gqa on raw device addresses (ints); returns the status code."""
    return load().fa2_fwd_gqa(q, k, v, o, lse, B, H_q, H_kv, N, d, float(scale), int(dtype),
                              stream or None)


def fa2_fwd_ptr(q, k, v, o, lse, B, H, N, d, scale, dtype, stream=0) -> int:
    """fa2_fwd on raw device addresses (ints); returns the status code."""
    return load().fa2_fwd(q, k, v, o, lse, B, H, N, d, float(scale), int(dtype), stream or None)


def fa2_fwd_ex_ptr(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, scale, causal, dtype, stream=0) -> int:
    """fa2_fwd_ex on raw device addresses (ints); returns the status code."""
    return load().fa2_fwd_ex(q, k, v, o, lse, B, H_q, H_kv, N_q, N_k, d, float(scale), int(causal),
                             int(dtype), stream or None)


def fa2_fwd_fp8_ptr(q, k, v, q_descale, k_descale, v_descale, o, lse, B, H_q, H_kv, N, d, scale,
                    stream=0) -> int:
    """fa2_fwd_fp8 on raw device addresses (ints); returns the status code."""
    return load().fa2_fwd_fp8(q, k, v, q_descale, k_descale, v_descale, o, lse, B, H_q, H_kv, N, d,
                              float(scale), stream or None)


def fa2_fwd_fp8_ex_ptr(q, k, v, q_descale, k_descale, v_descale, o, lse, B, H_q, H_kv, N_q, N_k, d, scale,
                       causal, stream=0) -> int:
    """fa2_fwd_fp8_ex on raw device addresses (ints); returns the status code."""
    return load().fa2_fwd_fp8_ex(q, k, v, q_descale, k_descale, v_descale, o, lse, B, H_q, H_kv, N_q, N_k, d,
                                 float(scale), int(causal), stream or None)


def fa2_bwd_ptr(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H_q, H_kv, N, d, scale, causal, dtype,
                stream=0) -> int:
    """fa2_bwd on raw device addresses (ints); returns the status code."""
    return load().fa2_bwd(q, k, v, o, lse, dout, dq, dk, dv, delta, B, H_q, H_kv, N, d, float(scale),
                          int(causal), int(dtype), stream or None)


def fa2_bwd_noalloc_ptr(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N, d, scale, causal, dtype,
                        stream=0) -> int:
    """fa2_bwd_noalloc on raw device addresses (ints): the backward without a
    caller-provided workspace, for callers that cannot allocate device
    memory (at most 2**20 query rows). Returns the status code."""
    return load().fa2_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N, d, float(scale),
                                  int(causal), int(dtype), stream or None)


def fa2_check_status(stream=0) -> int:
    return load().fa2_check_status(stream or None)


def fa2_set_wait_limit_ns(limit_ns: int) -> int:
    return load().fa2_set_wait_limit_ns(int(limit_ns))


def fa2_set_debug_flags(flags: int) -> int:
    return load().fa2_set_debug_flags(int(flags))


# bit 0 of fa2_set_tile_config: d = 64, equal lengths, on the 16-bit kernel's d = 64 path
TILE_CFG_D64_SHARED = 1


def fa2_set_tile_config(config: int) -> int:
    """Planner choice for d = 64 with equal lengths (see include/fa2.h);
    returns the previous value, -1 if `config` was rejected."""
    return load().fa2_set_tile_config(int(config))


def fa2_version() -> str:
    return load().fa2_version().decode()


# ------------------------------------------------------------------ torch tensors

def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return FA2_BF16
    if t.dtype == torch.float16:
        return FA2_FP16
    raise TypeError(f"q/k/v must be bf16 or fp16, got {t.dtype}")


def _stream_handle(stream, device) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def fa2_fwd_gqa(q, k, v, o=None, lse=None, scale=None, stream=None):
    """Attention forward on CUDA tensors q [B,Hq,N,d], k/v [B,Hkv,N,d].

    Allocates o / lse with torch when they are not given (that is device-memory
    plumbing; the library itself allocates nothing). Returns (o, lse).
    """
    import torch

    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, N, d]")
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, N, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, Hkv, N, d] with q's B, N and d")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k and v must be contiguous CUDA tensors")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    if o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous():
        raise ValueError("o must be a contiguous tensor like q")
    if tuple(lse.shape) != (B, Hq, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, Hq, N]")
    if scale is None:
        scale = d ** -0.5
    rc = fa2_fwd_gqa_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         B, Hq, Hkv, N, d, scale, _dtype_code(q), _stream_handle(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error(rc, "fa2_fwd_gqa")
    return o, lse


def fa2_fwd_ex(q, k, v, o=None, lse=None, scale=None, causal=False, stream=None):
    """General attention forward: q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d], any Nq, Nk,
    optional causal mask (end-aligned). Returns (o, lse)."""
    import torch

    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, N, d]")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nk, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, Hkv, Nk, d] with q's B and d")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k and v must be contiguous CUDA tensors")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    if o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous():
        raise ValueError("o must be a contiguous tensor like q")
    if tuple(lse.shape) != (B, Hq, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, Hq, Nq]")
    if scale is None:
        scale = d ** -0.5
    rc = fa2_fwd_ex_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, Hq, Hkv, Nq, Nk, d, scale, bool(causal), _dtype_code(q),
                        _stream_handle(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error(rc, "fa2_fwd_ex")
    return o, lse


def fa2_bwd(q, k, v, o, lse, dout, scale=None, causal=False, dq=None, dk=None, dv=None, delta=None,
            stream=None):
    """Gradients (dq, dk, dv) of the forward for upstream gradient dout.

    q, o, dout: [B, Hq, N, d]; k, v: [B, Hkv, N, d]; lse: fp32 [B, Hq, N]
    from the forward. Outputs and the fp32 workspace `delta` [B, Hq, N] are
    allocated with torch when not given (device-memory plumbing only).
    """
    import torch

    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    for t in (q, k, v, o, dout, lse):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    if tuple(k.shape) != (B, Hkv, N, d) or v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("shape mismatch")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    delta = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device) if delta is None else delta
    if scale is None:
        scale = d ** -0.5
    rc = fa2_bwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                     dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), delta.data_ptr(), B, Hq, Hkv, N, d, scale,
                     bool(causal), _dtype_code(q), _stream_handle(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error(rc, "fa2_bwd")
    return dq, dk, dv


def _fp8_prepare(q, k, v, q_descale, k_descale, v_descale, o, lse, same_len):
    """Check the FP8 arguments and allocate missing outputs; returns
    (o, lse, B, Hq, Hkv, Nq, Nk, d)."""
    import torch

    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, N, d]")
    B, Hq, N, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if same_len and Nk != N:
        raise ValueError("k and v must be [B, Hkv, N, d] with q's B, N and d")
    if tuple(k.shape) != (B, Hkv, Nk, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, Nk, d] with q's B and d")
    for t in (q, k, v):
        if t.element_size() != 1 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k and v must be contiguous one-byte (e4m3) CUDA tensors")
    for t in (q_descale, k_descale, v_descale):
        if t.dtype != torch.float32 or not t.is_cuda or t.numel() != B * Hkv or not t.is_contiguous():
            raise ValueError("descales must be contiguous fp32 CUDA tensors of B*Hkv elements")
    if o is None:
        o = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    if tuple(o.shape) != (B, Hq, N, d) or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("o must be a contiguous bf16 tensor [B, Hq, N, d]")
    if tuple(lse.shape) != (B, Hq, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [B, Hq, N]")
    return o, lse, B, Hq, Hkv, N, Nk, d


def fa2_fwd_fp8(q, k, v, q_descale, k_descale, v_descale, o=None, lse=None, scale=None, stream=None):
    """FP8 attention forward: q [B,Hq,N,d], k/v [B,Hkv,N,d] e4m3 codes as
    uint8 (or torch.float8_e4m3fn) CUDA tensors, descales fp32 [B*Hkv] CUDA
    tensors. Returns (o, lse) with o bf16 [B,Hq,N,d] and lse fp32 [B,Hq,N]."""
    o, lse, B, Hq, Hkv, N, _, d = _fp8_prepare(q, k, v, q_descale, k_descale, v_descale, o, lse, True)
    if scale is None:
        scale = d ** -0.5
    rc = fa2_fwd_fp8_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), q_descale.data_ptr(), k_descale.data_ptr(),
                         v_descale.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, N, d, scale,
                         _stream_handle(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error(rc, "fa2_fwd_fp8")
    return o, lse


def fa2_fwd_fp8_ex(q, k, v, q_descale, k_descale, v_descale, o=None, lse=None, scale=None, causal=False,
                   stream=None):
    """General FP8 attention forward: q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d] e4m3
    codes, any Nq, Nk, optional causal mask (end-aligned). Returns (o, lse)
    with o bf16 [B,Hq,Nq,d] and lse fp32 [B,Hq,Nq]."""
    o, lse, B, Hq, Hkv, Nq, Nk, d = _fp8_prepare(q, k, v, q_descale, k_descale, v_descale, o, lse, False)
    if scale is None:
        scale = d ** -0.5
    rc = fa2_fwd_fp8_ex_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), q_descale.data_ptr(), k_descale.data_ptr(),
                            v_descale.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, scale,
                            bool(causal), _stream_handle(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error(rc, "fa2_fwd_fp8_ex")
    return o, lse


def fa2_fwd(q, k, v, o=None, lse=None, scale=None, stream=None):
    """Multi-head attention forward: q, k, v all [B, H, N, d]. Returns (o, lse)."""
    if q.shape[1] != k.shape[1]:
        raise ValueError("fa2_fwd needs equal head counts; use fa2_fwd_gqa")
    return fa2_fwd_gqa(q, k, v, o, lse, scale, stream)

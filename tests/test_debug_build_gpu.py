"""The debug build (libfa2_debug.so, compiled with FA2_DEBUG).

In that build every tile start given to a TMA copy and every global row the
kernels store or load outside TMA is checked against the extents the host
planned with; a failed check reports FA2_ERR_BOUNDS through
fa2_check_status and skips the access instead of touching memory. It stands
in for a memory checker on machines where none can run. These tests drive
every entry point through the debug build on shapes that exercise the edge
paths (odd tile counts, ragged lengths, causal rows with no key, grouped
heads, FP8, the backward) and require that no check fires and that the
results are bit for bit those of the release build.
"""
import ctypes
import math

import numpy as np
import pytest

import gen
from attention_fa2_forward_03_gb300 import build, fa2

p_, i_, f_ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float


def _bind(path):
    lib = ctypes.CDLL(path)
    lib.fa2_fwd_gqa.argtypes = [p_, p_, p_, p_, p_, i_, i_, i_, i_, i_, f_, i_, p_]
    lib.fa2_fwd_ex.argtypes = [p_, p_, p_, p_, p_, i_, i_, i_, i_, i_, i_, f_, i_, i_, p_]
    lib.fa2_fwd_fp8.argtypes = [p_, p_, p_, p_, p_, p_, p_, p_, i_, i_, i_, i_, i_, f_, p_]
    lib.fa2_fwd_fp8_ex.argtypes = [p_, p_, p_, p_, p_, p_, p_, p_, i_, i_, i_, i_, i_, i_, f_, i_, p_]
    lib.fa2_bwd.argtypes = [p_] * 10 + [i_, i_, i_, i_, i_, f_, i_, i_, p_]
    lib.fa2_check_status.argtypes = [p_]
    lib.fa2_version.restype = ctypes.c_char_p
    for name in ("fa2_fwd_gqa", "fa2_fwd_ex", "fa2_fwd_fp8", "fa2_fwd_fp8_ex", "fa2_bwd", "fa2_check_status"):
        getattr(lib, name).restype = i_
    return lib


@pytest.fixture(scope="module")
def libs(gpu_lib):
    build.build()
    return _bind(build.LIB), _bind(build.DEBUG_LIB)


def _dev(x, dtype=None):
    import torch

    if x.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to("cuda")
        return t.view(torch.bfloat16 if dtype == gen.BF16 else torch.float16)
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda")


def _run_both(libs, launch, outs):
    """Runs `launch(lib)` on the release and the debug library into fresh
    copies of `outs` (filled with a pattern first) and returns both sets."""
    import torch

    results = []
    for lib in libs:
        bufs = [torch.full_like(o, 7.0) if o.is_floating_point() else torch.zeros_like(o) for o in outs]
        rc = launch(lib, bufs)
        assert rc == fa2.FA2_OK, rc
        rc = lib.fa2_check_status(torch.cuda.current_stream().cuda_stream)
        assert rc == fa2.FA2_OK, f"status {rc} (5 = FA2_ERR_BOUNDS)"
        results.append([b.clone() for b in bufs])
    return results


def _same(a, b):
    for x, y in zip(a, b):
        assert bool((x.view(-1).view(torch_int(x)) == y.view(-1).view(torch_int(y))).all())


def torch_int(t):
    import torch

    return {2: torch.int16, 4: torch.int32, 1: torch.uint8}[t.element_size()]


pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype", [
    (2, 4, 4, 512, 128, gen.BF16),
    (1, 6, 2, 384, 64, gen.FP16),      # grouped heads, odd tile count per KV head
])
def test_debug_build_equal_lengths(libs, B, Hq, Hkv, N, d, dtype):
    import torch

    q, k, v = gen.make_qkv(9100 + N, B, Hq, Hkv, N, d, dtype)
    tq, tk, tv = (_dev(x, dtype) for x in (q, k, v))
    o = torch.empty_like(tq)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    launch = lambda lib, b: lib.fa2_fwd_gqa(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), b[0].data_ptr(),
                                            b[1].data_ptr(), B, Hq, Hkv, N, d, d ** -0.5, dtype, s)
    rel, dbg = _run_both(libs, launch, [o, lse])
    _same(rel, dbg)


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 2, 1, 300, 300, 128, 1),
    (2, 2, 2, 500, 300, 64, 1),        # first 200 rows attend nothing
    (1, 4, 2, 200, 700, 128, 0),
    (1, 1, 1, 128, 128, 64, 0),        # single tile: general mode
])
def test_debug_build_general(libs, B, Hq, Hkv, Nq, Nk, d, causal):
    import torch

    q, _, _ = gen.make_qkv(9200 + Nq, B, Hq, Hkv, Nq, d, gen.BF16)
    _, k, v = gen.make_qkv(9300 + Nk, B, Hq, Hkv, Nk, d, gen.BF16)
    tq, tk, tv = (_dev(x, gen.BF16) for x in (q, k, v))
    o = torch.empty_like(tq)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    launch = lambda lib, b: lib.fa2_fwd_ex(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), b[0].data_ptr(),
                                           b[1].data_ptr(), B, Hq, Hkv, Nq, Nk, d, d ** -0.5, causal, gen.BF16, s)
    rel, dbg = _run_both(libs, launch, [o, lse])
    _same(rel, dbg)


@pytest.mark.parametrize("N,causal", [(512, 0), (300, 1)])
def test_debug_build_fp8(libs, N, causal):
    import torch

    B, Hq, Hkv = 1, 4, 2
    q, k, v, qd, kd, vd = gen.make_qkv_fp8(9400 + N, B, Hq, Hkv, N, 128)
    tq, tk, tv, tqd, tkd, tvd = (_dev(x) for x in (q, k, v, qd, kd, vd))
    o = torch.empty(tq.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    ptrs = (tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), tqd.data_ptr(), tkd.data_ptr(), tvd.data_ptr())
    if causal:
        launch = lambda lib, b: lib.fa2_fwd_fp8_ex(*ptrs, b[0].data_ptr(), b[1].data_ptr(), B, Hq, Hkv, N, N, 128,
                                                   0.09, 1, s)
    else:
        launch = lambda lib, b: lib.fa2_fwd_fp8(*ptrs, b[0].data_ptr(), b[1].data_ptr(), B, Hq, Hkv, N, 128, 0.09, s)
    rel, dbg = _run_both(libs, launch, [o, lse])
    _same(rel, dbg)


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [(1, 4, 2, 300, 128, 1), (2, 2, 2, 256, 64, 0)])
def test_debug_build_backward(libs, B, Hq, Hkv, N, d, causal):
    import torch

    q, k, v = gen.make_qkv(9500 + N, B, Hq, Hkv, N, d, gen.BF16)
    do, _, _ = gen.make_qkv(9501 + N, B, Hq, Hkv, N, d, gen.BF16)
    tq, tk, tv, tdo = (_dev(x, gen.BF16) for x in (q, k, v, do))
    o, lse = fa2.fa2_fwd_ex(tq, tk, tv, scale=d ** -0.5, causal=bool(causal))
    dq, dk, dv = torch.empty_like(tq), torch.empty_like(tk), torch.empty_like(tv)
    delta = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    launch = lambda lib, b: lib.fa2_bwd(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                        tdo.data_ptr(), b[0].data_ptr(), b[1].data_ptr(), b[2].data_ptr(),
                                        b[3].data_ptr(), B, Hq, Hkv, N, d, d ** -0.5, causal, gen.BF16, s)
    rel, dbg = _run_both(libs, launch, [dq, dk, dv, delta])
    _same(rel, dbg)

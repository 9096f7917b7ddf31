"""The backward entry point that allocates nothing (fa2_bwd_noalloc).

Some callers cannot allocate device memory for the backward's workspace: a
plugin that a host framework hands only its input and output tensors, or code
running where a device allocation is not allowed. fa2_bwd_noalloc keeps that
workspace in a fixed device array inside the library instead (at most 2^20
query rows). These tests call it twice in a row through the C ABI and check
both results against the allocating entry point (fa2_bwd, whose workspace
comes from the caller: bit for bit, the kernels being the same) and against
the fp64 oracle with the backward tests' elementwise bound. The file is
collected last and passes run alone or after the other GPU tests.
"""
import math

import numpy as np
import pytest

import gen
from test_backward_gpu import check_all

pytestmark = pytest.mark.gpu


def to_dev(x, dtype):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to("cuda")
    return t.view(torch.bfloat16 if dtype == gen.BF16 else torch.float16)


def noalloc_twice(fa2, tq, tk, tv, o, lse, tdo, B, Hq, Hkv, N, d, scale, causal, dtype):
    """Two fa2_bwd_noalloc calls in a row, each into outputs prefilled with
    garbage; returns both results."""
    import torch

    stream = torch.cuda.current_stream().cuda_stream
    out = []
    for fill in (9.0, -3.0):
        dq, dk, dv = (torch.full_like(t, fill) for t in (tq, tk, tv))
        rc = fa2.fa2_bwd_noalloc_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     tdo.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                     B, Hq, Hkv, N, d, scale, int(causal), dtype, stream)
        assert rc == fa2.FA2_OK, fa2.status_string(rc)
        assert fa2.fa2_check_status(stream) == fa2.FA2_OK
        out.append((dq, dk, dv))
    return out


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dtype,causal", [
    (2, 4, 2, 384, 128, gen.BF16, False),
    (2, 4, 2, 384, 128, gen.BF16, True),
    (1, 4, 2, 300, 64, gen.FP16, True),     # ragged N (not a multiple of 128), d = 64
    (2, 2, 2, 200, 64, gen.BF16, False),
])
def test_noalloc_backward_twice_matches_allocating_entry_and_oracle(gpu_lib, B, Hq, Hkv, N, d, dtype, causal):
    q, k, v = gen.make_qkv(4500 + N + d, B, Hq, Hkv, N, d, dtype)
    do, _, _ = gen.make_qkv(4501 + N + d, B, Hq, Hkv, N, d, dtype)
    scale = 1 / math.sqrt(d)
    tq, tk, tv, tdo = (to_dev(x, dtype) for x in (q, k, v, do))
    o, lse = gpu_lib.fa2_fwd_ex(tq, tk, tv, scale=scale, causal=causal)
    ref = gpu_lib.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=scale, causal=causal)
    fdt = gpu_lib.FA2_BF16 if dtype == gen.BF16 else gpu_lib.FA2_FP16
    for grads in noalloc_twice(gpu_lib, tq, tk, tv, o, lse, tdo, B, Hq, Hkv, N, d, scale, causal, fdt):
        for g, r in zip(grads, ref):
            assert bool((g == r).all())          # same kernels, same inputs: bit for bit
        check_all(*(g.float().cpu().numpy() for g in grads), q, k, v, do, scale, dtype, causal,
                  what="noalloc ")


def test_noalloc_backward_at_its_row_limit(gpu_lib):
    # B * H_q * N = 64 * 16 * 1024 = 2^20 query rows, exactly the size of the
    # fixed array: accepted, and equal bit for bit to fa2_bwd (an off-by-one
    # in the limit would write past the array or refuse this size).
    B, Hq, Hkv, N, d = 64, 16, 16, 1024, 128
    assert B * Hq * N == 1 << 20
    q, k, v = gen.make_qkv(4600, B, Hq, Hkv, N, d, gen.BF16)
    do, _, _ = gen.make_qkv(4601, B, Hq, Hkv, N, d, gen.BF16)
    tq, tk, tv, tdo = (to_dev(x, gen.BF16) for x in (q, k, v, do))
    scale = 1 / math.sqrt(d)
    o, lse = gpu_lib.fa2_fwd_gqa(tq, tk, tv, scale=scale)
    ref = gpu_lib.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=scale)
    for grads in noalloc_twice(gpu_lib, tq, tk, tv, o, lse, tdo, B, Hq, Hkv, N, d, scale, False,
                               gpu_lib.FA2_BF16):
        for g, r in zip(grads, ref):
            assert bool((g == r).all())


def test_noalloc_backward_rejects_rows_past_its_array(gpu_lib):
    import torch

    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    a = x.data_ptr()
    # 2 * 16 * 65536 = 2^21 query rows > 2^20: refused before anything runs
    rc = gpu_lib.fa2_bwd_noalloc_ptr(a, a, a, a, a, a, a, a, a, 2, 16, 16, 65536, 128, 0.1, 0, gpu_lib.FA2_BF16, 0)
    assert rc == gpu_lib.FA2_ERR_UNSUPPORTED
    # one row past the limit: 2^20 + 1 rows (B = 1, H = 1, N = 2^20 + 1)
    rc = gpu_lib.fa2_bwd_noalloc_ptr(a, a, a, a, a, a, a, a, a, 1, 1, 1, (1 << 20) + 1, 128, 0.1, 0,
                                     gpu_lib.FA2_BF16, 0)
    assert rc == gpu_lib.FA2_ERR_UNSUPPORTED

"""The backward entry point that allocates nothing (fa2_bwd_noalloc).

Some callers cannot allocate device memory for the backward's workspace: a
plugin that a host framework hands only its input and output tensors, or code
running where a device allocation is not allowed. fa2_bwd_noalloc keeps that
workspace in a fixed device array inside the library instead. This test calls
it twice in a row through the C ABI and checks both results against the
allocating entry point (fa2_bwd, whose workspace comes from the caller), with
the backward's normwise tolerance. It sits in a file of its own, collected
last, and passes run alone or after the other GPU tests.
"""
import math

import numpy as np
import pytest

import gen

pytestmark = pytest.mark.gpu


def to_dev(x, dtype):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to("cuda")
    return t.view(torch.bfloat16 if dtype == gen.BF16 else torch.float16)


def within(g, ref):
    # the backward tests' bf16 bounds: max error <= 2^-6 max|ref|, Frobenius <= 2^-7
    g, ref = g.double(), ref.double()
    err = (g - ref).abs()
    return (float(err.max()) <= 2.0 ** -6 * float(ref.abs().max())
            and float(err.norm()) <= 2.0 ** -7 * float(ref.norm()))


@pytest.mark.parametrize("causal", [False, True])
def test_noalloc_backward_matches_allocating_entry_twice(gpu_lib, causal):
    import torch

    B, Hq, Hkv, N, d = 2, 4, 2, 384, 128
    q, k, v = gen.make_qkv(4500, B, Hq, Hkv, N, d, gen.BF16)
    do, _, _ = gen.make_qkv(4501, B, Hq, Hkv, N, d, gen.BF16)
    scale = 1 / math.sqrt(d)
    tq, tk, tv, tdo = (to_dev(x, gen.BF16) for x in (q, k, v, do))
    o, lse = gpu_lib.fa2_fwd_ex(tq, tk, tv, scale=scale, causal=causal)
    ref = gpu_lib.fa2_bwd(tq, tk, tv, o, lse, tdo, scale=scale, causal=causal)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        dq, dk, dv = torch.full_like(tq, 9.0), torch.full_like(tk, 9.0), torch.full_like(tv, 9.0)
        rc = gpu_lib.fa2_bwd_noalloc_ptr(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                         tdo.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                         B, Hq, Hkv, N, d, scale, causal, gpu_lib.FA2_BF16, stream)
        assert rc == gpu_lib.FA2_OK
        assert gpu_lib.fa2_check_status(stream) == gpu_lib.FA2_OK
        for g, r in zip((dq, dk, dv), ref):
            assert within(g, r)


def test_noalloc_backward_rejects_rows_past_its_array(gpu_lib):
    import torch

    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    a = x.data_ptr()
    # 2 * 16 * 65536 = 2^21 query rows > 2^20: refused before anything runs
    rc = gpu_lib.fa2_bwd_noalloc_ptr(a, a, a, a, a, a, a, a, a, 2, 16, 16, 65536, 128, 0.1, 0, gpu_lib.FA2_BF16, 0)
    assert rc == gpu_lib.FA2_ERR_UNSUPPORTED

"""The C-ABI library loads, exports every symbol include/fa2.h declares, and
rejects invalid arguments on the host before touching a device (CPU only)."""
import ctypes
import os
import re

import pytest

from attention_fa2_forward_03_gb300 import build, fa2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa2.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa2.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa2_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_expected_api():
    assert set(header_functions()) == set(fa2.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    names = {0: "FA2_OK", 1: "FA2_ERR_INVALID_ARG", 2: "FA2_ERR_UNSUPPORTED",
             3: "FA2_ERR_CUDA", 4: "FA2_ERR_TIMEOUT", 5: "FA2_ERR_BOUNDS"}
    for code, name in names.items():
        assert fa2.status_string(code) == name
    assert fa2.status_string(99) == "FA2_ERR_UNKNOWN"
    assert fa2.fa2_version().startswith("fa2-sm103a")


A = 1 << 20  # a 16-byte aligned fake address: never dereferenced on these paths


@pytest.mark.parametrize("args,expected", [
    # (q, k, v, o, lse, B, Hq, Hkv, N, d, scale, dtype)
    ((0, A, A, A, A, 1, 1, 1, 128, 128, 0.1, 0), fa2.FA2_ERR_INVALID_ARG),   # NULL q
    ((A, A, A, A, 0, 1, 1, 1, 128, 128, 0.1, 0), fa2.FA2_ERR_INVALID_ARG),   # NULL lse
    ((A + 8, A, A, A, A, 1, 1, 1, 128, 128, 0.1, 0), fa2.FA2_ERR_INVALID_ARG),  # misaligned
    ((A, A, A, A, A + 4, 1, 1, 1, 128, 128, 0.1, 0), fa2.FA2_ERR_INVALID_ARG),  # misaligned lse
    ((A, A, A, A, A, 0, 1, 1, 128, 128, 0.1, 0), fa2.FA2_ERR_INVALID_ARG),   # B = 0
    ((A, A, A, A, A, 1, -2, 1, 128, 128, 0.1, 0), fa2.FA2_ERR_INVALID_ARG),  # Hq < 0
    ((A, A, A, A, A, 1, 1, 1, 0, 128, 0.1, 0), fa2.FA2_ERR_INVALID_ARG),     # N = 0
    ((A, A, A, A, A, 1, 6, 4, 128, 128, 0.1, 0), fa2.FA2_ERR_INVALID_ARG),   # Hq % Hkv
    ((A, A, A, A, A, 1, 1, 1, 128, 128, 0.0, 0), fa2.FA2_ERR_INVALID_ARG),   # scale = 0
    ((A, A, A, A, A, 1, 1, 1, 128, 128, -1.0, 0), fa2.FA2_ERR_INVALID_ARG),  # scale < 0
    ((A, A, A, A, A, 1, 1, 1, 128, 128, float("nan"), 0), fa2.FA2_ERR_INVALID_ARG),
    ((A, A, A, A, A, 1, 1, 1, 128, 128, float("inf"), 0), fa2.FA2_ERR_INVALID_ARG),
    ((A, A, A, A, A, 1, 1, 1, 128, 128, 0.1, 7), fa2.FA2_ERR_INVALID_ARG),   # dtype
    ((A, A, A, A, A, 1, 1, 1, 128, 96, 0.1, 0), fa2.FA2_ERR_UNSUPPORTED),    # d = 96
    ((A, A, A, A, A, 1, 1, 1, 128, 256, 0.1, 0), fa2.FA2_ERR_UNSUPPORTED),   # d = 256
    ((A, A, A, A, A, 1, 1, 1, 200, 128, 0.1, 0), fa2.FA2_ERR_UNSUPPORTED),   # N % 128
    ((A, A, A, A, A, 1, 1, 1, 64, 64, 0.1, 1), fa2.FA2_ERR_UNSUPPORTED),     # N < block
    ((A, A, A, A, A, 2048, 8, 8, 131072, 128, 0.1, 0), fa2.FA2_ERR_UNSUPPORTED),  # rows >= 2^31
])
def test_host_validation(lib, args, expected):
    assert fa2.fa2_fwd_gqa_ptr(*args) == expected


@pytest.mark.parametrize("args,expected", [
    # (q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, dtype)
    ((0, A, A, A, A, 1, 1, 1, 100, 70, 128, 0.1, 1, 0), fa2.FA2_ERR_INVALID_ARG),   # NULL q
    ((A, A, A, A, A + 4, 1, 1, 1, 100, 70, 128, 0.1, 1, 0), fa2.FA2_ERR_INVALID_ARG),  # lse align
    ((A, A, A, A, A, 1, 1, 1, 0, 70, 128, 0.1, 1, 0), fa2.FA2_ERR_INVALID_ARG),     # Nq = 0
    ((A, A, A, A, A, 1, 1, 1, 100, 0, 128, 0.1, 1, 0), fa2.FA2_ERR_INVALID_ARG),    # Nk = 0
    ((A, A, A, A, A, 1, 3, 2, 100, 70, 128, 0.1, 0, 0), fa2.FA2_ERR_INVALID_ARG),   # Hq % Hkv
    ((A, A, A, A, A, 1, 1, 1, 100, 70, 128, 0.1, 2, 0), fa2.FA2_ERR_INVALID_ARG),   # causal = 2
    ((A, A, A, A, A, 1, 1, 1, 100, 70, 128, -0.1, 1, 0), fa2.FA2_ERR_INVALID_ARG),  # scale
    ((A, A, A, A, A, 1, 1, 1, 100, 70, 96, 0.1, 1, 0), fa2.FA2_ERR_UNSUPPORTED),    # d = 96
    ((A, A, A, A, A, 1, 1, 1, 100, 70, 128, 0.1, 1, 5), fa2.FA2_ERR_INVALID_ARG),   # dtype
    ((A, A, A, A, A, 4096, 8, 8, 65537, 7, 64, 0.1, 0, 0), fa2.FA2_ERR_UNSUPPORTED),  # rows >= 2^31
])
def test_general_entry_host_validation(lib, args, expected):
    assert fa2.fa2_fwd_ex_ptr(*args) == expected


def test_backward_host_validation(lib):
    f = fa2.fa2_bwd_ptr
    ok = [A] * 10
    assert f(*([0] + ok[1:]), 1, 1, 1, 128, 128, 0.1, 0, 0) == fa2.FA2_ERR_INVALID_ARG   # NULL q
    assert f(*(ok[:9] + [A + 4]), 1, 1, 1, 128, 128, 0.1, 0, 0) == fa2.FA2_ERR_INVALID_ARG  # delta align
    assert f(*ok, 1, 1, 1, 128, 128, 0.1, 3, 0) == fa2.FA2_ERR_INVALID_ARG          # causal
    assert f(*ok, 1, 3, 2, 128, 128, 0.1, 0, 0) == fa2.FA2_ERR_INVALID_ARG          # Hq % Hkv
    assert f(*ok, 1, 1, 1, 128, 80, 0.1, 0, 0) == fa2.FA2_ERR_UNSUPPORTED           # d
    assert f(*ok, 1, 70000, 1, 128, 64, 0.1, 0, 0) == fa2.FA2_ERR_UNSUPPORTED       # B*Hq > 65535


def test_backward_noalloc_checks_arguments_before_size_and_device(lib):
    """fa2_bwd_noalloc runs fa2_bwd's argument checks before its own row limit
    and before any device call, so the same bad argument gives the same
    error, whatever the size (no GPU is touched on these paths)."""
    f = fa2.fa2_bwd_noalloc_ptr
    ok = [A] * 9
    big = (64, 32, 32, 1024)     # B*H_q*N = 2^21 query rows: past the fixed array
    assert f(*([0] + ok[1:]), *big, 128, 0.1, 0, 0) == fa2.FA2_ERR_INVALID_ARG     # NULL q, too many rows
    assert f(*(ok[:8] + [0]), *big, 128, 0.1, 0, 0) == fa2.FA2_ERR_INVALID_ARG     # NULL dv, too many rows
    assert f(*(ok[:4] + [A + 4] + ok[5:]), *big, 128, 0.1, 0, 0) == fa2.FA2_ERR_INVALID_ARG  # lse misaligned
    assert f(*ok, 64, 32, 24, 1024, 128, 0.1, 0, 0) == fa2.FA2_ERR_INVALID_ARG     # H_q % H_kv, too many rows
    assert f(*ok, 1, 3, 2, 128, 128, 0.1, 0, 0) == fa2.FA2_ERR_INVALID_ARG         # H_q % H_kv
    assert f(*ok, *big, 128, 0.1, 2, 0) == fa2.FA2_ERR_INVALID_ARG                 # causal = 2
    assert f(*ok, *big, 128, float("inf"), 0, 0) == fa2.FA2_ERR_INVALID_ARG        # scale
    assert f(*ok, *big, 128, 0.1, 0, 7) == fa2.FA2_ERR_INVALID_ARG                 # dtype
    assert f(*ok, *big, 96, 0.1, 0, 0) == fa2.FA2_ERR_UNSUPPORTED                  # d, before the row limit
    assert f(*ok, 1, 70000, 1, 128, 64, 0.1, 0, 0) == fa2.FA2_ERR_UNSUPPORTED      # B*H_q > 65535
    # and every one of them matches fa2_bwd with a valid workspace pointer
    for args in (([0] + ok[1:], big), (ok, (64, 32, 24, 1024))):
        assert (fa2.fa2_bwd_ptr(*args[0], A, *args[1], 128, 0.1, 0, 0)
                == f(*args[0], *args[1], 128, 0.1, 0, 0))


def test_fp8_entry_host_validation(lib):
    f = fa2.fa2_fwd_fp8_ptr
    ok = [A] * 8            # q, k, v, q/k/v descales, o, lse
    assert f(*([0] + ok[1:]), 1, 1, 1, 128, 128, 0.1) == fa2.FA2_ERR_INVALID_ARG         # NULL q
    assert f(*(ok[:4] + [0] + ok[5:]), 1, 1, 1, 128, 128, 0.1) == fa2.FA2_ERR_INVALID_ARG  # NULL k_descale
    assert f(*(ok[:3] + [A + 2] + ok[4:]), 1, 1, 1, 128, 128, 0.1) == fa2.FA2_ERR_INVALID_ARG  # descale align
    assert f(*(ok[:7] + [A + 4]), 1, 1, 1, 128, 128, 0.1) == fa2.FA2_ERR_INVALID_ARG      # lse align
    assert f(*ok, 1, 3, 2, 128, 128, 0.1) == fa2.FA2_ERR_INVALID_ARG                      # Hq % Hkv
    assert f(*ok, 1, 1, 1, 128, 128, 0.0) == fa2.FA2_ERR_INVALID_ARG                      # scale
    assert f(*ok, 1, 1, 1, 0, 128, 0.1) == fa2.FA2_ERR_INVALID_ARG                        # N = 0
    assert f(*ok, 1, 1, 1, 128, 64, 0.1) == fa2.FA2_ERR_UNSUPPORTED                       # d = 64
    assert f(*ok, 1, 1, 1, 200, 128, 0.1) == fa2.FA2_ERR_UNSUPPORTED                      # N % 128
    assert f(*ok, 2048, 8, 8, 131072, 128, 0.1) == fa2.FA2_ERR_UNSUPPORTED                # rows >= 2^31


def test_fp8_general_entry_host_validation(lib):
    f = fa2.fa2_fwd_fp8_ex_ptr
    ok = [A] * 8
    assert f(*([0] + ok[1:]), 1, 1, 1, 100, 100, 128, 0.1, 1) == fa2.FA2_ERR_INVALID_ARG        # NULL q
    assert f(*(ok[:5] + [0] + ok[6:]), 1, 1, 1, 100, 100, 128, 0.1, 1) == fa2.FA2_ERR_INVALID_ARG  # NULL v_descale
    assert f(*(ok[:5] + [A + 1] + ok[6:]), 1, 1, 1, 100, 100, 128, 0.1, 1) == fa2.FA2_ERR_INVALID_ARG  # align
    assert f(*(ok[:6] + [A + 8, A]), 1, 1, 1, 100, 100, 128, 0.1, 1) == fa2.FA2_ERR_INVALID_ARG  # o align
    assert f(*ok, 1, 4, 3, 100, 100, 128, 0.1, 1) == fa2.FA2_ERR_INVALID_ARG                    # Hq % Hkv
    assert f(*ok, 1, 1, 1, 0, 100, 128, 0.1, 1) == fa2.FA2_ERR_INVALID_ARG                      # N_q = 0
    assert f(*ok, 1, 1, 1, 100, 0, 128, 0.1, 0) == fa2.FA2_ERR_INVALID_ARG                      # N_k = 0
    assert f(*ok, 1, 1, 1, 100, 100, 128, 0.1, 2) == fa2.FA2_ERR_INVALID_ARG                    # causal = 2
    assert f(*ok, 1, 1, 1, 100, 100, 128, float("nan"), 1) == fa2.FA2_ERR_INVALID_ARG           # scale
    assert f(*ok, 1, 1, 1, 100, 100, 64, 0.1, 1) == fa2.FA2_ERR_UNSUPPORTED                     # d = 64
    assert f(*ok, 4096, 8, 8, 65536, 100, 128, 0.1, 1) == fa2.FA2_ERR_UNSUPPORTED               # rows >= 2^31
    # equal lengths, multiple of 128, no mask: forwarded to fa2_fwd_fp8 and its checks
    assert f(*ok, 2048, 8, 8, 131072, 131072, 128, 0.1, 0) == fa2.FA2_ERR_UNSUPPORTED


def test_mha_entry_forwards_to_gqa(lib):
    assert fa2.fa2_fwd_ptr(0, A, A, A, A, 1, 1, 128, 128, 0.1, 0) == fa2.FA2_ERR_INVALID_ARG
    assert fa2.fa2_fwd_ptr(A, A, A, A, A, 1, 1, 128, 80, 0.1, 0) == fa2.FA2_ERR_UNSUPPORTED


def test_wait_limit_and_debug_flags_round_trip(lib):
    prev = fa2.fa2_set_wait_limit_ns(12345)
    assert fa2.fa2_set_wait_limit_ns(prev) == 12345
    assert fa2.fa2_set_wait_limit_ns(0) == prev  # <= 0 restores the default
    fa2.fa2_set_wait_limit_ns(prev)
    old = fa2.fa2_set_debug_flags(1)
    assert fa2.fa2_set_debug_flags(old) == 1


def test_tile_config_round_trip(lib):
    prev = fa2.fa2_set_tile_config(fa2.TILE_CFG_D64_SHARED)
    assert prev in (0, fa2.TILE_CFG_D64_SHARED)
    assert fa2.fa2_set_tile_config(prev) == fa2.TILE_CFG_D64_SHARED
    assert fa2.fa2_set_tile_config(2) == -1          # unknown bit: rejected, unchanged
    assert fa2.fa2_set_tile_config(-1) == -1
    assert fa2.fa2_set_tile_config(prev) == prev


def test_tile_config_read_from_environment(tmp_path):
    """A fresh process picks FA2_TILE_CFG up on its first call."""
    import os
    import subprocess
    import sys

    code = ("from attention_fa2_forward_03_gb300 import fa2; "
            "print(fa2.fa2_set_tile_config(0))")
    for env_value, want in (("d64=shared", "1"), ("d64=split", "0"), (None, "0")):
        env = dict(os.environ)
        env.pop("FA2_TILE_CFG", None)
        if env_value is not None:
            env["FA2_TILE_CFG"] = env_value
        out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                             cwd=os.path.dirname(os.path.dirname(os.path.abspath(__file__))), timeout=120)
        assert out.returncode == 0, out.stderr
        assert out.stdout.strip().splitlines()[-1] == want


def test_binding_refuses_missing_library(tmp_path):
    saved = fa2._lib
    fa2._lib = None
    try:
        with pytest.raises(ImportError):
            fa2.load(str(tmp_path / "absent.so"))
    finally:
        fa2._lib = saved


def test_debug_library_exports_the_same_symbols(lib):
    """libfa2_debug.so (FA2_DEBUG: device-side bounds checks) is built beside
    the release library, exports the same calls and says which it is."""
    dbg = ctypes.CDLL(build.DEBUG_LIB)
    for name in header_functions():
        assert hasattr(dbg, name), name
    dbg.fa2_version.restype = ctypes.c_char_p
    assert dbg.fa2_version().decode().endswith("debug")
    assert not fa2.fa2_version().endswith("debug")
    dbg.fa2_status_string.restype = ctypes.c_char_p
    assert dbg.fa2_status_string(5).decode() == "FA2_ERR_BOUNDS"

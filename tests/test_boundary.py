"""The C ABI library without a GPU: it builds, loads, exports every function
include/attn.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import warp_specialized_gb300 as ws

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    return ws.load_library(build_if_missing=True)


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+|unsigned\s+|long\s+)*\w+\s*\*?\s*(attn_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert names == sorted(ws.EXPORTED_SYMBOLS), names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in ws.STATUS_NAMES.items():
        assert ws.attn_status_string(code) == name
    assert ws.attn_status_string(99) == "ATTN_ERR_UNKNOWN"


# Fake but aligned addresses: every call below fails an argument check, and
# the checks run before anything reads memory or calls CUDA.
A = 1 << 20


def _call(lib, q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=128, scale=0.1, causal=0,
          dtype=ws.ATTN_BF16):
    return lib.attn_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, None)


@pytest.mark.parametrize("kw,code", [
    ({"q": 0}, 1), ({"k": 0}, 1), ({"v": 0}, 1), ({"o": 0}, 1), ({"lse": 0}, 1),
    ({"B": 0}, 1), ({"H": -1}, 1), ({"N": 0}, 1), ({"d": 0}, 1),
    ({"N": (1 << 24) + 1}, 1), ({"B": 1 << 13, "H": 1 << 12}, 1),
    ({"B": 1 << 12, "H": 1 << 10, "N": 1 << 12}, 1),
    ({"scale": 0.0}, 1), ({"scale": -1.0}, 1), ({"scale": float("inf")}, 1),
    ({"scale": float("nan")}, 1), ({"causal": 2}, 1), ({"dtype": 4}, 1), ({"dtype": -1}, 1),
    ({"d": 96}, 2), ({"d": 32}, 2), ({"d": 512}, 2),
    ({"d": 256, "dtype": ws.ATTN_FP32}, 2), ({"d": 64, "dtype": ws.ATTN_FP8_E4M3}, 2),
    ({"q": A + 8}, 3), ({"k": A + 4}, 3), ({"v": A + 2}, 3), ({"o": A + 1}, 3), ({"lse": A + 2}, 3),
])
def test_bad_arguments_are_rejected(lib, kw, code):
    assert _call(lib, **kw) == code


def test_fp8_descales_are_checked(lib):
    f = lib.attn_fwd_fp8
    assert f(A, A, A, A, A, 1, 1, 128, 128, 0.1, 0, 0.0, 1.0, 1.0, None) == 1
    assert f(A, A, A, A, A, 1, 1, 128, 128, 0.1, 0, 1.0, float("nan"), 1.0, None) == 1
    assert f(A, A, A, A, A, 1, 1, 128, 128, 0.1, 0, 1.0, 1.0, -2.0, None) == 1
    assert f(A, A, A, A, A, 1, 1, 128, 64, 0.1, 0, 1.0, 1.0, 1.0, None) == 2


def test_watchdog_selftest_checks_its_limit(lib):
    assert lib.attn_watchdog_selftest(0, None) == 1
    assert lib.attn_watchdog_selftest(10_000_001, None) == 1


def test_no_device_is_reported():
    """Valid arguments on a machine without a CUDA device: ATTN_ERR_DEVICE,
    and nothing is launched.  (Only runs where no GPU is visible.)"""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    lib = ws.load_library(build_if_missing=True)
    assert _call(lib) == 4
    assert lib.attn_fwd_status(None) == 4


def test_bwd_workspace_size(lib):
    assert lib.attn_bwd_workspace_size(2, 3, 200) == 2 * 3 * 256 * 8
    assert lib.attn_bwd_workspace_size(1, 1, 128) == 128 * 8
    assert lib.attn_bwd_workspace_size(0, 1, 128) == 0


def _bwd(lib, q=A, k=A, v=A, o=A, do=A, lse=A, dq=A, dk=A, dv=A, ws=A, wsb=1 << 20, B=1, H=1,
         N=128, d=128, scale=0.1, causal=0, dtype=2):
    return lib.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, wsb, B, H, N, d, scale, causal,
                        dtype, None)


@pytest.mark.parametrize("kw,code", [
    ({"o": 0}, 1), ({"do": 0}, 1), ({"dq": 0}, 1), ({"dk": 0}, 1), ({"dv": 0}, 1), ({"ws": 0}, 1),
    ({"q": 0}, 1), ({"lse": 0}, 1), ({"N": 0}, 1), ({"scale": 0.0}, 1), ({"causal": 3}, 1),
    ({"wsb": 128 * 8 - 1}, 1), ({"dtype": 0}, 2), ({"dtype": 3}, 2), ({"dtype": 7}, 1),
    ({"d": 256}, 2), ({"d": 96}, 2),
    ({"o": A + 8}, 3), ({"do": A + 2}, 3), ({"dk": A + 4}, 3), ({"dv": A + 1}, 3),
    ({"ws": A + 8}, 3), ({"dq": A + 8}, 3),
])
def test_bwd_bad_arguments_are_rejected(lib, kw, code):
    assert _bwd(lib, **kw) == code


def _quant(lib, x=A, codes=A, scales=A, B=1, H=1, N=128, d=128, dtype=ws.ATTN_BF16, hadamard=1):
    return lib.attn_quantize_fp8(x, codes, scales, B, H, N, d, dtype, hadamard, None)


@pytest.mark.parametrize("kw,code", [
    ({"x": 0}, 1), ({"codes": 0}, 1), ({"scales": 0}, 1), ({"B": 0}, 1), ({"N": -3}, 1),
    ({"hadamard": 2}, 1), ({"dtype": 9}, 1), ({"dtype": ws.ATTN_FP8_E4M3}, 2), ({"d": 256}, 2),
    ({"d": 96}, 2), ({"x": A + 8}, 3), ({"codes": A + 4}, 3), ({"scales": A + 2}, 3),
])
def test_quantize_bad_arguments_are_rejected(lib, kw, code):
    assert _quant(lib, **kw) == code


def test_blockscaled_fwd_checks_its_scales(lib):
    f = lib.attn_fwd_fp8_blockscaled
    assert f(A, A, A, A, A, 1, 1, 128, 128, 0.1, 0, 0, A, 1.0, None) == 1
    assert f(A, A, A, A, A, 1, 1, 128, 128, 0.1, 0, A, 0, 1.0, None) == 1
    assert f(A, A, A, A, A, 1, 1, 128, 128, 0.1, 0, A + 2, A, 1.0, None) == 3
    assert f(A, A, A, A, A, 1, 1, 128, 128, 0.1, 0, A, A, 0.0, None) == 1
    assert f(A, A, A, A, A, 1, 1, 128, 64, 0.1, 0, A, A, 1.0, None) == 2

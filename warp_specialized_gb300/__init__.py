"""Python binding of libattn_sm103.so, the GB300 (sm_103a) fused attention
forward library.

Argument marshalling only: every step of the computation runs in the CUDA
library.  The functions take torch CUDA tensors for convenience (torch is
used for device memory and streams) and pass raw device pointers through the
C ABI of include/attn.h.  There is no fallback: if the library is missing or
the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "ATTN_FP32", "ATTN_FP16", "ATTN_BF16", "ATTN_FP8_E4M3", "AttnError", "lib_path",
    "load_library", "attn_fwd", "attn_fwd_fp8", "attn_fwd_status", "attn_status_string",
    "attn_watchdog_selftest", "attn_fwd_raw", "attn_bwd", "attn_bwd_workspace_size",
    "attn_bwd_noalloc", "attn_fwd_fp8_blockscaled", "attn_quantize_fp8", "EXPORTED_SYMBOLS",
    "attn_fwd_workspace_size", "attn_fwd_ws_raw", "attn_fwd_split_advised", "attn_fwd_opt_raw",
    "ATTN_OPT_EXP2_FMA",
]

ATTN_FP32, ATTN_FP16, ATTN_BF16, ATTN_FP8_E4M3 = 0, 1, 2, 3
ATTN_OPT_EXP2_FMA = 1  # a share of the exponentials on the FMA pipe (attn_fwd_opt)

STATUS_NAMES = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
    3: "ATTN_ERR_MISALIGNED", 4: "ATTN_ERR_DEVICE", 5: "ATTN_ERR_CUDA", 6: "ATTN_ERR_TIMEOUT",
}

EXPORTED_SYMBOLS = ("attn_fwd", "attn_fwd_fp8", "attn_fwd_status", "attn_status_string",
                    "attn_watchdog_selftest", "attn_bwd", "attn_bwd_workspace_size",
                    "attn_bwd_noalloc", "attn_fwd_fp8_blockscaled", "attn_quantize_fp8",
                    "attn_fwd_workspace_size", "attn_fwd_ws", "attn_fwd_fp8_ws",
                    "attn_fwd_split_advised", "attn_fwd_opt", "attn_fwd_fp8_opt")

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = "attn_fwd"):
        self.status = int(status)
        super().__init__(f"{what} failed: {STATUS_NAMES.get(self.status, self.status)}")


def lib_path() -> str:
    return os.path.join(_HERE, "_build", "libattn_sm103.so")


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load the shared library (optionally building it first)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if build_if_missing:
            from . import build as _build
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m warp_specialized_gb300.build` "
                "(there is no fallback implementation)")
        lib = ctypes.CDLL(path)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
        lib.attn_fwd.restype = i
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, f, f, f, vp]
        lib.attn_fwd_fp8.restype = i
        u64 = ctypes.c_ulonglong
        lib.attn_fwd_workspace_size.argtypes = [i, i]
        lib.attn_fwd_workspace_size.restype = u64
        lib.attn_fwd_ws.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, u64, vp]
        lib.attn_fwd_ws.restype = i
        lib.attn_fwd_fp8_ws.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, f, f, f, vp, u64,
                                        vp]
        lib.attn_fwd_fp8_ws.restype = i
        lib.attn_fwd_opt.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, ctypes.c_uint, vp]
        lib.attn_fwd_opt.restype = i
        lib.attn_fwd_fp8_opt.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, f, f, f,
                                         ctypes.c_uint, vp]
        lib.attn_fwd_fp8_opt.restype = i
        lib.attn_fwd_split_advised.argtypes = [i, i, i, i, i, i]
        lib.attn_fwd_split_advised.restype = i
        lib.attn_fwd_status.argtypes = [vp]
        lib.attn_fwd_status.restype = i
        lib.attn_status_string.argtypes = [i]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_watchdog_selftest.argtypes = [ctypes.c_uint, vp]
        lib.attn_watchdog_selftest.restype = i
        lib.attn_bwd_workspace_size.argtypes = [i, i, i]
        lib.attn_bwd_workspace_size.restype = u64
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, u64, i, i, i, i, f, i, i,
                                 vp]
        lib.attn_bwd.restype = i
        lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i,
                                         vp]
        lib.attn_bwd_noalloc.restype = i
        lib.attn_fwd_fp8_blockscaled.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp, f,
                                                 vp]
        lib.attn_fwd_fp8_blockscaled.restype = i
        lib.attn_quantize_fp8.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp]
        lib.attn_quantize_fp8.restype = i
        _lib = lib
        return lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _dtype_code(t):
    import torch
    codes = {torch.float32: ATTN_FP32, torch.float16: ATTN_FP16, torch.bfloat16: ATTN_BF16,
             torch.float8_e4m3fn: ATTN_FP8_E4M3}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def attn_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int, H: int,
                 N: int, d: int, scale: float, causal: bool, dtype: int, stream: int = 0) -> int:
    """The C call with raw device pointers; returns the status code."""
    return load_library().attn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d,
                                   float(scale), int(bool(causal)), int(dtype), stream)


def attn_fwd_ws_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int,
                    H: int, N: int, d: int, scale: float, causal: bool, dtype: int, ws_ptr: int,
                    ws_bytes: int, stream: int = 0) -> int:
    """attn_fwd_ws with raw device pointers; returns the status code."""
    return load_library().attn_fwd_ws(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d,
                                      float(scale), int(bool(causal)), int(dtype), ws_ptr,
                                      int(ws_bytes), stream)


def attn_fwd_opt_raw(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int, B: int,
                     H: int, N: int, d: int, scale: float, causal: bool, dtype: int, opts: int,
                     stream: int = 0) -> int:
    """attn_fwd_opt with raw device pointers; returns the status code."""
    return load_library().attn_fwd_opt(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d,
                                       float(scale), int(bool(causal)), int(dtype), int(opts),
                                       stream)


def attn_fwd_workspace_size(d: int, dtype: int) -> int:
    """Bytes of workspace the forward's tail launch needs on the current device."""
    return int(load_library().attn_fwd_workspace_size(int(d), int(dtype)))


def attn_fwd_split_advised(B: int, H: int, N: int, d: int, causal: bool, dtype: int) -> bool:
    """Whether splitting the leftover work (attn_fwd_ws) pays for this shape."""
    return bool(load_library().attn_fwd_split_advised(int(B), int(H), int(N), int(d),
                                                      int(bool(causal)), int(dtype)))


def _use_split(split_tail, workspace, stream, B, H, N, d, causal, code):
    if split_tail is False or (workspace is None and isinstance(stream, int)):
        return False
    if split_tail is None:
        return attn_fwd_split_advised(B, H, N, d, causal, code)
    return True


def _workspace(d, code, device, stream, workspace):
    """The caller's workspace, else a fresh one from torch's allocator on the
    stream the call runs on (so the allocator does not hand the memory to
    another stream while the kernels still use it)."""
    import torch
    if workspace is not None:
        if workspace.device != device or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on the inputs' device")
        return workspace
    size = attn_fwd_workspace_size(d, code)
    if size == 0:
        return None
    if stream is None:
        return torch.empty(size, dtype=torch.uint8, device=device)
    with torch.cuda.stream(stream):
        return torch.empty(size, dtype=torch.uint8, device=device)


def _check_qkv(q, k, v):
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share one dtype")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")


def attn_fwd(q, k, v, scale=None, causal: bool = False, out=None, lse=None, stream=None,
             split_tail=None, workspace=None, exp2_fma: bool = False):
    """O, LSE = attention forward of [B, H, N, d] CUDA tensors.

    scale defaults to 1/sqrt(d).  out / lse may be given preallocated
    ([B, H, N, d] of q's dtype, [B, H, N] fp32).  Asynchronous on `stream`
    (default: torch's current stream).  split_tail: True splits the work
    left after whole rounds of one item per SM along the keys over the SMs
    (attn_fwd_ws), False never does, None (default) does where
    attn_fwd_split_advised says it pays; the split uses a uint8 `workspace`
    of at least attn_fwd_workspace_size(d, dtype) bytes, else one allocated
    here.  exp2_fma: ATTN_OPT_EXP2_FMA (attn_fwd_opt; bf16 d = 64 / 128, no
    split).  Returns (out, lse)."""
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    code = _dtype_code(q)
    out_dtype = torch.bfloat16 if code == ATTN_FP8_E4M3 else q.dtype
    if out is None:
        out = torch.empty((B, H, N, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    ws = None
    if not exp2_fma and _use_split(split_tail, workspace, stream, B, H, N, d, causal, code):
        ws = _workspace(d, code, q.device, stream, workspace)
    if exp2_fma:
        st = attn_fwd_opt_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), B, H, N, d, scale, causal, code,
                              ATTN_OPT_EXP2_FMA, _stream_handle(stream))
    elif ws is None:
        st = attn_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr(), B, H, N, d, scale, causal, code, _stream_handle(stream))
    else:
        st = attn_fwd_ws_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             lse.data_ptr(), B, H, N, d, scale, causal, code, ws.data_ptr(),
                             ws.numel(), _stream_handle(stream))
    if st != 0:
        raise AttnError(st)
    return out, lse


def attn_fwd_fp8(q, k, v, q_descale: float, k_descale: float, v_descale: float, scale=None,
                 causal: bool = False, out=None, lse=None, stream=None, split_tail=None,
                 workspace=None, exp2_fma: bool = False):
    """Forward pass on e4m3 tensors with per-tensor descales; O is bf16.
    split_tail, workspace and exp2_fma as in attn_fwd (exp2_fma: d = 128)."""
    import torch
    _check_qkv(q, k, v)
    if q.dtype != torch.float8_e4m3fn:
        raise TypeError("attn_fwd_fp8 takes float8_e4m3fn tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    lib = load_library()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, d,
            float(scale), int(bool(causal)), float(q_descale), float(k_descale), float(v_descale))
    ws = None
    if not exp2_fma and _use_split(split_tail, workspace, stream, B, H, N, d, causal,
                                   ATTN_FP8_E4M3):
        ws = _workspace(d, ATTN_FP8_E4M3, q.device, stream, workspace)
    if exp2_fma:
        st = lib.attn_fwd_fp8_opt(*args, ATTN_OPT_EXP2_FMA, _stream_handle(stream))
    elif ws is None:
        st = lib.attn_fwd_fp8(*args, _stream_handle(stream))
    else:
        st = lib.attn_fwd_fp8_ws(*args, ws.data_ptr(), ws.numel(), _stream_handle(stream))
    if st != 0:
        raise AttnError(st, "attn_fwd_fp8")
    return out, lse


def attn_fwd_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device watchdog status."""
    return int(load_library().attn_fwd_status(_stream_handle(stream)))


def attn_watchdog_selftest(timeout_us: int = 2000, stream=None) -> int:
    """Run the watchdog self-test kernel; returns ATTN_ERR_TIMEOUT (6) when the
    bounded wait works."""
    return int(load_library().attn_watchdog_selftest(int(timeout_us), _stream_handle(stream)))


def attn_bwd_workspace_size(B: int, H: int, N: int) -> int:
    """Bytes of device workspace attn_bwd needs for this shape."""
    return int(load_library().attn_bwd_workspace_size(int(B), int(H), int(N)))


def attn_bwd(q, k, v, o, lse, dout, scale=None, causal: bool = False, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """dQ, dK, dV of the forward pass for the output gradient dout.

    q, k, v, o, dout: [B, H, N, d] fp16/bf16 CUDA tensors (o, lse from
    attn_fwd with the same scale and mask); lse: [B, H, N] fp32.  Outputs
    and the uint8 workspace are allocated with torch when not given.
    Asynchronous on `stream`.  Returns (dq, dk, dv)."""
    import torch
    _check_qkv(q, k, v)
    for t in (o, dout):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError("o and dout must match q")
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    code = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    need = attn_bwd_workspace_size(B, H, N)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = load_library().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), B, H, N, d,
                                 float(scale), int(bool(causal)), code, _stream_handle(stream))
    if st != 0:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def attn_bwd_noalloc(q, k, v, o, lse, dout, scale=None, causal: bool = False, dq=None, dk=None,
                     dv=None, stream=None):
    """attn_bwd without a caller workspace: the library's own device array
    serves as scratch (see include/attn.h for its size limit and for why
    calls that overlap on the device must be ordered).  Returns (dq, dk, dv)."""
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    st = load_library().attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         dout.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                         dk.data_ptr(), dv.data_ptr(), B, H, N, d, float(scale),
                                         int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    if st != 0:
        raise AttnError(st, "attn_bwd_noalloc")
    return dq, dk, dv


def attn_quantize_fp8(x, hadamard: bool = True, codes=None, scales=None, stream=None):
    """e4m3 codes and per-128-row-block scales of a [B, H, N, d] CUDA tensor
    (optionally after the 16 x 16 Walsh-Hadamard rotation of each group of
    16 channels).  Returns (codes: float8_e4m3fn, scales: fp32 [B, H, nt])."""
    import torch
    if x.dim() != 4 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous [B, H, N, d] CUDA tensor")
    B, H, N, d = x.shape
    nt = (N + 127) // 128
    codes = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device) if codes is None else codes
    scales = torch.empty((B, H, nt), dtype=torch.float32, device=x.device) if scales is None else scales
    st = load_library().attn_quantize_fp8(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), B, H,
                                          N, d, _dtype_code(x), int(bool(hadamard)),
                                          _stream_handle(stream))
    if st != 0:
        raise AttnError(st, "attn_quantize_fp8")
    return codes, scales


def attn_fwd_fp8_blockscaled(q, k, v, q_scales, k_scales, v_descale: float, scale=None,
                             causal: bool = False, out=None, lse=None, stream=None):
    """Forward pass on e4m3 Q, K with per-128-row-block scales ([B, H, nt]
    fp32 CUDA tensors, as attn_quantize_fp8 returns them) and e4m3 V with a
    per-tensor descale.  O is bf16."""
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = load_library().attn_fwd_fp8_blockscaled(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                 out.data_ptr(), lse.data_ptr(), B, H, N, d,
                                                 float(scale), int(bool(causal)),
                                                 q_scales.data_ptr(), k_scales.data_ptr(),
                                                 float(v_descale), _stream_handle(stream))
    if st != 0:
        raise AttnError(st, "attn_fwd_fp8_blockscaled")
    return out, lse

"""fp64 CPU oracle for the fused attention forward pass.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``.  The product library never imports,
links or calls anything here, and nothing here imports the product package.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64); this module only
compiles it with gcc and marshals numpy arrays through ctypes.  See the C
file's header for what is computed and which passage of the pages it follows
("Warp specialization" concept card, section "Implementation sketch").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into a shared library (OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                            ctypes.c_double, ctypes.c_int,
                                            ctypes.POINTER(i64), i64, ctypes.c_int]
            lib.oracle_attn_fwd.restype = ctypes.c_int
            lib.oracle_attn_fwd_blockwise.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64,
                                                      i64, ctypes.c_double, ctypes.c_int,
                                                      i64]
            lib.oracle_attn_fwd_blockwise.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64,
                                            ctypes.c_double, ctypes.c_int, ctypes.c_int]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    """Threads the oracle's parallel loop uses by default."""
    return int(_load().oracle_max_threads())


def attn_fwd(q, k, v, scale: float, causal: bool, rows=None, n_threads: int = 0):
    """Direct-form oracle.

    q, k, v: array-likes of shape [B, H, N, d] (converted to fp64).
    rows: None for every query row, else a 1-D list of row indices computed
    for every (b, h).  Returns (O [B, H, R, d], LSE [B, H, R]) as fp64 numpy
    arrays, R = N or len(rows).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    if rows is None:
        R, rows_p = N, None
    else:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        R = int(rows_a.size)
        rows_p = rows_a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    o = np.empty((B, H, R, d), dtype=np.float64)
    lse = np.empty((B, H, R), dtype=np.float64)
    rc = _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 B, H, N, d, float(scale), int(bool(causal)),
                                 rows_p, R, int(n_threads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return o, lse


def attn_fwd_blockwise(q, k, v, scale: float, causal: bool, block: int):
    """The blockwise online-softmax recurrence, key blocks of `block` keys.
    Same shapes as attn_fwd (every row)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = q.shape
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attn_fwd_blockwise(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                           B, H, N, d, float(scale), int(bool(causal)),
                                           int(block))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_blockwise rejected its arguments")
    return o, lse


def attn_bwd(q, k, v, dout, scale: float, causal: bool, n_threads: int = 0):
    """Gradients (dQ, dK, dV) of the forward pass for the output gradient
    dout, every row, fp64.  Shapes [B, H, N, d]."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    if q.ndim != 4 or any(x.shape != q.shape for x in (k, v, dout)):
        raise ValueError("q, k, v, dout must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    dq, dk, dv = (np.empty_like(q) for _ in range(3))
    rc = _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                                 int(n_threads))
    if rc != 0:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    return dq, dk, dv


# ---------------------------------------------------------------------------
# FP8 block quantisation with the 16 x 16 Walsh-Hadamard rotation
# ("Inside FlashAttention-3 & Warp-Specialized CUDA Kernels", section 5:
# rotate Q and K by an orthogonal Hadamard transform, Q' = Q H, K' = K H, so
# that Q' K'^T = Q K^T while outlier channels are spread out, then quantise
# to e4m3 with a scale per block).  The pages fix neither the block nor the
# order of the transform's additions; the readings taken (and implemented
# identically on the GPU, so that codes match bit for bit):
#   - the transform acts on each group of 16 consecutive channels of a row,
#     as the fast butterfly: for h = 1, 2, 4, 8, every pair (i, i+h) with
#     i & h == 0 becomes (a + b, a - b) in fp32; then every value is
#     multiplied by 1/4 (exact), which makes H orthonormal and symmetric;
#   - a block is one 128-row tile of one (b, h) (the attention tile);
#     scale = amax / 448 in fp32 (1 when the block is all zero), code =
#     e4m3(value / scale), round to nearest even.

def wht16_fp32(x):
    """The 16-point Walsh-Hadamard butterfly on the last axis groups of 16
    (last axis length a multiple of 16), fp32, in the order stated above."""
    v = np.array(x, dtype=np.float32, copy=True)
    shape = v.shape
    v = v.reshape(-1, 16)
    for h in (1, 2, 4, 8):
        for i in range(16):
            if i & h == 0:
                a = v[:, i].copy()
                b = v[:, i + h].copy()
                v[:, i] = a + b
                v[:, i + h] = a - b
    v = v * np.float32(0.25)
    return v.reshape(shape)


def quantize_fp8_blocks(x, hadamard: bool, block: int = 128):
    """e4m3 codes and per-block scales of a [B, H, N, d] tensor (values as
    the GPU reads them, i.e. already rounded to the input type).  Returns
    (codes: torch.float8_e4m3fn [B, H, N, d], scales: float32 [B, H,
    ceil(N / block)])."""
    import torch
    x = np.asarray(x, dtype=np.float32)
    B, H, N, d = x.shape
    v = wht16_fp32(x) if hadamard else x.copy()
    nt = (N + block - 1) // block
    scales = np.empty((B, H, nt), dtype=np.float32)
    q = np.empty_like(v)
    for t in range(nt):
        blk = v[:, :, t * block:(t + 1) * block, :]
        amax = np.abs(blk).max(axis=(2, 3)).astype(np.float32)
        sc = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
        scales[:, :, t] = sc
        q[:, :, t * block:(t + 1) * block, :] = blk / sc[:, :, None, None]
    q = np.clip(q, -448.0, 448.0).astype(np.float32)
    codes = torch.from_numpy(q).to(torch.float8_e4m3fn)
    return codes, scales

"""Shared helpers of the GPU parity tests: run the CUDA library on seeded
inputs and compare with the fp64 oracle, element by element.

Tolerances (O against the fp64 oracle; LSE in natural-log units):
  fp16 / bf16 / fp32: max |dO| <= 1e-2, mean |dO| <= 1e-3, max |dLSE| <= 1e-3
  e4m3:              max |dO| <= 6e-2, max |dLSE| <= 1e-3
The 16-bit and e4m3 bounds are the ones the method's target states; fp32
takes the 16-bit bounds (it runs in exact fp32 arithmetic on the CUDA
cores, not on the tensor cores).
"""
from __future__ import annotations

import numpy as np
import torch

import attn_inputs as ai
import oracle
import warp_specialized_gb300 as ws

TOL = {
    "fp32": dict(o_max=1e-2, o_mean=1e-3, lse=1e-3),
    "fp16": dict(o_max=1e-2, o_mean=1e-3, lse=1e-3),
    "bf16": dict(o_max=1e-2, o_mean=1e-3, lse=1e-3),
    "fp8": dict(o_max=6e-2, o_mean=None, lse=1e-3),
}

GUARD = 256  # canary elements before and after each output


def run_gpu(inp: ai.AttnInputs, causal: bool, guard: bool = True, split_tail=None,
            workspace=None, exp2_fma: bool = False):
    """Runs the library on the inputs (copied to cuda:0).  O and LSE are
    NaN-prefilled and surrounded by canaries; returns (O, LSE) on the CPU and
    asserts the canaries are intact.  split_tail / workspace / exp2_fma: as
    attn_fwd."""
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    B, H, N, d = inp.shape
    out_dtype = torch.bfloat16 if inp.dtype == "fp8" else q.dtype
    g = GUARD if guard else 0
    o_buf = torch.full((B * H * N * d + 2 * g,), float("nan"), dtype=out_dtype, device=dev)
    l_buf = torch.full((B * H * N + 2 * g,), float("nan"), dtype=torch.float32, device=dev)
    if g:
        o_buf[:g] = 7.0
        o_buf[-g:] = 7.0
        l_buf[:g] = 7.0
        l_buf[-g:] = 7.0
    o = o_buf[g:g + B * H * N * d].view(B, H, N, d)
    lse = l_buf[g:g + B * H * N].view(B, H, N)
    if inp.dtype == "fp8":
        ws.attn_fwd_fp8(q, k, v, inp.descale["q"], inp.descale["k"], inp.descale["v"],
                        scale=inp.scale, causal=causal, out=o, lse=lse, split_tail=split_tail,
                        workspace=workspace, exp2_fma=exp2_fma)
    else:
        ws.attn_fwd(q, k, v, scale=inp.scale, causal=causal, out=o, lse=lse,
                    split_tail=split_tail, workspace=workspace, exp2_fma=exp2_fma)
    torch.cuda.synchronize()
    st = ws.attn_fwd_status()
    assert st == 0, f"watchdog status {ws.STATUS_NAMES.get(st, st)}"
    if g:
        for buf in (o_buf, l_buf):
            assert torch.all(buf[:g].float() == 7.0) and torch.all(buf[-g:].float() == 7.0), \
                "output canaries overwritten"
    return o.float().cpu(), lse.cpu()


def sample_rows(N: int, n_random: int, seed: int):
    """First and last 128-row tiles plus n_random seeded rows."""
    rows = set(range(min(128, N))) | set(range(max(0, N - 128), N))
    g = np.random.default_rng(seed)
    rows |= set(g.integers(0, N, size=n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def oracle_ref(inp: ai.AttnInputs, causal: bool, heads=None, rows=None):
    """fp64 oracle on the values the GPU reads.  heads: list of (b, h) or
    None for all; rows: array of rows or None for all.  Returns
    (O [n_heads, R, d], LSE [n_heads, R])."""
    q, k, v = (x.numpy() for x in inp.as_float64())
    B, H, N, d = inp.shape
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    qs = np.stack([q[b, h] for b, h in heads])[None]
    ks = np.stack([k[b, h] for b, h in heads])[None]
    vs = np.stack([v[b, h] for b, h in heads])[None]
    o, lse = oracle.attn_fwd(qs, ks, vs, inp.scale, causal, rows=rows)
    return o[0], lse[0]


def compare(inp: ai.AttnInputs, causal: bool, o_gpu, lse_gpu, heads=None, rows=None):
    """Element-wise comparison; returns the error statistics and asserts the
    dtype's tolerance."""
    B, H, N, d = inp.shape
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    o_ref, lse_ref = oracle_ref(inp, causal, heads, rows)
    og = torch.stack([o_gpu[b, h] for b, h in heads]).double().numpy()
    lg = torch.stack([lse_gpu[b, h] for b, h in heads]).double().numpy()
    if rows is not None:
        og = og[:, rows]
        lg = lg[:, rows]
    assert np.isfinite(og).all(), "non-finite (or unwritten) O"
    assert np.isfinite(lg).all(), "non-finite (or unwritten) LSE"
    err_o = np.abs(og - o_ref)
    err_l = np.abs(lg - lse_ref)
    stats = dict(o_max=float(err_o.max()), o_mean=float(err_o.mean()), lse=float(err_l.max()))
    tol = TOL[inp.dtype]
    assert stats["o_max"] <= tol["o_max"], stats
    if tol["o_mean"] is not None:
        assert stats["o_mean"] <= tol["o_mean"], stats
    assert stats["lse"] <= tol["lse"], stats
    return stats

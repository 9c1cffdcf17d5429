"""Parity of the CUDA backward pass (dQ, dK, dV) with the fp64 backward
oracle, on seeded inputs, through the C ABI.  The forward that produces O and
LSE is the library's own; the oracle differentiates the exact definition.

Tolerance: the gradients pass through three 16-bit roundings on the GPU
(P and dS rounded to the input type before their matrix products, and the
outputs rounded once), each about 2^-9 relative for bf16, plus D computed
from the rounded O.  The bound used, per tensor, is
    max |g - g_ref| <= 2e-2 * max |g_ref|   and   mean |g - g_ref| <= 5e-3 * mean |g_ref|
for bf16 and a quarter of that for fp16 (3 more mantissa bits).
"""
import json
import os

import numpy as np
import pytest
import torch

import attn_inputs as ai
import oracle
import warp_specialized_gb300 as ws

pytestmark = pytest.mark.gpu

STATS = []
TOL = {"bf16": (2e-2, 5e-3), "fp16": (5e-3, 1.25e-3)}


@pytest.fixture(scope="module", autouse=True)
def _built_and_report():
    ws.load_library(build_if_missing=True)
    yield
    rec = os.environ.get("ATTN_RECORD_DIR")
    if rec:  # optional JSON record of the measured errors
        os.makedirs(rec, exist_ok=True)
        with open(os.path.join(rec, "bwd_stats.json"), "w") as f:
            json.dump(STATS, f, indent=1)


def run_bwd(inp: ai.AttnInputs, causal: bool, dout: torch.Tensor):
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    o, lse = ws.attn_fwd(q, k, v, scale=inp.scale, causal=causal)
    do = dout.to(dev)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    ws.attn_bwd(q, k, v, o, lse, do, scale=inp.scale, causal=causal, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert ws.attn_fwd_status() == 0
    return dq.float().cpu(), dk.float().cpu(), dv.float().cpu()


def compare_grads(inp, causal, dout, got, heads=None, label=""):
    B, H, N, d = inp.shape
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    q, k, v = (x.numpy() for x in inp.as_float64())
    do = dout.double().numpy()
    sel = lambda x: np.stack([x[b, h] for b, h in heads])[None]
    ref = oracle.attn_bwd(sel(q), sel(k), sel(v), sel(do), inp.scale, causal)
    tmax, tmean = TOL[inp.dtype]
    out = {"label": label, "shape": [B, H, N, d], "dtype": inp.dtype, "causal": causal}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        gs = sel(g.double().numpy())
        assert np.isfinite(gs).all(), f"non-finite (or unwritten) {name}"
        err = np.abs(gs - r)
        out[name] = dict(max_err=float(err.max()), mean_err=float(err.mean()),
                         max_ref=float(np.abs(r).max()), mean_ref=float(np.abs(r).mean()))
    STATS.append(out)
    for name in ("dq", "dk", "dv"):
        s = out[name]
        assert s["max_err"] <= tmax * s["max_ref"] + 1e-6, (name, out)
        assert s["mean_err"] <= tmean * s["mean_ref"] + 1e-7, (name, out)
    return out


SMALL = [
    (1, 2, 128, 128, "bf16"),
    (1, 2, 256, 64, "bf16"),
    (2, 2, 200, 128, "bf16"),
    (1, 2, 333, 64, "bf16"),
    (1, 1, 1, 128, "bf16"),
    (1, 3, 512, 128, "bf16"),
    (1, 2, 300, 128, "fp16"),
    (1, 2, 256, 64, "fp16"),
]


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("B,H,N,d,dtype", SMALL, ids=lambda x: str(x))
def test_bwd_small(B, H, N, d, dtype, causal):
    inp = ai.make_inputs(B, H, N, d, dtype, seed=300 + N + d)
    dout = ai.make_inputs(B, H, N, d, dtype, seed=900 + N + d).q  # seeded N(0,1), same dtype
    got = run_bwd(inp, causal, dout)
    compare_grads(inp, causal, dout, got, label="small")


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_bwd_many_items(causal):
    """More work items than SMs in both backward kernels."""
    inp = ai.make_inputs(2, 100, 256, 128, "bf16", seed=31)
    dout = ai.make_inputs(2, 100, 256, 128, "bf16", seed=32).q
    got = run_bwd(inp, causal, dout)
    compare_grads(inp, causal, dout, got, heads=[(0, 0), (0, 99), (1, 50)], label="many_items")


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_bwd_n2048_workload(causal):
    """The bf16 N=2048 d=128 workload (B=4, H=16); the oracle checks four
    heads."""
    inp = ai.workload("bf16_n2048_d128")
    B, H, N, d = inp.shape
    dout = ai.make_inputs(B, H, N, d, "bf16", seed=1234 + 51).q
    got = run_bwd(inp, causal, dout)
    for g in got:
        assert torch.isfinite(g).all()
    compare_grads(inp, causal, dout, got, heads=[(0, 0), (1, 7), (2, 11), (3, 15)], label="n2048")


def test_bwd_repeatable():
    inp = ai.make_inputs(1, 4, 384, 128, "bf16", seed=41)
    dout = ai.make_inputs(1, 4, 384, 128, "bf16", seed=42).q
    a = run_bwd(inp, True, dout)
    b = run_bwd(inp, True, dout)
    for x, y in zip(a, b):
        assert torch.equal(x, y)

"""FP8 block quantisation with the Walsh-Hadamard rotation, on the GPU:
codes and scales bit-exact against the oracle, block-scaled e4m3 attention
against the fp64 oracle, and the RMSE comparison the source makes (rotation
plus block scales against one per-tensor scale, on inputs with outlier
channels)."""
import json
import os

import numpy as np
import pytest
import torch

import attn_inputs as ai
import oracle
import warp_specialized_gb300 as ws
from attn_check import sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ws.load_library(build_if_missing=True)


@pytest.mark.parametrize("hadamard", [False, True], ids=["plain", "hadamard"])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64), ("fp32", 128), ("bf16", 64)])
def test_quantisation_is_bit_exact(dtype, d, hadamard):
    x = ai.make_inputs(2, 3, 300, d, dtype, seed=5 + d, outliers=4).q
    codes, scales = ws.attn_quantize_fp8(x.cuda(), hadamard=hadamard)
    torch.cuda.synchronize()
    want_codes, want_scales = oracle.quantize_fp8_blocks(x.float().numpy(), hadamard)
    assert torch.equal(codes.cpu().view(torch.uint8), want_codes.view(torch.uint8))
    np.testing.assert_array_equal(scales.cpu().numpy(), want_scales)


@pytest.mark.parametrize("hadamard", [False, True], ids=["plain", "hadamard"])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 128), ("fp32", 64), ("bf16", 64)])
def test_quantisation_bit_exact_across_block_magnitudes(dtype, d, hadamard):
    """Many tiles whose magnitudes step by powers of two from block to block
    (one all-zero block per head), with a ragged last tile.  For bf16 and
    fp32 two tiles sit at 2^-80 and 2^75, where the block scale leaves the
    range of the kernel's refined quotient and it divides in IEEE instead."""
    x = ai.make_inputs(2, 2, 33 * 128 + 77, d, dtype, seed=40 + d, outliers=4).q.float()
    B, H, N, _ = x.shape
    nt = (N + 127) // 128
    lo, hi = (-8, 6) if dtype == "fp16" else (-30, 30)
    e = torch.tensor([lo + (t * 7) % (hi - lo + 1) for t in range(nt)], dtype=torch.float32)
    if dtype != "fp16":
        e[9], e[20] = -80.0, 75.0
    f = torch.pow(2.0, e).repeat_interleave(128)[:N]
    f[5 * 128:6 * 128] = 0.0
    x = (x * f[None, None, :, None]).to(ai.DTYPES[dtype])
    codes, scales = ws.attn_quantize_fp8(x.cuda(), hadamard=hadamard)
    torch.cuda.synchronize()
    want_codes, want_scales = oracle.quantize_fp8_blocks(x.float().numpy(), hadamard)
    assert torch.equal(codes.cpu().view(torch.uint8), want_codes.view(torch.uint8))
    np.testing.assert_array_equal(scales.cpu().numpy(), want_scales)
    assert (scales.cpu()[:, :, 5] == 1.0).all()
    if dtype != "fp16":
        assert (scales.cpu()[:, :, 9] < 2.0 ** -60).all() and (scales.cpu()[:, :, 20] > 2.0 ** 60).all()


def _dequant(codes, scales):
    B, H, N, d = codes.shape
    c = codes.to(torch.float64)
    s = scales.to(torch.float64).repeat_interleave(128, dim=2)[:, :, :N]
    return c * s[..., None]


def _quantised_inputs(inp, hadamard):
    q, k = inp.q.cuda(), inp.k.cuda()
    qc, qs = ws.attn_quantize_fp8(q, hadamard=hadamard)
    kc, ks = ws.attn_quantize_fp8(k, hadamard=hadamard)
    vf = inp.v.float()
    v_scale = float(vf.abs().max()) / 448.0
    vc = (vf / v_scale).to(torch.float8_e4m3fn)
    return qc, qs, kc, ks, vc, v_scale


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_blockscaled_attention_parity(causal):
    inp = ai.make_inputs(1, 4, 700, 128, "bf16", seed=21, outliers=4, v_dist="uniform")
    qc, qs, kc, ks, vc, v_scale = _quantised_inputs(inp, True)
    o, lse = ws.attn_fwd_fp8_blockscaled(qc, kc, vc.cuda(), qs, ks, v_scale, scale=inp.scale,
                                         causal=causal)
    torch.cuda.synchronize()
    assert ws.attn_fwd_status() == 0
    qd, kd = _dequant(qc.cpu(), qs.cpu()), _dequant(kc.cpu(), ks.cpu())
    vd = vc.to(torch.float64) * v_scale
    o_ref, lse_ref = oracle.attn_fwd(qd.numpy(), kd.numpy(), vd.numpy(), inp.scale, causal)
    err = np.abs(o.float().cpu().double().numpy() - o_ref)
    assert err.max() <= 6e-2, err.max()
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= 1e-3


def test_hadamard_block_fp8_lowers_rmse_on_outliers():
    """Q and K with 4 outlier channels x20 (the d = 128 version of the
    outlier workload); RMSE of O against the exact attention of the bf16
    inputs, for one per-tensor scale and for rotation + block scales."""
    inp = ai.make_inputs(2, 8, 2048, 128, "bf16", seed=1234 + 3, outliers=4, v_dist="uniform")
    B, H, N, d = inp.shape
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    # per-tensor e4m3 (amax / 448 per tensor), the fp8 workload's recipe
    def per_tensor(t):
        f = t.float()
        sc = float(f.abs().max()) / 448.0
        return (f / sc).to(torch.float8_e4m3fn), sc
    q8, sq = per_tensor(q)
    k8, sk = per_tensor(k)
    v8, sv = per_tensor(v)
    o_pt, _ = ws.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, scale=inp.scale)
    qc, qs, kc, ks, vc, v_scale = _quantised_inputs(inp, True)
    o_hb, _ = ws.attn_fwd_fp8_blockscaled(qc, kc, vc.cuda(), qs, ks, v_scale, scale=inp.scale)
    torch.cuda.synchronize()
    rows = sample_rows(N, 64, seed=3)
    heads = [(0, 0), (0, 5), (1, 2), (1, 7)]
    q64, k64, v64 = (x.numpy() for x in inp.as_float64())
    sel = lambda x: np.stack([x[b, h] for b, h in heads])[None]
    o_ref, _ = oracle.attn_fwd(sel(q64), sel(k64), sel(v64), inp.scale, False, rows=rows)
    def rmse(o):
        g = np.stack([o.float().cpu().double().numpy()[b, h][rows] for b, h in heads])[None]
        return float(np.sqrt(np.mean((g - o_ref) ** 2)))
    r_pt, r_hb = rmse(o_pt), rmse(o_hb)
    rec = os.environ.get("ATTN_RECORD_DIR")
    if rec:  # optional JSON record of the two errors
        os.makedirs(rec, exist_ok=True)
        with open(os.path.join(rec, "fp8_rmse.json"), "w") as f:
            json.dump({"per_tensor": r_pt, "hadamard_block": r_hb, "ratio": r_pt / r_hb}, f)
    assert r_hb < r_pt, (r_pt, r_hb)

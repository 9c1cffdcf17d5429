"""Long sequences: one head spans hundreds of query tiles and every work item
walks hundreds of key blocks, so the ring, the barrier phases and the
persistent schedule run far longer than at the named workloads.  Checked
against the fp64 oracle on sampled rows (forward) and on every row of one
head (backward)."""
import numpy as np
import pytest
import torch

import attn_inputs as ai
import oracle
import warp_specialized_gb300 as ws
from attn_check import compare, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ws.load_library(build_if_missing=True)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("d", [128, 64])
def test_forward_n65536(d, causal):
    inp = ai.make_inputs(1, 2, 65536 + 37, d, "bf16", seed=500 + d)  # ragged last tile
    o, lse = run_gpu(inp, causal, guard=False)
    rows = sample_rows(inp.shape[2], 48, seed=d)
    compare(inp, causal, o, lse, rows=rows)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_backward_n8192_one_head(causal):
    inp = ai.make_inputs(1, 1, 8192, 128, "bf16", seed=611)
    dout = ai.make_inputs(1, 1, 8192, 128, "bf16", seed=612).q
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    o, lse = ws.attn_fwd(q, k, v, scale=inp.scale, causal=causal)
    dq, dk, dv = ws.attn_bwd(q, k, v, o, lse, dout.to(dev), scale=inp.scale, causal=causal)
    torch.cuda.synchronize()
    assert ws.attn_fwd_status() == 0
    q64, k64, v64 = (x.numpy() for x in inp.as_float64())
    ref = oracle.attn_bwd(q64, k64, v64, dout.double().numpy(), inp.scale, causal)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        gs = g.float().cpu().double().numpy()
        assert np.isfinite(gs).all(), name
        err = np.abs(gs - r)
        # the bf16 bounds of the backward parity tests
        assert err.max() <= 2e-2 * np.abs(r).max() + 1e-6, (name, float(err.max()))
        assert err.mean() <= 5e-3 * np.abs(r).mean() + 1e-7, (name, float(err.mean()))

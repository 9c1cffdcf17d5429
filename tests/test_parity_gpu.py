"""Parity of the CUDA library with the fp64 oracle on seeded inputs, through
the C ABI (via the ctypes binding).  Needs a GB300 (sm_103a)."""
import numpy as np
import pytest
import torch

import attn_inputs as ai
from attn_check import compare, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import warp_specialized_gb300 as ws
    ws.load_library(build_if_missing=True)
    assert torch.cuda.is_available()


# ---------------------------------------------------------------- small cases
# Several tiles and ragged tails, full oracle.

SMALL = [
    # (B, H, N, d, dtype)
    (1, 2, 128, 128, "bf16"),
    (1, 2, 256, 128, "bf16"),
    (1, 1, 1, 128, "bf16"),
    (1, 2, 63, 128, "bf16"),
    (1, 2, 127, 128, "bf16"),
    (1, 2, 129, 128, "bf16"),
    (2, 2, 200, 128, "bf16"),
    (1, 3, 300, 128, "bf16"),
    (1, 2, 640, 128, "bf16"),
    (1, 2, 333, 64, "bf16"),
    (1, 2, 256, 64, "fp16"),
    (1, 2, 1, 64, "bf16"),
    (1, 2, 100, 64, "bf16"),
    (1, 2, 129, 64, "fp16"),
    (1, 2, 333, 256, "bf16"),
    (1, 2, 256, 256, "fp16"),
    (1, 2, 200, 128, "fp16"),
    (1, 1, 128, 64, "fp32"),
    (1, 2, 333, 64, "fp32"),
    (1, 2, 200, 128, "fp32"),
    (1, 2, 256, 128, "fp8"),
    (1, 2, 333, 128, "fp8"),
]


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("B,H,N,d,dtype", SMALL, ids=lambda x: str(x))
def test_small_shapes(B, H, N, d, dtype, causal):
    inp = ai.make_inputs(B, H, N, d, dtype, seed=100 + N + d)
    o, lse = run_gpu(inp, causal)
    compare(inp, causal, o, lse)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_persistent_loop_more_items_than_sms(causal):
    """B*H*pairs well above the SM count: every CTA walks several items."""
    inp = ai.make_inputs(2, 160, 256, 128, "bf16", seed=7)
    o, lse = run_gpu(inp, causal)
    heads = [(0, 0), (0, 77), (1, 5), (1, 159)]
    compare(inp, causal, o, lse, heads=heads)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("N", [128, 512, 640])
def test_d64_s_buffers_across_items(N, causal):
    """d = 64 uses its three S buffers in turn across all of a CTA's work
    items.  At N = 512 and 640 an item's S count (n[0] + n[1]: 8 / 10
    non-causal, 3 and 7 / 3, 7 and 10 causal) is not always a multiple of
    three, so each item starts the rotation at another buffer; at N = 128
    every item is one block (two S products, none issued ahead); 400 heads
    give every CTA several items."""
    inp = ai.make_inputs(1, 400, N, 64, "bf16", seed=31 + N)
    o, lse = run_gpu(inp, causal)
    heads = [(0, 0), (0, 1), (0, 151), (0, 152), (0, 303), (0, 399)]
    compare(inp, causal, o, lse, heads=heads)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_schedule_partial_reversed_round(causal):
    """200 work items on a 152-CTA grid: the second round runs in reversed
    CTA order and is only partly filled."""
    inp = ai.make_inputs(1, 200, 256, 128, "bf16", seed=9)
    o, lse = run_gpu(inp, causal)
    heads = [(0, 0), (0, 151), (0, 152), (0, 199)]
    compare(inp, causal, o, lse, heads=heads)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_outlier_channels_small(causal):
    inp = ai.make_inputs(2, 4, 512, 64, "fp16", seed=11, outliers=4, v_dist="uniform")
    o, lse = run_gpu(inp, causal)
    compare(inp, causal, o, lse)


def test_large_scores_no_overflow():
    """Scores of several hundred (scaled): the running max keeps every
    exponential in range."""
    inp = ai.make_inputs(1, 2, 384, 128, "bf16", seed=12, scale=3.0)
    for causal in (False, True):
        o, lse = run_gpu(inp, causal)
        compare(inp, causal, o, lse)


def test_repeat_calls_are_bitwise_identical():
    inp = ai.make_inputs(1, 4, 512, 128, "bf16", seed=13)
    o1, l1 = run_gpu(inp, True)
    o2, l2 = run_gpu(inp, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------- the named workloads
# Full sizes, in the launch configuration the benchmark times; the oracle
# checks every head on the first and last 128-row tiles plus seeded rows.

def _workload_case(name, dtype, causal, n_random, head_stride=1):
    inp = ai.workload(name, dtype)
    B, H, N, d = inp.shape
    o, lse = run_gpu(inp, causal, guard=False)
    heads = [(b, h) for b in range(B) for h in range(H)][::head_stride]
    rows = sample_rows(N, n_random, seed=len(name) + N)
    stats = compare(inp, causal, o, lse, heads=heads, rows=rows)
    # properties at every element: finite, and |O| bounded by max |V|
    vmax = float(inp.as_float64()[2].abs().max())
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    assert float(o.abs().max()) <= vmax * 1.01 + 1e-2
    return stats


def test_workload_fp32_n128_d64():
    inp = ai.workload("fp32_n128_d64")
    o, lse = run_gpu(inp, False)
    compare(inp, False, o, lse)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_workload_bf16_n2048(causal):
    inp = ai.workload("bf16_n2048_d128")
    o, lse = run_gpu(inp, causal, guard=False)
    compare(inp, causal, o, lse)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_workload_bf16_n8192(causal):
    _workload_case("bf16_n8192_d128", None, causal, n_random=256)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("name", ["outlier_d64", "outlier_d256"])
def test_workload_outliers(name, dtype, causal):
    _workload_case(name, dtype, causal, n_random=64, head_stride=8)


def test_workload_fp8_n8192():
    _workload_case("fp8_n8192_d128", None, False, n_random=128, head_stride=2)

"""ATTN_OPT_EXP2_FMA on the GPU: the forward with 4 of every 32
exponentials computed on the FMA pipe (attn_fwd_opt / attn_fwd_fp8_opt)
against the fp64 oracle, element by element, at the same bounds as the
default path (the polynomial's 7.5e-5 relative error is far below the
rounding of P); plus its argument checks.  Needs a GB300 (sm_103a)."""
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


CASES = [
    (1, 2, 333, 64, "bf16"),
    (1, 2, 640, 128, "bf16"),
    (1, 1, 1, 128, "bf16"),
    (2, 3, 1100, 128, "bf16"),
    (1, 2, 333, 128, "fp8"),
    (1, 2, 1024, 128, "fp8"),
]


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
@pytest.mark.parametrize("B,H,N,d,dtype", CASES, ids=lambda x: str(x))
def test_exp2_fma_parity(B, H, N, d, dtype, causal):
    inp = ai.make_inputs(B, H, N, d, dtype, seed=900 + N + d)
    o, lse = run_gpu(inp, causal, exp2_fma=True)
    compare(inp, causal, o, lse)


@pytest.mark.parametrize("causal", [False, True], ids=["nc", "causal"])
def test_exp2_fma_workload_sampled(causal):
    """The headline workload's shape (B2 H16 N8192 d128, bf16) on sampled rows."""
    inp = ai.workload("bf16_n8192_d128")
    o, lse = run_gpu(inp, causal, exp2_fma=True)
    rows = sample_rows(inp.shape[2], 64, seed=3)
    compare(inp, causal, o, lse, heads=[(0, 0), (1, 15)], rows=rows)


def test_exp2_fma_checks():
    import warp_specialized_gb300 as ws
    dev = torch.device("cuda", 0)
    for dt, d in ((torch.float16, 128), (torch.bfloat16, 256)):
        q = torch.randn(1, 1, 256, d, device=dev, dtype=dt)
        with pytest.raises(ws.AttnError) as e:
            ws.attn_fwd(q, q, q, exp2_fma=True)
        assert e.value.status == 2  # ATTN_ERR_UNSUPPORTED
    q = torch.randn(1, 1, 256, 128, device=dev, dtype=torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 256, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(), 1, 1, 256,
            128, 0.088, False, ws.ATTN_BF16)
    assert ws.attn_fwd_opt_raw(*args, 2, s) == 1   # unknown option bit
    assert ws.attn_fwd_opt_raw(*args, 0, s) == 0   # no option: attn_fwd
    assert ws.attn_fwd_opt_raw(*args, ws.ATTN_OPT_EXP2_FMA, s) == 0
    torch.cuda.synchronize()
    assert ws.attn_fwd_status() == 0

"""attn_bwd_noalloc: the backward pass for callers that cannot allocate
device memory when they call it (their device memory belongs to a pool they
manage, or their host framework owns every allocation, or a step must not
risk an allocation failing halfway).  The entry point takes no workspace and
uses an array inside the library instead.

Its GPU test calls it through the C ABI twice in a row and checks both
results against attn_bwd with a caller-provided workspace, within the
backward tolerance the other backward tests use.  This file is collected
last so that a run stopping at the first failure has already run the rest.
"""
import pytest
import torch

import attn_inputs as ai
import warp_specialized_gb300 as ws

A = 1 << 20  # fake, 16-byte aligned address: the size check rejects first

# bf16 bounds of the backward tests: max |g - g_ref| <= 2e-2 max |g_ref|,
# mean |g - g_ref| <= 5e-3 mean |g_ref|
TOL_MAX, TOL_MEAN = 2e-2, 5e-3


def test_rejects_shapes_beyond_its_array():
    """More than 2^20 padded query rows do not fit the library's 8 MiB array:
    a clear ATTN_ERR_INVALID_ARG before anything touches the device."""
    lib = ws.load_library(build_if_missing=True)
    # 64 heads x 16,512 rows (N = 16,385 rounds up to 129 tiles) > 2^20
    rc = lib.attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, 4, 16, 16385, 128, 0.1, 0, ws.ATTN_BF16,
                              None)
    assert rc == 1
    assert lib.attn_bwd_noalloc(A, A, A, A, A, A, A, A, A, 0, 16, 128, 128, 0.1, 0,
                                ws.ATTN_BF16, None) == 1


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    lib = ws.load_library(build_if_missing=True)
    dev = torch.device("cuda", 0)
    B, H, N, d = 2, 3, 1000, 128
    inp = ai.make_inputs(B, H, N, d, "bf16", seed=77)
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    dout = ai.make_inputs(B, H, N, d, "bf16", seed=78).q.to(dev)
    for causal in (True, False):
        o, lse = ws.attn_fwd(q, k, v, scale=inp.scale, causal=causal)
        ref = ws.attn_bwd(q, k, v, o, lse, dout, scale=inp.scale, causal=causal)
        torch.cuda.synchronize()
        assert ws.attn_fwd_status() == 0
        stream = torch.cuda.current_stream().cuda_stream
        for _ in range(2):
            got = [torch.full_like(q, float("nan")) for _ in range(3)]
            rc = lib.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      dout.data_ptr(), lse.data_ptr(), got[0].data_ptr(),
                                      got[1].data_ptr(), got[2].data_ptr(), B, H, N, d,
                                      inp.scale, int(causal), ws.ATTN_BF16, stream)
            assert rc == 0, ws.attn_status_string(rc)
            torch.cuda.synchronize()
            assert ws.attn_fwd_status() == 0
            for g, r in zip(got, ref):
                g, r = g.float(), r.float()
                assert torch.isfinite(g).all()
                err = (g - r).abs()
                assert err.max() <= TOL_MAX * r.abs().max()
                assert err.mean() <= TOL_MEAN * r.abs().mean()

"""The forward pass on caller streams: two problems of different instances
(bf16 d=128 causal, fp16 d=64) launched alternately on two streams must give
bitwise the results of the same calls made one at a time on the default
stream, and the watchdog word must stay clear."""
import pytest
import torch

import attn_inputs as ai
import warp_specialized_gb300 as ws

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ws.load_library(build_if_missing=True)


def _problem(B, H, N, d, dtype, seed):
    inp = ai.make_inputs(B, H, N, d, dtype, seed=seed)
    return inp, tuple(t.cuda() for t in (inp.q, inp.k, inp.v))


def test_two_streams_match_serial_runs():
    pa, (qa, ka, va) = _problem(2, 4, 1000, 128, "bf16", 71)
    pb, (qb, kb, vb) = _problem(1, 6, 777, 64, "fp16", 72)
    ref_a = ws.attn_fwd(qa, ka, va, scale=pa.scale, causal=True)
    ref_b = ws.attn_fwd(qb, kb, vb, scale=pb.scale, causal=False)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(4):
        with torch.cuda.stream(sa):
            outs.append(("a", ws.attn_fwd(qa, ka, va, scale=pa.scale, causal=True, stream=sa)))
        with torch.cuda.stream(sb):
            outs.append(("b", ws.attn_fwd(qb, kb, vb, scale=pb.scale, causal=False, stream=sb)))
    torch.cuda.synchronize()
    assert ws.attn_fwd_status() == 0
    for name, (o, lse) in outs:
        ro, rl = ref_a if name == "a" else ref_b
        assert torch.equal(o, ro) and torch.equal(lse, rl), name


def test_pointers_off_the_device_are_rejected():
    """Host memory (pinned, so the GPU could reach it) and unregistered host
    memory in place of a device buffer: ATTN_ERR_INVALID_ARG, nothing runs."""
    inp = ai.make_inputs(1, 1, 128, 128, "bf16", seed=3)
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    pinned = torch.empty_like(inp.q).pin_memory()
    plain = torch.empty_like(inp.q)
    lib = ws.load_library()
    sh = torch.cuda.current_stream().cuda_stream
    for bad in (pinned, plain):
        args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr()]
        for pos in range(4):
            a = list(args)
            a[pos] = bad.data_ptr()
            assert lib.attn_fwd(*a, 1, 1, 128, 128, inp.scale, 0, ws.ATTN_BF16, sh) == 1
    torch.cuda.synchronize()
    assert ws.attn_fwd_status() == 0

"""The forward pass on caller streams: two problems launched alternately on
two streams (one taking the two-CTA cluster launch, one the single-CTA
launch) must give bitwise the results of the same calls made one at a time
on the default stream, and the watchdog word must stay clear."""
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
    pa, (qa, ka, va) = _problem(2, 4, 1000, 128, "bf16", 71)   # two-CTA clusters
    pb, (qb, kb, vb) = _problem(1, 6, 777, 64, "fp16", 72)     # one CTA per item
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

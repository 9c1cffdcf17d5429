"""The seeded input generator: determinism, shapes and the workload recipe."""
import torch

import attn_inputs as ai


def test_same_seed_same_bits():
    a = ai.make_inputs(1, 2, 33, 16, "bf16", seed=7)
    b = ai.make_inputs(1, 2, 33, 16, "bf16", seed=7)
    c = ai.make_inputs(1, 2, 33, 16, "bf16", seed=8)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert not torch.equal(a.q, c.q)


def test_outlier_channels_shared_by_q_and_k():
    x = ai.make_inputs(2, 2, 256, 64, "fp32", seed=3, outliers=4, v_dist="uniform")
    qa = x.q.abs().amax(dim=(0, 1, 2))
    ka = x.k.abs().amax(dim=(0, 1, 2))
    top_q = set(torch.topk(qa, 4).indices.tolist())
    top_k = set(torch.topk(ka, 4).indices.tolist())
    assert top_q == top_k
    assert x.v.min() >= -1.0 and x.v.max() <= 1.0


def test_fp8_quantisation_recipe():
    x = ai.make_inputs(1, 2, 128, 128, "fp8", seed=5)
    assert x.q.dtype == torch.float8_e4m3fn
    for name, t in (("q", x.q), ("k", x.k), ("v", x.v)):
        # per-tensor scale amax/448: the largest code is 448 (or its rounding)
        assert abs(float(t.to(torch.float32).abs().max()) - 448.0) <= 16.0
        assert x.descale[name] > 0
    q64, _, _ = x.as_float64()
    assert q64.dtype == torch.float64


def test_workload_table():
    assert ai.WORKLOADS["bf16_n8192_d128"][:5] == (2, 16, 8192, 128, "bf16")
    B, H, N, d = ai.WORKLOADS["outlier_d64"][:4]
    assert B * H * N == 2 ** 19
    assert ai.workload_flops(2, 16, 8192, 128, False) == 4.0 * 2 * 16 * 8192 ** 2 * 128
    assert ai.workload_flops(2, 16, 8192, 128, True) == 2.0 * 2 * 16 * 8192 ** 2 * 128

"""Pins of the fp64 backward oracle.

None re-types its formulas: the gradients are checked against central finite
differences of the forward oracle, against torch.autograd in fp64, and
against identities that follow from softmax rows summing to one.
"""
import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _loss(q, k, v, dout, scale, causal):
    o, _ = oracle.attn_fwd(q, k, v, scale, causal)
    return float((o * dout).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_finite_differences(causal):
    """dL/dx for L = sum(dO * O) against central differences of the forward
    oracle at a few seeded coordinates of each input."""
    B, H, N, d, scale = 1, 2, 11, 5, 0.7
    q, k, v = _rand((B, H, N, d), 1), _rand((B, H, N, d), 2), _rand((B, H, N, d), 3)
    dout = _rand((B, H, N, d), 4)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, scale, causal)
    g = np.random.default_rng(5)
    h = 1e-5
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(g.integers(0, s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num = (_loss(args_p["q"], args_p["k"], args_p["v"], dout, scale, causal) -
                   _loss(args_m["q"], args_m["k"], args_m["v"], dout, scale, causal)) / (2 * h)
            assert abs(num - grad[idx]) <= 1e-7 * max(1.0, abs(num)), (name, idx, num, grad[idx])


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_torch_autograd(causal):
    B, H, N, d, scale = 2, 2, 37, 16, 0.25
    q, k, v = _rand((B, H, N, d), 6, 2.0), _rand((B, H, N, d), 7, 2.0), _rand((B, H, N, d), 8)
    dout = _rand((B, H, N, d), 9)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, scale, causal)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ tv
    o.backward(torch.from_numpy(dout))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_identities(causal):
    """Rows of P sum to one, so (per head) sum_j dV_j = sum_i dO_i and
    sum_j dK_j = 0; adding one vector to every key shifts each score row by
    a constant, which leaves O, hence dQ, unchanged."""
    B, H, N, d, scale = 1, 3, 29, 8, 0.5
    q, k, v = _rand((B, H, N, d), 10), _rand((B, H, N, d), 11), _rand((B, H, N, d), 12)
    dout = _rand((B, H, N, d), 13)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dout, scale, causal)
    np.testing.assert_allclose(dv.sum(axis=2), dout.sum(axis=2), atol=1e-11)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-11)
    shift = _rand((1, 1, 1, d), 14, 3.0)
    dq2, _, dv2 = oracle.attn_bwd(q, k + shift, v, dout, scale, causal)
    np.testing.assert_allclose(dq2, dq, atol=1e-10)
    np.testing.assert_allclose(dv2, dv, atol=1e-10)


def test_single_key():
    """N = 1: P = 1, so dV = dO and dQ = dK = 0."""
    q, k, v = _rand((2, 2, 1, 6), 15), _rand((2, 2, 1, 6), 16), _rand((2, 2, 1, 6), 17)
    dout = _rand((2, 2, 1, 6), 18)
    for causal in (False, True):
        dq, dk, dv = oracle.attn_bwd(q, k, v, dout, 0.9, causal)
        np.testing.assert_allclose(dv, dout, atol=1e-14)
        np.testing.assert_allclose(dq, 0.0, atol=1e-14)
        np.testing.assert_allclose(dk, 0.0, atol=1e-14)

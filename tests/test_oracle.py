"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these re-calls the oracle's own formula to check it: each compares it
with a hand-derived value (tests/golden), a closed form, an invariant, the
card's blockwise recurrence, or a library routine (torch.softmax in fp64).
The definition being pinned is the "Warp specialization" concept card,
section "Implementation sketch" (output / row_sum, row_max + log(row_sum)).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _num(x):
    if isinstance(x, str):
        assert x.startswith("ln")
        return math.log(float(x[2:]))
    return float(x)


def _arr(rows):
    return np.array([[_num(x) for x in r] for r in rows], dtype=np.float64)


def _golden_cases():
    with open(GOLDEN) as f:
        data = json.load(f)
    for case in data["cases"]:
        for mode in ("noncausal", "causal"):
            yield case, mode


def _run_case(case, mode, swap_qk=False, scale=None):
    q = _arr(case["q"])[None, None]
    k = _arr(case["k"])[None, None]
    v = _arr(case["v"])[None, None]
    if swap_qk:
        q, k = k, q
    s = case["scale"] if scale is None else scale
    return oracle.attn_fwd(q, k, v, s, mode == "causal")


@pytest.mark.parametrize("case,mode", list(_golden_cases()),
                         ids=lambda x: x if isinstance(x, str) else x["name"])
def test_golden_hand_cases(case, mode):
    o, lse = _run_case(case, mode)
    want_o = _arr(case[mode]["o"])
    want_lse = np.array([_num(x) for x in case[mode]["lse"]])
    np.testing.assert_allclose(o[0, 0], want_o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], want_lse, rtol=0, atol=1e-13)


def _golden_matches(case, mode, **kw):
    o, lse = _run_case(case, mode, **kw)
    want_o = _arr(case[mode]["o"])
    want_lse = np.array([_num(x) for x in case[mode]["lse"]])
    return np.allclose(o[0, 0], want_o, atol=1e-9) and np.allclose(lse[0, 0], want_lse, atol=1e-9)


def test_golden_cases_detect_planted_mistakes():
    """The fixtures are sensitive: a transposed product (K.Q^T), a dropped
    scale or a flipped mask (planted here by feeding the oracle the wrong
    operands) does not reproduce them."""
    cases = {c["name"]: c for c, _ in _golden_cases()}
    three = cases["three_keys_ratios"]
    two = cases["two_keys_scale_half"]
    assert not _golden_matches(three, "noncausal", swap_qk=True)
    assert not _golden_matches(two, "noncausal", scale=1.0)
    # flipped mask direction == causal on the reversed sequence
    o_rev, _ = oracle.attn_fwd(_arr(three["q"])[::-1][None, None], _arr(three["k"])[::-1][None, None],
                               _arr(three["v"])[::-1][None, None], three["scale"], True)
    assert not np.allclose(o_rev[0, 0][::-1], _arr(three["causal"]["o"]), atol=1e-9)


def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * scale


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    """With V = I (d = N) the output row is the probability row itself:
    non-negative, summing to 1, and exactly 0 above the diagonal when causal."""
    N = 24
    q = _rand((1, 2, N, N), 1)
    k = _rand((1, 2, N, N), 2)
    v = np.broadcast_to(np.eye(N), (1, 2, N, N)).copy()
    p, _ = oracle.attn_fwd(q, k, v, 0.3, causal)
    assert (p >= 0).all()
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-13)
    if causal:
        iu = np.triu_indices(N, 1)
        assert (p[..., iu[0], iu[1]] == 0.0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_give_column_mean(causal):
    """Q = 0 makes every visible score 0: O_i is the mean of the visible V
    rows and LSE_i = ln(#visible) = ln N, or ln(i+1) when causal."""
    B, H, N, d = 2, 3, 37, 5
    q = np.zeros((B, H, N, d))
    k = _rand((B, H, N, d), 3)
    v = _rand((B, H, N, d), 4)
    o, lse = oracle.attn_fwd(q, k, v, 0.7, causal)
    for i in range(N):
        nvis = i + 1 if causal else N
        np.testing.assert_allclose(o[:, :, i], v[:, :, :nvis].mean(axis=2), atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(nvis), atol=1e-13)


def test_one_dominant_key_selects_its_value_row():
    """q_i = a e0, k_{j*} = b e0, other keys 0, scale a b = 60: O_i = v_{j*}
    up to (N-1) e^-60 and LSE_i = 60 + ln(1 + (N-1) e^-60)."""
    N, d, jstar = 50, 4, 17
    a, b, scale = 3.0, 4.0, 5.0
    q = np.zeros((1, 1, N, d))
    q[..., 0] = a
    k = np.zeros((1, 1, N, d))
    k[0, 0, jstar, 0] = b
    v = _rand((1, 1, N, d), 5)
    o, lse = oracle.attn_fwd(q, k, v, scale, False)
    eps = (N - 1) * math.exp(-60.0)
    assert np.abs(o[0, 0] - v[0, 0, jstar]).max() <= eps * (np.abs(v).max() * 2 + 1)
    np.testing.assert_allclose(lse[0, 0], 60.0 + math.log1p(eps), rtol=0, atol=1e-12)


def test_lse_is_log_sum_exp_of_scaled_scores():
    """LSE against a direct log(sum(exp)) without max subtraction, summed
    exactly (math.fsum) on small scores where no overflow can occur."""
    N, d, scale = 19, 6, 0.25
    q = _rand((1, 1, N, d), 6)
    k = _rand((1, 1, N, d), 7)
    v = _rand((1, 1, N, d), 8)
    for causal in (False, True):
        _, lse = oracle.attn_fwd(q, k, v, scale, causal)
        for i in range(N):
            terms = []
            for j in range(N if not causal else i + 1):
                s = scale * math.fsum(q[0, 0, i, c] * k[0, 0, j, c] for c in range(d))
                terms.append(math.exp(s))
            assert abs(lse[0, 0, i] - math.log(math.fsum(terms))) <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("block", [1, 3, 16, 40])
def test_blockwise_recurrence_matches_direct(causal, block):
    """The card's blockwise online-softmax recurrence (running max, rescale
    by exp(row_max - new_max)) agrees with the direct form on brute-force
    tiny inputs, for blocks that do and do not divide N."""
    B, H, N, d = 2, 2, 40, 8
    q = _rand((B, H, N, d), 9, 2.0)
    k = _rand((B, H, N, d), 10, 2.0)
    v = _rand((B, H, N, d), 11)
    o1, l1 = oracle.attn_fwd(q, k, v, 0.6, causal)
    o2, l2 = oracle.attn_fwd_blockwise(q, k, v, 0.6, causal, block)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("c", [-1000.0, 1000.0, 37.5])
@pytest.mark.parametrize("causal", [False, True])
def test_shift_invariance(c, causal):
    """An extra channel adding the constant c to every score leaves O
    unchanged and adds c to LSE, with no overflow at c = +-1000."""
    B, H, N, d, scale = 1, 2, 30, 6, 0.5
    q = _rand((B, H, N, d), 12)
    k = _rand((B, H, N, d), 13)
    v = _rand((B, H, N, d), 14)
    q2 = np.concatenate([q, np.ones((B, H, N, 1))], axis=-1)
    k2 = np.concatenate([k, np.full((B, H, N, 1), c / scale)], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, H, N, 1))], axis=-1)
    o1, l1 = oracle.attn_fwd(q, k, v, scale, causal)
    o2, l2 = oracle.attn_fwd(q2, k2, v2, scale, causal)
    assert np.isfinite(o2).all() and np.isfinite(l2).all()
    np.testing.assert_allclose(o2[..., :d], o1, rtol=0, atol=1e-11)
    np.testing.assert_allclose(l2 - c, l1, rtol=0, atol=1e-9)


def test_permutation_equivariance_noncausal():
    """Permuting the (K, V) rows together changes nothing (non-causal);
    permuting the queries permutes the outputs."""
    B, H, N, d = 1, 2, 33, 7
    q = _rand((B, H, N, d), 15)
    k = _rand((B, H, N, d), 16)
    v = _rand((B, H, N, d), 17)
    perm = np.random.default_rng(18).permutation(N)
    o1, l1 = oracle.attn_fwd(q, k, v, 0.4, False)
    o2, l2 = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(l2, l1, atol=1e-13)
    o3, l3 = oracle.attn_fwd(q[:, :, perm], k, v, 0.4, False)
    np.testing.assert_allclose(o3, o1[:, :, perm], atol=1e-13)
    np.testing.assert_allclose(l3, l1[:, :, perm], atol=1e-13)


def test_causal_row_zero_and_single_key():
    """Causal row 0 sees only key 0: O_0 = v_0, LSE_0 = scale q_0.k_0.
    With N = 1 the same holds with or without the mask."""
    B, H, N, d, scale = 2, 2, 9, 5, 0.8
    q = _rand((B, H, N, d), 19)
    k = _rand((B, H, N, d), 20)
    v = _rand((B, H, N, d), 21)
    o, lse = oracle.attn_fwd(q, k, v, scale, True)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0], scale * (q[:, :, 0] * k[:, :, 0]).sum(-1), atol=1e-13)
    for causal in (False, True):
        o1, l1 = oracle.attn_fwd(q[:, :, :1], k[:, :, :1], v[:, :, :1], scale, causal)
        np.testing.assert_allclose(o1, v[:, :, :1], atol=1e-14)
        np.testing.assert_allclose(l1[..., 0], scale * (q[:, :, 0] * k[:, :, 0]).sum(-1), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_softmax_fp64(causal):
    """Special case that reduces to library routines: torch.softmax and
    torch.logsumexp in fp64 on the CPU on small shapes."""
    B, H, N, d, scale = 2, 3, 45, 16, 0.25
    q = _rand((B, H, N, d), 22, 3.0)
    k = _rand((B, H, N, d), 23, 3.0)
    v = _rand((B, H, N, d), 24)
    o, lse = oracle.attn_fwd(q, k, v, scale, causal)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    want_o = torch.softmax(s, dim=-1) @ tv
    want_lse = torch.logsumexp(s, dim=-1)
    np.testing.assert_allclose(o, want_o.numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, want_lse.numpy(), atol=1e-12)


def test_row_subset_matches_full():
    B, H, N, d = 2, 2, 70, 8
    q = _rand((B, H, N, d), 25)
    k = _rand((B, H, N, d), 26)
    v = _rand((B, H, N, d), 27)
    rows = [0, 5, 69, 33, 5]
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, 0.3, causal)
        os_, ls_ = oracle.attn_fwd(q, k, v, 0.3, causal, rows=rows)
        np.testing.assert_array_equal(os_, o[:, :, rows])
        np.testing.assert_array_equal(ls_, lse[:, :, rows])


def test_rejects_bad_arguments():
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q, q, 1.0, False, rows=[4])
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q, q, 1.0, False, rows=[-1])
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q[:, :, :3], q, 1.0, False)

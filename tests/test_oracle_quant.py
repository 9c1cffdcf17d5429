"""Pins of the FP8 block quantisation oracle with the Walsh-Hadamard
rotation: the transform against scipy's Hadamard matrix and its algebra, the
quantisation against the e4m3 grid."""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle


def test_wht_matches_the_hadamard_matrix():
    H = scipy.linalg.hadamard(16).astype(np.float64) / 4.0   # Sylvester order, orthonormal
    x = np.random.default_rng(0).standard_normal((5, 3, 32)).astype(np.float32)
    y = oracle.wht16_fp32(x).astype(np.float64)
    ref = (x.astype(np.float64).reshape(-1, 16) @ H).reshape(x.shape)
    np.testing.assert_allclose(y, ref, atol=1e-5)


def test_wht_is_orthonormal_and_preserves_dot_products():
    g = np.random.default_rng(1)
    q = g.standard_normal((7, 64)).astype(np.float32)
    k = g.standard_normal((9, 64)).astype(np.float32)
    twice = oracle.wht16_fp32(oracle.wht16_fp32(q))
    np.testing.assert_allclose(twice, q, atol=1e-5)          # H H = I
    qr, kr = oracle.wht16_fp32(q), oracle.wht16_fp32(k)
    np.testing.assert_allclose(qr @ kr.T, q @ k.T, atol=1e-4)  # Q H (K H)^T = Q K^T
    e = np.zeros((1, 16), np.float32)
    e[0, 3] = 1.0
    assert np.all(np.abs(oracle.wht16_fp32(e)) == 0.25)       # a unit vector spreads evenly


def test_wht_spreads_an_outlier_channel():
    x = np.random.default_rng(2).standard_normal((256, 16)).astype(np.float32)
    x[:, 5] *= 20.0
    y = oracle.wht16_fp32(x)
    assert np.abs(y).max() < 0.5 * np.abs(x).max()


@pytest.mark.parametrize("hadamard", [False, True])
def test_block_quantisation_grid(hadamard):
    g = np.random.default_rng(3)
    x = g.standard_normal((2, 3, 300, 64)).astype(np.float32)
    x[0, 1, 130:140] = 0.0
    x[1, 2, 256:] = 0.0                                       # an all-zero block: scale 1
    codes, scales = oracle.quantize_fp8_blocks(x, hadamard)
    assert codes.dtype == torch.float8_e4m3fn and scales.shape == (2, 3, 3)
    c = codes.to(torch.float32).numpy()
    assert np.abs(c).max() <= 448.0
    v = oracle.wht16_fp32(x) if hadamard else x
    for b in range(2):
        for h in range(3):
            for t in range(3):
                blk = v[b, h, t * 128:(t + 1) * 128]
                amax = np.abs(blk).max()
                if amax == 0:
                    assert scales[b, h, t] == 1.0
                    continue
                assert scales[b, h, t] == np.float32(amax) / np.float32(448.0)
                assert np.abs(c[b, h, t * 128:(t + 1) * 128]).max() == 448.0
                # every code is the e4m3 value nearest to value / scale: within
                # half an e4m3 step (3 mantissa bits: 2^-4 relative, 2^-10 floor)
                r = blk / scales[b, h, t]
                cc = c[b, h, t * 128:(t + 1) * 128]
                step = np.maximum(np.abs(r) * 2.0 ** -3, 2.0 ** -9)
                assert np.all(np.abs(cc - r) <= 0.5 * step + 1e-6)

"""The optional FMA-pipe exponential of the forward kernel
(ATTN_OPT_EXP2_FMA), checked on the host: the polynomial's coefficients in
the kernel source are the Remez fit that fit_exp2_poly.py computes, the fit
reaches the minimax error it should, and the whole computation (Cody and
Waite's reduction x = n + f, the polynomial, n added to the exponent field),
restated in numpy fp32, follows 2^x within that error over the range the
softmax feeds it (x <= 0, results normal for x >= -125; between -126 and
-125 the result may land on a subnormal encoding, off by far less than the
row sums it joins), with exact zeros below -126.  No GPU needed."""
import os
import re

import numpy as np
import pytest

from warp_specialized_gb300 import fit_exp2_poly as fit

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNEL = os.path.join(ROOT, "warp_specialized_gb300", "csrc", "attn_fwd_kernel.cuh")


def _kernel_coefficients():
    src = open(KERNEL).read()
    body = src[src.index("void exp2_fma2("):]
    body = body[:body.index("\n}\n")]
    lits = [float(x) for x in re.findall(r"f2_pack\(([-0-9.e]+)f, \1f\)", body)]
    # the packed constants in order: 1.5*2^23, -1.5*2^23, -1, c3, c2, c1, c0
    assert lits[:3] == [12582912.0, -12582912.0, -1.0], lits
    c3, c2, c1, c0 = lits[3:7]
    return np.array([c0, c1, c2, c3], dtype=np.float32)


def test_kernel_constants_are_the_fit():
    got = _kernel_coefficients()
    want = fit.coefficients_f32()
    assert np.array_equal(got, want), (got, want)


def test_fit_is_minimax():
    """Degree 3 on [-1/2, 1/2]: the equioscillating error level is 7.48e-5
    (a wrong interval, degree or weight moves it by orders of magnitude),
    and the error alternates in sign at DEGREE + 2 points."""
    c, err = fit.fit()
    assert 7.0e-5 < err < 7.6e-5
    x = np.linspace(-0.5, 0.5, 20001)
    e = fit.rel_err(c, x)
    assert abs(e[0]) > 0.99 * err and abs(e[-1]) > 0.99 * err
    signs = np.sign(e[np.abs(e) > 0.99 * err])
    assert np.count_nonzero(np.diff(signs)) >= fit.DEGREE + 1
    # a plain least-squares fit on the same points is worse than minimax
    ls = np.polynomial.polynomial.polyfit(x, 2.0 ** x, fit.DEGREE)
    assert np.max(np.abs(fit.rel_err(ls, x))) > err


def _exp2_fma_f32(x):
    """The kernel's exp2_fma2, restated in numpy fp32 (each fma rounded once)."""
    x = np.asarray(x, dtype=np.float32)
    c0, c1, c2, c3 = (np.float32(v) for v in _kernel_coefficients())
    xx = np.maximum(x, np.float32(-127.0))
    magic = np.float32(12582912.0)
    t = (xx + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (xx.astype(np.float64) - n.astype(np.float64)).astype(np.float32)

    def fma(a, b, c):
        return (a.astype(np.float64) * b + c).astype(np.float32)

    q = fma(np.full_like(f, c3), f, c2)
    q = fma(q, f, c1)
    q = fma(q, f, c0)
    bits = q.view(np.int32) + (t.view(np.int32) << 23)
    e = bits.view(np.float32)
    return np.where(x < -126.0, np.float32(0.0), e)


def test_reduction_and_polynomial_track_exp2():
    rng = np.random.default_rng(5)
    x = np.concatenate([np.linspace(-126.0, 0.0, 400001), -rng.exponential(3.0, 100000),
                        np.arange(-126, 1, dtype=np.float64) + 0.5,
                        np.arange(-126, 1, dtype=np.float64)]).astype(np.float32)
    x = x[x >= -126.0]
    got = _exp2_fma_f32(x).astype(np.float64)
    want = 2.0 ** x.astype(np.float64)
    normal = x >= -125.0
    rel = np.abs(got[normal] / want[normal] - 1.0)
    assert rel.max() < 7.5e-5 + 3e-7, float(rel.max())
    assert np.max(np.abs(got[~normal] - want[~normal])) < 2.0 ** -126 * 2e-4


@pytest.mark.parametrize("x", [-np.inf, -1e30, -127.0, -126.5])
def test_below_range_is_zero(x):
    assert _exp2_fma_f32([x])[0] == 0.0


def test_exact_at_integers_up_to_c0():
    """At integer x the reduction leaves f = 0, so the result is c0 * 2^x."""
    c0 = float(_kernel_coefficients()[0])
    for n in range(-125, 1):
        assert _exp2_fma_f32([float(n)])[0] == np.float32(c0 * 2.0 ** n)

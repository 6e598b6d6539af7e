"""The E2M1 digit-plane representation of decode activations, restated in
numpy on the CPU (the CUDA prologue writes the same digits): a token's values
x, scaled by the power of two 2^-e that brings max |x| into (3, 6], are
written as six E2M1 digits d_0..d_5 with x 2^-e = sum_p d_p 6^-p + rest.
d_p is the round-to-nearest-even E2M1 value of the running residual r_p and
r_{p+1} = (r_p - d_p) 6.  These tests pin the two facts the decode relies on:
every residual stays inside the E2M1 range (no digit saturates), and the
rest is at most 6^-5 of the scale, below half an ulp of bf16 at the token's
largest value."""

import numpy as np
import pytest

from oracle import formats

PLANES = 6


def scale_exponent(amax: float) -> int:
    """Smallest e with amax <= 6 2^e (then amax 2^-e lies in (3, 6])."""
    m, e = np.frexp(np.float64(amax))  # amax = m 2^e, 0.5 <= m < 1
    return int(e) - 2 if m > 0.75 else int(e) - 3


def digits(x: np.ndarray):
    """Digit values [PLANES, n] and the final residual of one token."""
    amax = float(np.max(np.abs(x)))
    e = scale_exponent(amax) if amax > 0 else 0
    r = (x.astype(np.float64) * 2.0 ** -e).astype(np.float32)
    out = []
    for _ in range(PLANES):
        assert np.all(np.abs(r) <= 6.0)
        d = formats.e2m1_value(formats.e2m1_rne(r)).astype(np.float32)
        out.append(d)
        r = ((r - d) * np.float32(6.0)).astype(np.float32)
    return np.array(out), r, e


def _tokens():
    g = np.random.default_rng(11)
    yield g.standard_normal(4096).astype(np.float32)
    yield (g.standard_normal(4096) * np.exp2(g.integers(-30, 30, 4096))).astype(np.float32)
    yield np.array([6.0, -6.0, 5.0, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25, 0.0], np.float32)
    yield np.array([3.0 + 2.0 ** -6, 3.0, 6.0 - 2.0 ** -5, 1e-38, -2e-39], np.float32)
    v = g.standard_normal(2048).astype(np.float32)
    v[17] = 3.0e4  # one outlier channel
    yield v


@pytest.mark.parametrize("i", range(5))
def test_residuals_in_range_and_rest_bounded(i):
    x = list(_tokens())[i]
    x = formats.bf16_rne(x).astype(np.float32)  # the decode's inputs are bf16
    d, rest, e = digits(x)
    scaled = x.astype(np.float64) * 2.0 ** -e
    approx = sum(d[p].astype(np.float64) * 6.0 ** -p for p in range(PLANES))
    err = np.abs(scaled - approx)
    assert np.all(err <= 6.0 ** -(PLANES - 1) + 1e-12)
    # the rest equals the last residual over 6^PLANES (each step exact or within an fp32 rounding)
    assert np.allclose(err, np.abs(rest.astype(np.float64)) * 6.0 ** -PLANES, rtol=1e-5, atol=1e-12)
    amax = np.max(np.abs(scaled))
    if amax > 0:
        assert 3.0 < amax <= 6.0


def test_scale_exponent_boundaries():
    assert scale_exponent(6.0) == 0       # 6 maps to 6
    assert scale_exponent(6.0001) == 1    # just above: halves to 3.00005
    assert scale_exponent(3.0) == -1      # 3 maps to 6
    assert scale_exponent(3.0001) == 0
    assert scale_exponent(1.0) == -2      # 1 maps to 4


def test_powers_of_two_are_single_digits():
    """+-2^k scales to +-4: one digit and no rest, the case the one-hot GPU
    test relies on for bit-exact outputs."""
    for k in range(-20, 20):
        d, rest, e = digits(np.array([2.0 ** k, -(2.0 ** k)], np.float32))
        assert np.array_equal(d[0], [4.0, -4.0]) and not np.any(d[1:]) and not np.any(rest)

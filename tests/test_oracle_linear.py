"""Pins for the oracle's W4A16 + LoRA linear: naive loops, closed forms, and the
acceptance tolerance itself."""

import numpy as np

from oracle import formats, linear, nvfp4


def _setup(rng, m=3, n=5, k=32, r=2):
    w = formats.bf16_rne(rng.standard_normal((n, k)) * 0.02)
    x = formats.bf16_rne(rng.standard_normal((m, k)))
    a = formats.bf16_rne(rng.standard_normal((r, k)) * 0.01)
    b = formats.bf16_rne(rng.standard_normal((n, r)) * 0.01)
    codes, scales, s_t = nvfp4.quantize(w)
    return x, w, a, b, codes, scales, s_t


def test_against_naive_loops(rng):
    x, w, a, b, codes, scales, s_t = _setup(rng)
    alpha = 4.0
    y = linear.linear_nvfp4_lora(x, codes, scales, s_t, a, b, alpha)
    c = nvfp4.unpack_nibbles(codes)
    m, k = x.shape
    n, r = b.shape
    for i in range(m):
        for j in range(n):
            acc = 0.0
            for kk in range(k):
                w_hat = formats.E2M1_VALUES[c[j, kk]] * formats.E4M3_VALUES[scales[j, kk // 16]] * float(s_t)
                acc += float(x[i, kk]) * w_hat
            lora = 0.0
            for q in range(r):
                t = sum(float(x[i, kk]) * float(a[q, kk]) for kk in range(k))
                lora += t * float(b[j, q])
            acc += alpha / r * lora
            assert abs(acc - y[i, j]) <= 1e-12 * (abs(acc) + 1e-6)


def test_closed_forms(rng):
    x, w, a, b, codes, scales, s_t = _setup(rng, m=4, n=6, k=64, r=3)
    w_hat = nvfp4.dequantize(codes, scales, s_t)
    # x = 0 -> y = 0
    assert not linear.linear_nvfp4_lora(np.zeros_like(x), codes, scales, s_t, a, b, 2.0).any()
    # alpha = 0, A = 0 or B = 0 -> plain W4A16
    base = x.astype(np.float64) @ w_hat.T
    assert np.allclose(linear.linear_nvfp4_lora(x, codes, scales, s_t, a, b, 0.0), base, rtol=0, atol=1e-15)
    assert np.array_equal(linear.linear_nvfp4_lora(x, codes, scales, s_t, np.zeros_like(a), b, 2.0), base)
    assert np.array_equal(linear.linear_nvfp4_lora(x, codes, scales, s_t, None, None, 2.0), base)
    # one-hot x = e_k -> y[:, n] = w_hat[n, k] + (alpha/r) sum_j A[j, k] B[n, j]
    k0 = 37
    e = np.zeros((1, 64), np.float32)
    e[0, k0] = 1.0
    y = linear.linear_nvfp4_lora(e, codes, scales, s_t, a, b, 3.0)
    want = w_hat[:, k0] + 3.0 / 3 * (b.astype(np.float64) @ a[:, k0].astype(np.float64))
    assert np.allclose(y[0], want, rtol=1e-14, atol=0)
    # W = 0 -> LoRA term only
    zc, zs, zt = nvfp4.quantize(np.zeros_like(w))
    y = linear.linear_nvfp4_lora(x, zc, zs, zt, a, b, 2.0)
    want = 2.0 / 3 * (x.astype(np.float64) @ a.T.astype(np.float64)) @ b.T.astype(np.float64)
    assert np.allclose(y, want, rtol=1e-14, atol=0)


def test_rows_match_full(rng):
    x, w, a, b, codes, scales, s_t = _setup(rng, m=5, n=9, k=64, r=4)
    full = linear.linear_nvfp4_lora(x, codes, scales, s_t, a, b, 8.0)
    w_hat = nvfp4.dequantize(codes, scales, s_t)
    rows = [1, 4]
    cols = [0, 8, 3]
    part = linear.linear_rows(x[rows], w_hat[cols], a, b[cols], 8.0)
    assert np.allclose(part, full[np.ix_(rows, cols)], rtol=1e-14, atol=1e-18)


def test_tolerance_gate(rng):
    y_ref = rng.standard_normal((8, 64))
    assert linear.within_tolerance(y_ref, y_ref)[0]
    assert linear.within_tolerance(formats.bf16_rne(y_ref), y_ref)[0]  # bf16 output rounding passes
    assert not linear.within_tolerance(y_ref * 1.01, y_ref)[0]  # 1% scale error fails
    bad = y_ref.copy()
    bad[3, 5] += 0.5
    assert not linear.within_tolerance(bad, y_ref)[0]  # one wrong element fails
    nan = y_ref.copy()
    nan[0, 0] = np.nan
    assert not linear.within_tolerance(nan, y_ref)[0]

"""Pins of the LoRA backward oracle: central finite differences of the
forward oracle's loss L = sum(y * dY) (an independent route to every
gradient), naive loops for dX, and closed forms (dY = 0, alpha = 0, A = 0,
B = 0, one-hot dY), plus planted mistakes."""

import numpy as np
import pytest

import oracle
from oracle import linear, lora_backward as lb, nvfp4
from oracle.formats import bf16_rne


def _case(seed, m=5, n=32, k=64, r=4):
    g = np.random.default_rng(seed)
    w = bf16_rne((g.standard_normal((n, k)) * 0.05).astype(np.float32))
    codes, scales, s_t = nvfp4.quantize(w)
    x = bf16_rne(g.standard_normal((m, k)).astype(np.float32))
    a = bf16_rne((g.standard_normal((r, k)) * 0.1).astype(np.float32))
    b = bf16_rne((g.standard_normal((n, r)) * 0.1).astype(np.float32))
    dy = bf16_rne(g.standard_normal((m, n)).astype(np.float32))
    return dy, x, codes, scales, s_t, a, b, 2.0 * r


def _loss(dy, x, codes, scales, s_t, a, b, alpha):
    return float(np.sum(linear.linear_nvfp4_lora(x, codes, scales, s_t, a, b, alpha) * dy))


def test_finite_differences():
    dy, x, codes, scales, s_t, a, b, alpha = _case(0)
    dx, da, db = lb.lora_backward(dy, x, codes, scales, s_t, a, b, alpha)
    h = 1e-4
    g = np.random.default_rng(1)
    for name, arr, grad in (("x", x, dx), ("a", a, da), ("b", b, db)):
        for _ in range(12):
            idx = tuple(g.integers(0, s) for s in arr.shape)
            plus = np.array(arr, np.float64)
            minus = np.array(arr, np.float64)
            plus[idx] += h
            minus[idx] -= h
            args = {"x": x, "a": a, "b": b}
            args[name] = plus
            lp = _loss(dy, args["x"], codes, scales, s_t, args["a"], args["b"], alpha)
            args[name] = minus
            lm = _loss(dy, args["x"], codes, scales, s_t, args["a"], args["b"], alpha)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_dx_naive_loops():
    dy, x, codes, scales, s_t, a, b, alpha = _case(2, m=3, n=16, k=32, r=2)
    w_hat = nvfp4.dequantize(codes, scales, s_t)
    dx, _, _ = lb.lora_backward(dy, x, codes, scales, s_t, a, b, alpha)
    m, n = dy.shape
    k = x.shape[1]
    r = a.shape[0]
    for i in range(m):
        for kk in range(k):
            acc = 0.0
            for nn in range(n):
                acc += float(dy[i, nn]) * float(w_hat[nn, kk])
            lora = 0.0
            for j in range(r):
                u = sum(float(dy[i, nn]) * float(b[nn, j]) for nn in range(n))
                lora += u * float(a[j, kk])
            ref = acc + alpha / r * lora
            assert abs(dx[i, kk] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_closed_forms():
    dy, x, codes, scales, s_t, a, b, alpha = _case(3)
    dx, da, db = lb.lora_backward(np.zeros_like(dy), x, codes, scales, s_t, a, b, alpha)
    assert not dx.any() and not da.any() and not db.any()
    dx, da, db = lb.lora_backward(dy, x, codes, scales, s_t, a, b, 0.0)
    assert not da.any() and not db.any()
    assert np.allclose(dx, dy.astype(np.float64) @ nvfp4.dequantize(codes, scales, s_t), rtol=0, atol=1e-12)
    _, _, db = lb.lora_backward(dy, x, codes, scales, s_t, np.zeros_like(a), b, alpha)
    assert not db.any()
    _, da, _ = lb.lora_backward(dy, x, codes, scales, s_t, a, np.zeros_like(b), alpha)
    assert not da.any()
    # one-hot dY: dX row = W_hat row n0 + (alpha/r) B[n0] . A; dB row n0 = (alpha/r) x_m . A^T
    oh = np.zeros_like(dy)
    oh[1, 7] = 1.0
    dx, da, db = lb.lora_backward(oh, x, codes, scales, s_t, a, b, alpha)
    c = alpha / a.shape[0]
    w_hat = nvfp4.dequantize(codes, scales, s_t)
    assert np.allclose(dx[1], w_hat[7] + c * (b[7].astype(np.float64) @ a), rtol=0, atol=1e-12)
    assert np.allclose(db[7], c * (x[1].astype(np.float64) @ a.T.astype(np.float64)), rtol=0, atol=1e-12)
    assert not np.delete(db, 7, axis=0).any()


def test_no_adapter():
    dy, x, codes, scales, s_t, a, b, alpha = _case(4)
    dx, da, db = lb.lora_backward(dy, x, codes, scales, s_t, None, None, 0.0)
    assert da is None and db is None
    assert np.allclose(dx, lb.lora_backward_dx_rows(dy, nvfp4.dequantize(codes, scales, s_t), None, None, 0.0))


@pytest.mark.parametrize("mutation", ["transpose_b", "scale", "drop_lora"])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    orig = lb.lora_backward

    def bad(dy, x, codes, scales, s_t, a, b, alpha):
        dx, da, db = orig(dy, x, codes, scales, s_t, a, b, alpha)
        if mutation == "transpose_b":  # dB from dY . t without the transpose, reshaped
            db = np.asarray(db)[::-1]
        elif mutation == "scale":
            da = 2.0 * da
        else:
            dx = dy.astype(np.float64) @ nvfp4.dequantize(codes, scales, s_t)
        return dx, da, db

    monkeypatch.setattr(lb, "lora_backward", bad)
    with pytest.raises(AssertionError):
        test_finite_differences()


def test_package_exports_module():
    assert oracle.lora_backward is lb

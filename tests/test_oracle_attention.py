"""Pins of the FP8-KV decode attention oracle: closed forms (one cached token
returns its value row; equal keys average the values; a dominant score picks
its row), brute force in plain Python on tiny cases, permutation invariance
over cached tokens, the grouped-query head mapping, the cache rows' 1x128
quantization against the FP8 activation quantizer, and planted mistakes."""

import math

import numpy as np
import pytest

from oracle import attention as att
from oracle import fp8
from oracle.formats import bf16_rne


def _cache(g, b, hkv, lmax, d=128, scale=1.0):
    k = bf16_rne((g.standard_normal((b, hkv, lmax, d)) * scale).astype(np.float32))
    v = bf16_rne((g.standard_normal((b, hkv, lmax, d)) * scale).astype(np.float32))
    kq, ks = att.kv_quantize(k)
    vq, vs = att.kv_quantize(v)
    return kq, ks, vq, vs


def test_kv_rows_follow_the_1x128_rule():
    g = np.random.default_rng(0)
    rows = bf16_rne(g.standard_normal((2, 3, 5, 128)).astype(np.float32))
    for mode in (0, 1):
        q, s = att.kv_quantize(rows, mode)
        rq, rs = fp8.quantize_a1x128(rows.reshape(-1, 128), mode)
        assert np.array_equal(q.reshape(-1, 128), rq) and np.array_equal(s.reshape(-1), rs.reshape(-1))


def test_single_token_returns_its_value():
    g = np.random.default_rng(1)
    kq, ks, vq, vs = _cache(g, 2, 2, 4)
    q = bf16_rne(g.standard_normal((2, 8, 128)).astype(np.float32))
    o = att.attention_decode(q, kq, ks, vq, vs, np.array([1, 1]))
    v0 = att.kv_dequantize(vq[:, :, 0], vs[:, :, 0])  # [B, Hkv, d]
    for h in range(8):
        assert np.allclose(o[:, h], v0[:, h // 4], rtol=0, atol=1e-12)


def test_equal_keys_average_values_and_dominant_score_selects():
    g = np.random.default_rng(2)
    kq, ks, vq, vs = _cache(g, 1, 1, 6)
    kq[:] = kq[:, :, :1]
    ks[:] = ks[:, :, :1]
    q = bf16_rne(g.standard_normal((1, 2, 128)).astype(np.float32))
    o = att.attention_decode(q, kq, ks, vq, vs, np.array([6]))
    mean_v = att.kv_dequantize(vq[0, 0], vs[0, 0]).mean(axis=0)
    assert np.allclose(o[0, 0], mean_v, rtol=0, atol=1e-12)
    # a key aligned with a large query dominates the softmax
    kq2, ks2, vq2, vs2 = _cache(g, 1, 1, 5, scale=0.01)
    qq = np.zeros((1, 1, 128), np.float32)
    qq[0, 0, 0] = 100.0
    kd = np.zeros((1, 1, 5, 128), np.float32)
    kd[0, 0, 3, 0] = 100.0
    kq2, ks2 = att.kv_quantize(kd)
    o2 = att.attention_decode(qq, kq2, ks2, vq2, vs2, np.array([5]))
    assert np.allclose(o2[0, 0], att.kv_dequantize(vq2[0, 0, 3], vs2[0, 0, 3]), rtol=0, atol=1e-12)


def test_brute_force_tiny():
    g = np.random.default_rng(3)
    kq, ks, vq, vs = _cache(g, 1, 2, 3)
    q = bf16_rne(g.standard_normal((1, 4, 128)).astype(np.float32))
    o = att.attention_decode(q, kq, ks, vq, vs, np.array([3]))
    kv = att.kv_dequantize(kq, ks)
    vv = att.kv_dequantize(vq, vs)
    for h in range(4):
        gg = h // 2
        sc = [sum(float(q[0, h, i]) * float(kv[0, gg, t, i]) for i in range(128)) / math.sqrt(128) for t in range(3)]
        mx = max(sc)
        w = [math.exp(s - mx) for s in sc]
        z = sum(w)
        for i in range(0, 128, 17):
            ref = sum(w[t] / z * float(vv[0, gg, t, i]) for t in range(3))
            assert abs(o[0, h, i] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_token_order_does_not_matter_and_lengths_cut():
    g = np.random.default_rng(4)
    kq, ks, vq, vs = _cache(g, 1, 1, 7)
    q = bf16_rne(g.standard_normal((1, 1, 128)).astype(np.float32))
    perm = g.permutation(7)
    o1 = att.attention_decode(q, kq, ks, vq, vs, np.array([7]))
    o2 = att.attention_decode(q, kq[:, :, perm], ks[:, :, perm], vq[:, :, perm], vs[:, :, perm], np.array([7]))
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-12)
    # tokens past the length are never read
    kq2 = kq.copy()
    kq2[:, :, 5:] = 0x7E  # 448
    assert np.allclose(att.attention_decode(q, kq, ks, vq, vs, np.array([5])),
                       att.attention_decode(q, kq2, ks, vq, vs, np.array([5])), rtol=0, atol=0)
    assert not att.attention_decode(q, kq, ks, vq, vs, np.array([0])).any()


@pytest.mark.parametrize("mutation", ["no_sqrt", "head_map"])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    orig = att.attention_decode
    if mutation == "no_sqrt":
        def bad(q, kq, ks, vq, vs, lens):
            return orig(np.asarray(q, np.float64) * np.sqrt(128.0), kq, ks, vq, vs, lens)
        monkeypatch.setattr(att, "attention_decode", bad)
        with pytest.raises(AssertionError):
            test_brute_force_tiny()
    else:
        def bad(q, kq, ks, vq, vs, lens):  # query head h reads KV head h % Hkv
            q = np.asarray(q)
            hq, hkv = q.shape[1], kq.shape[1]
            perm = np.array([(h % hkv) * (hq // hkv) + h // hkv for h in range(hq)])
            return orig(q[:, perm], kq, ks, vq, vs, lens)[:, np.argsort(perm)]
        monkeypatch.setattr(att, "attention_decode", bad)
        with pytest.raises(AssertionError):
            test_single_token_returns_its_value()

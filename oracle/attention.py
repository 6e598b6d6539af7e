"""Decode attention over an FP8 (E4M3) key/value cache, in float64.

Test infrastructure only (see the package docstring).

What it follows.  NVIDIA's FP8 recipe for RL ("NVIDIA NeMo RL behaalt 48%
snelheidswinst met end-to-end FP8-precisietraining", section "Praktische
prestatiewinsten") extends FP8 from the linear layers to the KV cache and the
attention operations, which takes the speedup from 15-25 % to about 48 %; the
recipe's activations are quantized blockwise in 1x128 blocks to E4M3 (section
"De technische doorbraak").  The page gives no further detail.  Readings:

* the cache holds each key and value row (one token, one KV head,
  head_dim = 128 values) as E4M3 codes with one fp32 scale per row -- the
  recipe's 1x128 activation rule (``fp8.quantize_a1x128``), in either scale
  mode;
* decode attention (one new query token per sequence, grouped-query heads:
  query head h reads KV head h // (Hq / Hkv)) is
  ``o = softmax(q . K^T / sqrt(d)) . V`` over the sequence's cached tokens,
  with K and V the dequantized cache (code value x row scale) and q in bf16;
* layout: cache [B][Hkv][Lmax][d] bytes, scales [B][Hkv][Lmax] fp32,
  q and o [B][Hq][d] bf16, lens [B] cached tokens per sequence.

Everything is float64 on the exact dequantized values.
"""

import numpy as np

from . import fp8
from .formats import e4m3_value


def kv_quantize(rows: np.ndarray, mode: int = fp8.SCALE_FP32):
    """E4M3 codes and per-row scales of rows [..., 128] (the 1x128 rule)."""
    rows = np.asarray(rows, np.float32)
    shape = rows.shape
    q, s = fp8.quantize_a1x128(rows.reshape(-1, shape[-1]), mode)
    return q.reshape(shape), s.reshape(shape[:-1])


def kv_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    return e4m3_value(codes) * np.asarray(scales, np.float64)[..., None]


def attention_decode(q, k_codes, k_scales, v_codes, v_scales, lens) -> np.ndarray:
    """o [B, Hq, d] float64 for q [B, Hq, d] and caches [B, Hkv, Lmax, d]."""
    q = np.asarray(q, np.float64)
    b_, hq, d = q.shape
    hkv = k_codes.shape[1]
    group = hq // hkv
    out = np.zeros((b_, hq, d), np.float64)
    for b in range(b_):
        n = int(lens[b])
        if n == 0:
            continue
        for h in range(hq):
            g = h // group
            k = kv_dequantize(k_codes[b, g, :n], k_scales[b, g, :n])
            v = kv_dequantize(v_codes[b, g, :n], v_scales[b, g, :n])
            s = (k @ q[b, h]) / np.sqrt(d)
            p = np.exp(s - s.max())
            out[b, h] = (p / p.sum()) @ v
    return out

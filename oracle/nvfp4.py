"""NVFP4 quantization and dequantization of one BF16 weight matrix.

Test infrastructure only (see the package docstring).

What it follows.  QeRL keeps the policy's weights in 4-bit NVFP4 ("QeRL:
Beyond Efficiency -- Quantization-enhanced Reinforcement Learning for LLMs",
abstract; "NVIDIA and MIT Collaborate on QeRL", the paragraph after Key
Features: the weight path moves to NVFP4).  The NVFP4 layout is the standard
one, which the pages name but do not spell out:

* one FP32 scale for the whole tensor, ``s_t``;
* one E4M3 scale ``s_b`` per 16 consecutive elements of a row (along K);
* one E2M1 code per element; element (n, k) decodes to
  ``e2m1(code) * e4m3(s_b) * s_t``.

Readings taken where the pages are silent:

* ``s_t = amax_t / (6 * 448)`` so that the largest block scale lands on the
  top of the E4M3 range (6 is the E2M1 maximum, 448 the E4M3 maximum);
* ``s_b = e4m3_rne(amax_b / (6 * s_t))``;
* ``d_b = e4m3(s_b) * s_t`` and ``code = e2m1_rne(x / d_b)``;
* every one of these is a single IEEE float32 operation, correctly rounded
  (division, not multiplication by a reciprocal), and the E2M1 decision is
  taken on the float32 quotient;
* an all-zero tensor gives ``s_t = 0``; a block whose ``d_b`` is zero gets
  all-zero codes (0x0) and no division;
* codes are packed two per byte, the element with the even K index in the
  low nibble.
"""

import numpy as np

from .formats import e2m1_rne, e4m3_rne, e2m1_value, e4m3_value

BLOCK = 16
TENSOR_SCALE_DIVISOR = np.float32(6.0 * 448.0)  # 2688


def tensor_scale(amax_t) -> np.float32:
    """s_t = fp32(amax_t / 2688)."""
    return np.float32(np.float32(amax_t) / TENSOR_SCALE_DIVISOR)


def block_scale_codes(amax_b: np.ndarray, s_t: np.float32) -> np.ndarray:
    """E4M3 byte of each block scale: e4m3_rne(fp32(amax_b / fp32(6 * s_t)))."""
    amax_b = np.asarray(amax_b, dtype=np.float32)
    if s_t == 0:
        return np.zeros(amax_b.shape, dtype=np.uint8)
    six_st = np.float32(np.float32(6.0) * s_t)
    ratio = (amax_b / six_st).astype(np.float32)
    return e4m3_rne(ratio)


def block_divisor(sb_codes: np.ndarray, s_t: np.float32) -> np.ndarray:
    """d_b = fp32(e4m3(s_b) * s_t)."""
    return (e4m3_value(sb_codes).astype(np.float32) * np.float32(s_t)).astype(np.float32)


def element_codes(blocks: np.ndarray, d_b: np.ndarray) -> np.ndarray:
    """E2M1 code of every element of ``blocks`` [..., 16] given d_b [...]."""
    blocks = np.asarray(blocks, dtype=np.float32)
    d = np.asarray(d_b, dtype=np.float32)[..., None]
    safe = np.where(d > 0, d, np.float32(1.0))
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (blocks / safe).astype(np.float32)
    codes = e2m1_rne(q)
    return np.where(d > 0, codes, np.uint8(0)).astype(np.uint8)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[..., K] 4-bit codes -> [..., K/2] bytes, even K index in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def quantize(w: np.ndarray):
    """Quantize a bf16-valued float32 matrix W [N, K] (K a multiple of 16).

    Returns ``(codes uint8 [N, K/2], scales uint8 [N, K/16], s_t float32)``.
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % BLOCK:
        raise ValueError("K must be a multiple of 16")
    amax_t = np.float32(np.max(np.abs(w))) if w.size else np.float32(0)
    s_t = tensor_scale(amax_t)
    blocks = w.reshape(n, k // BLOCK, BLOCK)
    if s_t == 0:
        return (np.zeros((n, k // 2), np.uint8), np.zeros((n, k // BLOCK), np.uint8), s_t)
    amax_b = np.max(np.abs(blocks), axis=-1)
    sb = block_scale_codes(amax_b, s_t)
    d_b = block_divisor(sb, s_t)
    codes = element_codes(blocks, d_b).reshape(n, k)
    return pack_nibbles(codes), sb, s_t


def quantize_rows(w_rows: np.ndarray, s_t: np.float32):
    """Codes and scales of some rows of a tensor whose tensor scale is s_t.

    For checking sampled rows of a large tensor: ``s_t`` comes from the whole
    tensor's absmax (``tensor_scale(max|W|)``), the rows are then encoded
    exactly as ``quantize`` does.
    """
    w_rows = np.asarray(w_rows, dtype=np.float32)
    n, k = w_rows.shape
    if s_t == 0:
        return np.zeros((n, k // 2), np.uint8), np.zeros((n, k // BLOCK), np.uint8)
    blocks = w_rows.reshape(n, k // BLOCK, BLOCK)
    sb = block_scale_codes(np.max(np.abs(blocks), axis=-1), s_t)
    codes = element_codes(blocks, block_divisor(sb, s_t)).reshape(n, k)
    return pack_nibbles(codes), sb


def dequantize(codes: np.ndarray, scales: np.ndarray, s_t) -> np.ndarray:
    """W_hat [N, K] in float64: e2m1(code) * e4m3(s_b) * s_t (exact in float64)."""
    c = unpack_nibbles(codes)
    n, k = c.shape
    vals = e2m1_value(c).reshape(n, k // BLOCK, BLOCK)
    sb = e4m3_value(scales)[..., None]
    return (vals * sb * np.float64(np.float32(s_t))).reshape(n, k)

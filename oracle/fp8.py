"""Blockwise E4M3 (FP8) quantization and the blockwise-scaled FP8 GEMM.

Test infrastructure only (see the package docstring).

What it follows.  NVIDIA's FP8 recipe for RL ("NVIDIA NeMo RL behaalt 48%
snelheidswinst met end-to-end FP8-precisietraining", section "De technische
doorbraak") quantizes blockwise to E4M3 with 128x128 tiles for weights and
1x128 row blocks for activations, runs the linear layers in FP8, and (last
paragraph before "Waarom dit belangrijk is") offers power-of-two scale factors
as an option.

Readings taken where the page is silent:

* one scale per tile (weights) or per 1x128 row block (activations), stored
  as float32; the code of element x is ``e4m3_rne(x / s)``;
* FP32 scales: ``s = fp32(amax / 448)`` and the quotient ``fp32(x / s)`` is a
  correctly-rounded float32 division;
* power-of-two scales: ``s = 2^e`` with e the smallest integer such that
  ``2^e >= fp32(amax / 448)``; ``x * 2^-e`` is then exact and is rounded once;
* a tile whose amax is 0 gets ``s = 0`` and all-zero codes (0x00);
* weight tiles are counted ``ceil(N/128) x K/128``, the last tile row may be
  short; K must be a multiple of 128;
* the GEMM is ``y[m, n] = sum_kb sa[m, kb] * sw[n // 128, kb] *
  sum_{k in kb} e4m3(qa[m, k]) * e4m3(qw[n, k])`` formed in float64.
"""

import numpy as np

from .formats import e4m3_rne, e4m3_value

TILE = 128
FP8_MAX = np.float32(448.0)
SCALE_FP32 = 0
SCALE_POW2 = 1


def scale_of(amax, mode: int) -> np.ndarray:
    """Block scale(s) for the given block absmax value(s) (float32)."""
    amax = np.asarray(amax, dtype=np.float32)
    v = (amax / FP8_MAX).astype(np.float32)
    if mode == SCALE_FP32:
        return v
    if mode != SCALE_POW2:
        raise ValueError("unknown scale mode")
    m, e = np.frexp(v.astype(np.float64))  # v = m * 2^e with 0.5 <= m < 1
    e = np.where(m == 0.5, e - 1, e)  # exact powers of two keep their exponent
    s = np.ldexp(1.0, e)
    return np.where(v == 0, 0.0, s).astype(np.float32)


def _codes(block: np.ndarray, s: np.ndarray, mode: int) -> np.ndarray:
    """E4M3 codes of ``block`` [..., L] with scales ``s`` [...]."""
    block = np.asarray(block, dtype=np.float32)
    s32 = np.asarray(s, dtype=np.float32)[..., None]
    safe = np.where(s32 > 0, s32, np.float32(1.0))
    if mode == SCALE_FP32:
        q = (block / safe).astype(np.float32)  # one float32 division
    else:
        _, e = np.frexp(safe.astype(np.float64))
        q = np.ldexp(block.astype(np.float64), -(e - 1))  # x * 2^-e, exact
    codes = e4m3_rne(q)
    return np.where(s32 > 0, codes, np.uint8(0)).astype(np.uint8)


def quantize_a1x128(x: np.ndarray, mode: int = SCALE_FP32):
    """Activations x [M, K] (bf16-valued float32), K % 128 == 0.

    Returns ``(q uint8 [M, K], s float32 [M, K/128])``.
    """
    x = np.asarray(x, dtype=np.float32)
    m, k = x.shape
    if k % TILE:
        raise ValueError("K must be a multiple of 128")
    blocks = x.reshape(m, k // TILE, TILE)
    amax = np.max(np.abs(blocks), axis=-1) if x.size else np.zeros((m, k // TILE), np.float32)
    s = scale_of(amax, mode)
    q = _codes(blocks, s, mode).reshape(m, k)
    return q, s


def quantize_w128x128(w: np.ndarray, mode: int = SCALE_FP32):
    """Weights W [N, K] (bf16-valued float32), K % 128 == 0, any N >= 0.

    Returns ``(q uint8 [N, K], s float32 [ceil(N/128), K/128])``.
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % TILE:
        raise ValueError("K must be a multiple of 128")
    nt = -(-n // TILE)
    q = np.zeros((n, k), dtype=np.uint8)
    s = np.zeros((nt, k // TILE), dtype=np.float32)
    for ti in range(nt):
        rows = w[ti * TILE:(ti + 1) * TILE]  # last tile may be short
        tiles = rows.reshape(rows.shape[0], k // TILE, TILE).transpose(1, 0, 2)  # [kb, r, 128]
        amax = np.max(np.abs(tiles.reshape(k // TILE, -1)), axis=-1)
        s[ti] = scale_of(amax, mode)
        codes = _codes(tiles.reshape(k // TILE, -1), s[ti], mode)
        q[ti * TILE:(ti + 1) * TILE] = codes.reshape(k // TILE, rows.shape[0], TILE).transpose(1, 0, 2).reshape(rows.shape[0], k)
    return q, s


def dequantize_a1x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    m, k = q.shape
    return (e4m3_value(q).reshape(m, k // TILE, TILE) * np.asarray(s, np.float64)[..., None]).reshape(m, k)


def dequantize_w128x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    n, k = q.shape
    row_s = np.repeat(np.asarray(s, np.float64), TILE, axis=0)[:n]  # [N, K/128]
    return (e4m3_value(q).reshape(n, k // TILE, TILE) * row_s[..., None]).reshape(n, k)


def gemm_blockwise(qa: np.ndarray, sa: np.ndarray, qw: np.ndarray, sw: np.ndarray) -> np.ndarray:
    """y [M, N] float64 = sum over 128-wide K blocks of sa * sw * (qa . qw)."""
    m, k = qa.shape
    n = qw.shape[0]
    va = e4m3_value(qa)
    vw = e4m3_value(qw)
    sw_rows = np.repeat(np.asarray(sw, np.float64), TILE, axis=0)[:n]  # [N, K/128]
    y = np.zeros((m, n), dtype=np.float64)
    for kb in range(k // TILE):
        ks = slice(kb * TILE, (kb + 1) * TILE)
        partial = va[:, ks] @ vw[:, ks].T  # exact: integer multiples of 2^-18, < 2^53
        y += np.asarray(sa, np.float64)[:, kb:kb + 1] * sw_rows[None, :, kb] * partial
    return y

"""Adaptive Quantization Noise (AQN): noise added to the policy's weights
before they are re-quantized, with a strength that changes over training.

Test infrastructure only (see the package docstring).

What it follows.  QeRL ("QeRL: Beyond Efficiency -- Quantization-enhanced
Reinforcement Learning for LLMs", Abstract; and the QeRL summary page,
"Enhancing Exploration through Quantization") finds that quantization noise
raises the policy's entropy and helps exploration, and adds an Adaptive
Quantization Noise mechanism that adjusts the noise during training.  The
pages give neither the noise's form nor its schedule.  Readings taken:

* the noise is zero-mean, of standard deviation sigma, added to every element
  of every bf16 master weight just before the weight is re-quantized:
  ``W' = bf16(fp32(W) + fp32(sigma * z))``, then W' is quantized as usual
  (NVFP4 or FP8), so the policy the rollout sees carries it;
* "adaptive" is a geometric schedule over the training steps s = 0 .. S-1,
  ``sigma_s = sigma_start * (sigma_end / sigma_start) ** (s / (S - 1))``
  (``sigma_end`` from step S - 1 on), computed in double precision and
  handed to the kernel as one fp32 number;
* z is drawn per element from the counter-based generator Philox4x32-10
  (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC'11):
  counter (e // 4 low word, e // 4 high word, tensor index j, step s), key
  (seed low word, seed high word); element e takes output word r[e % 4];
* z is the standardized sum of four uniforms (the Irwin-Hall
  approximation of a normal variable, variance 65535/65536, support within
  +-2 sqrt 3): the four bytes k_i of the word give
  ``z = fp32((k1 + k2 + k3 + k4 - 510) * 2^-8) * fp32(sqrt 3)``, each uniform
  being (k_i + 1/2) / 256.  It is chosen because every step is an integer
  operation or a single correctly-rounded fp32 operation, so the noise is
  reproducible bit for bit on any IEEE machine, and one generator call
  serves four elements.
"""

import numpy as np

from . import fp8 as _fp8
from . import nvfp4 as _nvfp4
from .formats import bf16_rne

M0, M1 = 0xD2511F53, 0xCD9E8D57  # Philox multipliers
W0, W1 = 0x9E3779B9, 0xBB67AE85  # Weyl increments of the key
SQRT3 = np.float32(np.sqrt(3.0))
MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds on arrays of 32-bit words (uint64 arithmetic)."""
    c = [np.asarray(x, np.uint64) & MASK for x in (c0, c1, c2, c3)]
    k0 = np.asarray(k0, np.uint64) & MASK
    k1 = np.asarray(k1, np.uint64) & MASK
    for _ in range(10):
        p0 = np.uint64(M0) * c[0]  # < 2^64: exact in uint64
        p1 = np.uint64(M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
        k0 = (k0 + np.uint64(W0)) & MASK
        k1 = (k1 + np.uint64(W1)) & MASK
    return [x.astype(np.uint32) for x in c]


def noise(n: int, seed: int, tensor: int, step: int, start: int = 0) -> np.ndarray:
    """z for elements start .. start + n - 1 of a tensor (float32)."""
    e = np.arange(start, start + n, dtype=np.uint64)
    quad = e >> np.uint64(2)
    r = philox4x32_10(quad & MASK, quad >> np.uint64(32), np.full_like(quad, tensor), np.full_like(quad, step),
                      np.uint64(seed) & MASK, np.uint64(seed) >> np.uint64(32))
    sel = (e & np.uint64(3)).astype(np.int64)
    w = np.choose(sel, r).astype(np.int64)
    ksum = (w & 0xFF) + ((w >> 8) & 0xFF) + ((w >> 16) & 0xFF) + (w >> 24)
    zc = ((ksum - 510).astype(np.float32) * np.float32(2.0 ** -8)).astype(np.float32)  # exact
    return (zc * SQRT3).astype(np.float32)


def sigma_at(step: int, steps: int, sigma_start: float, sigma_end: float) -> np.float32:
    """The schedule's sigma for a step, as the fp32 number a kernel receives."""
    if steps <= 1 or step >= steps - 1:
        return np.float32(sigma_end)
    return np.float32(sigma_start * (sigma_end / sigma_start) ** (step / (steps - 1)))


def noisy_weight(w: np.ndarray, sigma, seed: int, tensor: int, step: int) -> np.ndarray:
    """bf16(fp32(W) + fp32(sigma * z)) (float32 holding bf16 values)."""
    w = np.asarray(w, np.float32)
    z = noise(w.size, seed, tensor, step).reshape(w.shape)
    add = (np.float32(sigma) * z).astype(np.float32)
    return bf16_rne((w + add).astype(np.float32))


def requantize_aqn(weights, sigma, seed: int, step: int, fmt: str = "nvfp4", mode: int = 0):
    """Quantize every noisy master W'_j (tensor index j = list position)."""
    out = []
    for j, w in enumerate(weights):
        wn = noisy_weight(w, sigma, seed, j, step)
        out.append(_nvfp4.quantize(wn) if fmt == "nvfp4" else _fp8.quantize_w128x128(wn, mode))
    return out

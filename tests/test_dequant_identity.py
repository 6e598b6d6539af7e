"""The bf16 dequantization identity the prefill kernel relies on, checked
exhaustively on the host: for every E2M1 code v and every finite E4M3 block
scale s_b, the f16 bit pattern of v with its exponent and mantissa fields
shifted down three bits is the bf16 of v 2^-112, and the bf16 product of that
with bf16(s_b 2^112) equals v s_b exactly (NVFP4 element value times block
scale: the NVFP4 element decode, "QeRL: Beyond Efficiency -- Quantization-
enhanced Reinforcement Learning for LLMs", abstract)."""

import numpy as np

from oracle import formats


def _bf16_bits_to_f64(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def _f64_to_bf16_bits_exact(x):
    f = np.asarray(x, np.float32)
    assert np.array_equal(f.astype(np.float64), x), "not an fp32 value"
    bits = f.view(np.uint32)
    assert not np.any(bits & 0xFFFF), "not a bf16 value"
    return (bits >> 16).astype(np.uint32)


def test_e2m1_rebias_times_scale_is_exact():
    codes = np.arange(16, dtype=np.uint8)
    v = formats.e2m1_value(codes)                       # exact E2M1 values
    h = np.asarray(v, np.float16).view(np.uint16).astype(np.uint32)
    assert np.array_equal(np.asarray(v, np.float16).astype(np.float64), v)
    t = ((h & 0x7FFF) >> 3) | (h & 0x8000)              # one half of the packed step
    tv = _bf16_bits_to_f64(t)
    assert np.array_equal(tv, v * 2.0**-112)
    s = formats.e4m3_value(np.arange(256, dtype=np.uint8))
    s = s[np.isfinite(s)]
    s_bits = _f64_to_bf16_bits_exact(s * 2.0**112)      # the scale operand, exact in bf16
    prod = tv[:, None] * _bf16_bits_to_f64(s_bits)[None, :]
    # exact in float64; exactly representable in bf16, so a correctly rounded
    # bf16 multiply returns it unchanged, and every operand is a normal number
    _f64_to_bf16_bits_exact(prod)
    assert np.array_equal(prod, v[:, None] * s[None, :])
    nz = tv != 0
    assert np.all(np.abs(tv[nz]) >= 2.0**-126)


def test_packed_shift_does_not_leak_between_halves():
    codes = np.arange(16, dtype=np.uint8)
    h = np.asarray(formats.e2m1_value(codes), np.float16).view(np.uint16).astype(np.uint64)
    lo, hi = np.meshgrid(h, h, indexing="ij")
    w = (hi << 16) | lo
    t = ((w & 0x7FFF7FFF) >> 3) | (w & 0x80008000)
    want_lo = ((lo & 0x7FFF) >> 3) | (lo & 0x8000)
    want_hi = ((hi & 0x7FFF) >> 3) | (hi & 0x8000)
    assert np.array_equal(t & 0xFFFF, want_lo)
    assert np.array_equal(t >> 16, want_hi)

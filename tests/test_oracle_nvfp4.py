"""Pins for the oracle's NVFP4 quantizer: grid survival, the block-absmax
invariant, per-element brute force, exact-arithmetic agreement, error bounds
and the degenerate cases."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import formats, nvfp4


def _bf16(a):
    return formats.bf16_rne(np.asarray(a, np.float64))


def _random_w(rng, n, k, std=0.02, outliers=True):
    w = rng.standard_normal((n, k)) * std
    if outliers:
        idx = rng.choice(n * k, max(1, n * k // 1000), replace=False)
        w.reshape(-1)[idx] *= 20
    return _bf16(w)


def test_grid_survival(rng):
    """Entries already on the NVFP4 grid come back with the planted codes.

    With a tensor absmax of 2688 * 2^f the tensor scale is exactly 2^f.  A
    block whose entries are val(c) * S with absmax 6 * S gets the block scale
    S / 2^f exactly (S a power of two, or 448 * 2^f for the block holding the
    tensor absmax), and every entry divides back onto its planted code.
    """
    n, k, f = 8, 64, -3
    codes = rng.integers(0, 16, (n, k)).astype(np.uint8)
    blk = codes.reshape(n, k // 16, 16)
    blk[:, :, 0] = 7  # every block carries its absmax (+6) at slot 0
    S = 2.0 ** rng.integers(-8, 5, (n, k // 16)).astype(np.float64)  # S / 2^f in [2^-5, 2^7]
    S[0, 0] = 448.0 * 2.0 ** f  # this block holds the tensor absmax 2688 * 2^f
    w = (formats.e2m1_value(blk) * S[..., None]).reshape(n, k)
    assert np.max(np.abs(w)) == 2688.0 * 2.0 ** f
    assert formats.is_bf16_valued(w.astype(np.float32))
    packed, scales, s_t = nvfp4.quantize(w.astype(np.float32))
    assert s_t == np.float32(2.0 ** f)
    assert np.array_equal(scales, formats.e4m3_rne(S / 2.0 ** f))
    assert scales[0, 0] == 0x7E
    # -0.0 entries (code 0x8) keep their sign, +0.0 entries stay 0x0
    assert np.array_equal(nvfp4.unpack_nibbles(packed), codes)
    # dequantize -> quantize is the identity
    w_hat = nvfp4.dequantize(packed, scales, s_t)
    assert np.array_equal(w_hat, w)
    p2, s2, t2 = nvfp4.quantize(w_hat.astype(np.float32))
    assert np.array_equal(p2, packed) and np.array_equal(s2, scales) and t2 == s_t


def test_block_absmax_maps_to_six(rng):
    """Every block whose scale is normal has |code| = 7 (value 6) at its absmax.

    E4M3's relative half-step is at most 2^-4, so absmax / d_b >= 6 / (1 + 2^-4)
    > 5 (rounds to 6) or saturates.
    """
    w = _random_w(rng, 64, 256)
    packed, scales, s_t = nvfp4.quantize(w)
    codes = nvfp4.unpack_nibbles(packed).reshape(64, 16, 16)
    blocks = np.abs(w.reshape(64, 16, 16))
    arg = np.argmax(blocks, axis=-1)
    top = np.take_along_axis(codes, arg[..., None], axis=-1)[..., 0] & 7
    normal = scales >= 0x08
    assert normal.sum() > 0.9 * normal.size
    assert np.all(top[normal] == 7)


def test_tensor_absmax_block_scale_is_448(rng):
    w = _random_w(rng, 16, 128)
    _, scales, s_t = nvfp4.quantize(w)
    blocks = np.abs(w.reshape(16, 8, 16)).max(-1)
    i = np.unravel_index(np.argmax(blocks), blocks.shape)
    assert scales[i] == 0x7E
    assert s_t == np.float32(np.float32(np.abs(w).max()) / np.float32(2688.0))


def test_elementwise_bruteforce(rng):
    """Each code is the argmin over all 16 codes of |q - val(c)|, q = fp32(x / d_b)."""
    w = _random_w(rng, 6, 64)
    packed, scales, s_t = nvfp4.quantize(w)
    codes = nvfp4.unpack_nibbles(packed)
    d = (formats.e4m3_value(scales).astype(np.float32) * s_t).astype(np.float32)
    vals = formats.E2M1_VALUES
    for n in range(6):
        for k in range(64):
            q = float(np.float32(np.float32(w[n, k]) / d[n, k // 16]))
            sign = 8 if np.signbit(q) else 0
            best = None
            for c in range(sign, sign + 8):
                if abs(q) >= 6:
                    key = (0 if c & 7 == 7 else 1, 0)
                else:
                    key = (abs(q - vals[c]), c & 1)
                if best is None or key < best[0]:
                    best = (key, c)
            assert codes[n, k] == best[1], (n, k, q)


def test_exact_arithmetic_agreement(rng):
    """Against rounding the exact quotient x / d_b (rationals), the fp32
    quotient may only disagree where it sits within 1 ulp of a midpoint."""
    w = _random_w(rng, 8, 128)
    packed, scales, s_t = nvfp4.quantize(w)
    codes = nvfp4.unpack_nibbles(packed)
    d = (formats.e4m3_value(scales).astype(np.float32) * s_t).astype(np.float32)
    mids = [Fraction(m) for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)]
    grid = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    disagreements = 0
    for n in range(8):
        for k in range(128):
            q = Fraction(float(w[n, k])) / Fraction(float(d[n, k // 16]))
            a = abs(q)
            if a >= 6:
                mag = 7
            else:
                dist = [abs(a - g) for g in grid]
                best = min(dist)
                cands = [i for i, dd in enumerate(dist) if dd == best]
                mag = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
            if (codes[n, k] & 7) != mag:
                disagreements += 1
                q32 = np.float32(np.float32(w[n, k]) / d[n, k // 16])
                ulp = np.spacing(np.abs(q32))
                assert min(abs(float(abs(q32)) - float(m)) for m in mids) <= ulp
    assert disagreements <= 2


def test_error_bound(rng):
    """|x - w_hat| is at most half the E2M1 gap at x (times d_b) plus the
    float32 rounding of the quotient, or |x| - 6 d_b once it saturates."""
    w = _random_w(rng, 32, 256)
    packed, scales, s_t = nvfp4.quantize(w)
    w_hat = nvfp4.dequantize(packed, scales, s_t)
    d = np.repeat((formats.e4m3_value(scales) * np.float64(s_t)), 16, axis=1)
    q = np.abs(w) / d
    half_gap = np.where(q < 2, 0.25, np.where(q < 4, 0.5, 1.0))
    bound = np.where(q > 6, np.abs(w) - 6 * d, half_gap * d) * (1 + 2.0 ** -20) + 1e-30
    assert np.all(np.abs(w - w_hat) <= bound)
    # and it is small in the norm: NVFP4 keeps ~2 significant bits
    rel = np.linalg.norm(w - w_hat) / np.linalg.norm(w)
    assert 0.01 < rel < 0.2


def test_dequant_is_exact_in_bf16(rng):
    """e2m1(code) * e4m3(s_b) has at most 6 significant bits: exact in bf16."""
    w = _random_w(rng, 16, 256)
    packed, scales, _ = nvfp4.quantize(w)
    c = nvfp4.unpack_nibbles(packed)
    prod = formats.e2m1_value(c).reshape(16, 16, 16) * formats.e4m3_value(scales)[..., None]
    assert np.array_equal(formats.bf16_rne(prod).astype(np.float64), prod)


def test_all_zero_and_signed_zero():
    w = np.zeros((4, 32), np.float32)
    p, s, t = nvfp4.quantize(w)
    assert t == 0 and not p.any() and not s.any()
    w[1, 3] = -0.0
    p, s, t = nvfp4.quantize(w)
    assert t == 0 and not p.any()


def test_single_nonzero():
    w = np.zeros((2, 32), np.float32)
    w[1, 17] = -3.0
    p, s, t = nvfp4.quantize(w)
    codes = nvfp4.unpack_nibbles(p)
    assert t == np.float32(np.float32(3.0) / np.float32(2688.0))
    assert codes[1, 17] == 0xF and s[1, 1] == 0x7E
    assert np.count_nonzero(codes) == 1 and np.count_nonzero(s) == 1
    # zero entries of a live block stay +0 (code 0x0)
    assert codes[1, 16] == 0x0


def test_underflowing_block_scale():
    """A block far below the tensor absmax gets scale 0 and all-zero codes."""
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = 1000.0
    w[0, 16:] = 1e-6  # 1e-6 / (6 * 1000/2688) << 2^-10 -> s_b rounds to 0
    p, s, t = nvfp4.quantize(formats.bf16_rne(w))
    assert s[0, 1] == 0
    assert not nvfp4.unpack_nibbles(p)[0, 16:].any()


def test_nibble_order():
    w = np.zeros((1, 16), np.float32)
    w[0, 0] = 6.0   # even k -> low nibble
    w[0, 1] = -1.0  # odd k -> high nibble
    p, s, t = nvfp4.quantize(w)
    # s_t = 6/2688, block scale 448: d = 6/6 -> codes 6.0 -> 0x7, -1.0 -> 0xA
    assert p[0, 0] == (0x7 | (0xA << 4))


def test_quantize_rows_matches_full(rng):
    w = _random_w(rng, 40, 64)
    p, s, t = nvfp4.quantize(w)
    rows = np.array([0, 7, 39])
    pr, sr = nvfp4.quantize_rows(w[rows], t)
    assert np.array_equal(pr, p[rows]) and np.array_equal(sr, s[rows])


def test_k_must_be_multiple_of_16():
    with pytest.raises(ValueError):
        nvfp4.quantize(np.zeros((2, 20), np.float32))

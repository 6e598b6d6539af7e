"""Pins for the oracle's blockwise FP8 quantizers and GEMM: the library's own
float8 cast, grid survival, power-of-two scale properties, ragged tiles and a
naive-loop GEMM."""

import numpy as np
import torch

from oracle import formats, fp8


def _bf16(a):
    return formats.bf16_rne(np.asarray(a, np.float64))


def _acts(rng, m, k):
    x = rng.standard_normal((m, k))
    cols = rng.choice(k, max(1, k // 100), replace=False)
    x[:, cols] *= 10
    return _bf16(x)


def _torch_blocks(x_blocks, mode):
    """Library restatement on [B, L] blocks: torch float32 ops + float8 cast."""
    t = torch.from_numpy(np.ascontiguousarray(x_blocks, np.float32))
    amax = t.abs().amax(dim=1)
    v = amax / 448.0
    if mode == fp8.SCALE_FP32:
        s = v
        q = t / torch.where(s > 0, s, torch.ones_like(s))[:, None]
    else:
        m, e = torch.frexp(v.double())
        e = torch.where(m == 0.5, e - 1, e)
        s = torch.where(v > 0, torch.ldexp(torch.ones_like(v.double()), e), torch.zeros_like(v.double())).float()
        q = torch.ldexp(t.double(), -e[:, None].double())
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8)
    codes = torch.where((s > 0)[:, None], codes, torch.zeros_like(codes))
    return codes.numpy(), s.numpy()


def test_a1x128_matches_library(rng):
    x = _acts(rng, 33, 512)
    for mode in (fp8.SCALE_FP32, fp8.SCALE_POW2):
        q, s = fp8.quantize_a1x128(x, mode)
        lq, ls = _torch_blocks(x.reshape(-1, 128), mode)
        assert np.array_equal(s.reshape(-1), ls), mode
        assert np.array_equal(q.reshape(-1, 128), lq), mode


def test_w128x128_matches_library_ragged(rng):
    """N = 200: the second tile row is 72 rows high."""
    w = _bf16(rng.standard_normal((200, 256)) * 0.02)
    for mode in (fp8.SCALE_FP32, fp8.SCALE_POW2):
        q, s = fp8.quantize_w128x128(w, mode)
        assert s.shape == (2, 2)
        for ti, rows in enumerate((slice(0, 128), slice(128, 200))):
            for kb in range(2):
                tile = w[rows, kb * 128:(kb + 1) * 128]
                lq, ls = _torch_blocks(tile.reshape(1, -1), mode)
                assert s[ti, kb] == ls[0]
                assert np.array_equal(q[rows, kb * 128:(kb + 1) * 128].reshape(-1), lq[0])


def test_grid_survival(rng):
    """A tile holding e4m3 values times 2^e with absmax 448 * 2^e comes back exact."""
    codes = rng.integers(0, 256, (128, 128)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10  # no NaN codes
    codes[0, 0] = 0x7E  # 448
    e = -5
    w = formats.e4m3_value(codes) * 2.0 ** e
    for mode in (fp8.SCALE_FP32, fp8.SCALE_POW2):
        q, s = fp8.quantize_w128x128(w.astype(np.float32), mode)
        assert s[0, 0] == np.float32(2.0 ** e)
        assert np.array_equal(q, codes)
        assert np.array_equal(fp8.dequantize_w128x128(q, s), w)


def test_pow2_scale_properties(rng):
    amax = np.concatenate([rng.random(1000) * 10.0 ** rng.integers(-38, 38, 1000),
                           [448.0, 896.0, 1.0, 2.0 ** -133]]).astype(np.float32)
    s = fp8.scale_of(amax, fp8.SCALE_POW2).astype(np.float64)
    v = (amax / np.float32(448)).astype(np.float32).astype(np.float64)
    m, _ = np.frexp(s)
    assert np.all(m == 0.5)  # powers of two
    assert np.all(s >= v) and np.all(s / 2 < v)


def test_zero_blocks():
    x = np.zeros((2, 256), np.float32)
    x[1, 200] = 3.0
    for mode in (fp8.SCALE_FP32, fp8.SCALE_POW2):
        q, s = fp8.quantize_a1x128(x, mode)
        assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0 and s[1, 1] > 0
        assert not q[0].any() and not q[1, :128].any()
        # FP32: the block absmax lands on 448; POW2: s = 2^-7 >= 3/448, 3 * 2^7 = 384
        assert q[1, 200] == (0x7E if mode == fp8.SCALE_FP32 else 0x7C)


def test_absmax_maps_to_448_fp32(rng):
    x = _acts(rng, 8, 256)
    q, s = fp8.quantize_a1x128(x, fp8.SCALE_FP32)
    blocks = np.abs(x.reshape(8, 2, 128))
    arg = np.argmax(blocks, -1)
    top = np.take_along_axis(q.reshape(8, 2, 128), arg[..., None], -1)[..., 0] & 0x7F
    assert np.all(top == 0x7E)


def test_gemm_against_naive_loops(rng):
    m, n, k = 2, 131, 256  # two weight tile rows, the second one 3 rows high
    qa = rng.integers(0, 256, (m, k)).astype(np.uint8)
    qw = rng.integers(0, 256, (n, k)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0
    qw[(qw & 0x7F) == 0x7F] = 0
    sa = rng.random((m, 2)).astype(np.float32)
    sw = rng.random((2, 2)).astype(np.float32)
    y = fp8.gemm_blockwise(qa, sa, qw, sw)
    va, vw = formats.E4M3_VALUES[qa], formats.E4M3_VALUES[qw]
    for i in range(m):
        for j in range(n):
            acc = 0.0
            for kb in range(2):
                part = 0.0
                for kk in range(kb * 128, (kb + 1) * 128):
                    part += va[i, kk] * vw[j, kk]
                acc += float(sa[i, kb]) * float(sw[j // 128, kb]) * part
            assert abs(acc - y[i, j]) <= 1e-12 * (abs(acc) + 1)


def test_gemm_exact_integers():
    """Integer-valued codes with power-of-two scales: the result is an exact integer sum."""
    m, n, k = 4, 130, 256
    a = (np.arange(m * k).reshape(m, k) % 7 - 3).astype(np.float64)
    w = (np.arange(n * k).reshape(n, k) % 5 - 2).astype(np.float64)
    qa, qw = formats.e4m3_rne(a), formats.e4m3_rne(w)
    sa = np.full((m, 2), 0.5, np.float32)
    sw = np.full((2, 2), 4.0, np.float32)
    y = fp8.gemm_blockwise(qa, sa, qw, sw)
    assert np.array_equal(y, 2.0 * (a @ w.T))


def test_dequant_roundtrip_error(rng):
    x = _acts(rng, 16, 512)
    q, s = fp8.quantize_a1x128(x, fp8.SCALE_FP32)
    xh = fp8.dequantize_a1x128(q, s)
    # E4M3 keeps 4 significant bits: relative error <= 2^-4 for normal codes
    big = np.abs(x) > np.repeat(s, 128, axis=1) * 2.0 ** -6
    assert np.all(np.abs(x - xh)[big] <= 2.0 ** -4 * np.abs(x)[big] * (1 + 1e-6))

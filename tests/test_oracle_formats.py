"""Pins for the oracle's E2M1 / E4M3 rounding: hand-derived golden values,
brute-force search over all codes, and the library's own E4M3 conversion."""

import os

import numpy as np
import pytest
import torch

from oracle import formats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            v, c = line.split()
            rows.append((float(v), int(c, 16)))
    return rows


def test_e2m1_golden():
    for v, c in _load("e2m1_rounding.txt"):
        assert int(formats.e2m1_rne(np.float64(v))) == c, v


def test_e4m3_golden():
    for v, c in _load("e4m3_rounding.txt"):
        assert int(formats.e4m3_rne(np.float64(v))) == c, v


def test_e4m3_decode_matches_library():
    """All 256 E4M3FN bytes decode like torch.float8_e4m3fn."""
    codes = torch.arange(256, dtype=torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = formats.E4M3_VALUES
    assert np.array_equal(np.isnan(lib), np.isnan(ours))
    ok = ~np.isnan(lib)
    assert np.array_equal(lib[ok], ours[ok])
    assert np.array_equal(np.signbit(lib[ok]), np.signbit(ours[ok]))


def _brute(v, values, nonneg_count):
    """Argmin over all codes of the same sign, ties to the even code, saturate."""
    out = np.empty(len(v), dtype=np.uint8)
    top = values[nonneg_count - 1]
    sign_bit = nonneg_count if nonneg_count == 8 else 128
    for i, x in enumerate(v):
        a = abs(float(x))
        best, best_d = None, None
        if a >= top:
            best = nonneg_count - 1
        else:
            for c in range(nonneg_count):
                d = abs(a - values[c])
                if best is None or d < best_d or (d == best_d and c % 2 == 0):
                    best, best_d = c, d
        out[i] = best | (sign_bit if np.signbit(x) else 0)
    return out


def _probe_values(grid, rng, n_random):
    """Float32 midpoints of a grid, their neighbours, specials and randoms."""
    g = np.asarray(grid, np.float64)
    mids = (g[1:] + g[:-1]) / 2
    pts = [np.float32(0.0), np.float32(-0.0)]
    for m in np.concatenate([g, mids, [g[-1] * 1.03, g[-1] * 7.0]]):
        f = np.float32(m)
        pts.extend([f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))])
    base = np.array(pts, dtype=np.float32)
    base = np.concatenate([base, -base])
    rnd = rng.uniform(-1.2 * g[-1], 1.2 * g[-1], n_random).astype(np.float32)
    bits = rng.integers(0, 2**32, n_random, dtype=np.uint64).astype(np.uint32).view(np.float32)
    bits = bits[np.isfinite(bits)]
    return np.concatenate([base, rnd, bits])


def test_e2m1_against_bruteforce(rng):
    v = _probe_values(formats.E2M1_VALUES[:8], rng, 20000)
    assert np.array_equal(formats.e2m1_rne(v), _brute(v, formats.E2M1_VALUES, 8))


def test_e4m3_against_bruteforce(rng):
    v = _probe_values(formats.E4M3_VALUES[:127], rng, 3000)
    assert np.array_equal(formats.e4m3_rne(v), _brute(v, formats.E4M3_VALUES, 127))


def test_e4m3_rounding_matches_library_cast(rng):
    """Inside the finite range, RNE onto E4M3 equals torch's float8 cast.

    Dense sweep: 2^14 evenly spaced float32 bit patterns in every binade from
    2^-12 to 2^9, plus every midpoint and its float32 neighbours.
    """
    chunks = []
    for e in range(-12, 9):
        lo = np.float32(2.0 ** e).view(np.uint32)
        step = (1 << 23) // (1 << 14)
        chunks.append((lo + np.arange(0, 1 << 23, step, dtype=np.uint32)).view(np.float32))
    g = formats.E4M3_VALUES[:127]
    mids = ((g[1:] + g[:-1]) / 2).astype(np.float32)
    chunks += [mids, np.nextafter(mids, np.float32(1e9)), np.nextafter(mids, np.float32(0))]
    v = np.concatenate(chunks)
    v = v[np.abs(v) <= 448.0]
    v = np.concatenate([v, -v])
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(formats.e4m3_rne(v), lib)


def test_e4m3_saturates():
    v = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3e38], np.float32)
    assert np.all(formats.e4m3_rne(v) == 0x7E)
    assert np.all(formats.e4m3_rne(-v) == 0xFE)


def test_e2m1_decode_bits():
    # sign symmetry and monotone magnitudes straight from the bit fields
    vals = formats.E2M1_VALUES
    assert np.array_equal(vals[8:], -vals[:8])
    assert np.all(np.diff(vals[:8]) > 0)
    assert vals[7] == 6.0 and vals[1] == 0.5


def test_bf16_rne_matches_library(rng):
    """On float32 inputs (one rounding step in the library too), bf16_rne
    equals torch's bf16 cast, subnormals and ties included."""
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-40, 38, 100000),
                        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 2.0 ** -130])])
    x = x.astype(np.float32)
    lib = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    ours = formats.bf16_rne(x)
    fin = np.isfinite(lib)
    assert np.array_equal(lib[fin], ours[fin])


def test_nan_rejected():
    with pytest.raises(ValueError):
        formats.e2m1_rne(np.array([np.nan]))

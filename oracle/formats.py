"""E2M1 and E4M3 number formats: decode tables and round-to-nearest-even.

Test infrastructure only (see the package docstring).

The pages name the two element formats without defining them: 4-bit NVFP4
weights ("QeRL: Beyond Efficiency", abstract; "NVIDIA and MIT Collaborate on
QeRL", Key Features) and E4M3 FP8 ("NVIDIA NeMo RL behaalt 48%
snelheidswinst ...", section "De technische doorbraak").  The definitions
written out here are the standard ones:

* E2M1: 1 sign, 2 exponent, 1 mantissa bit.  Magnitude codes 0..7 mean
  0, 0.5, 1, 1.5, 2, 3, 4, 6.  Bit 3 is the sign.
* E4M3 ("FN" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
  infinities; 0x7F / 0xFF are NaN; largest finite 448; smallest normal 2^-6;
  subnormals m * 2^-9.

Rounding (reading of "round to nearest"): the input is rounded to the nearest
grid value; an exact tie goes to the code whose last bit is 0 (the even
mantissa); magnitudes beyond the largest finite value saturate to it; the sign
of the input is kept, so a negative input that rounds to zero gives the
negative-zero code.  NaN input is outside the contract.
"""

import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0


def e2m1_decode_table() -> np.ndarray:
    """Value of every 4-bit code 0..15 (float64), from the bit fields."""
    vals = np.zeros(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 0x8 else 1.0
        exp = (code >> 1) & 0x3
        man = code & 0x1
        if exp == 0:
            mag = 0.5 * man  # subnormal: m * 2^-1
        else:
            mag = (1.0 + 0.5 * man) * 2.0 ** (exp - 1)
        vals[code] = sign * mag
    return vals


def e4m3_decode_table() -> np.ndarray:
    """Value of every byte 0..255 as E4M3FN (float64, NaN for 0x7F/0xFF)."""
    vals = np.zeros(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp = (code >> 3) & 0xF
        man = code & 0x7
        if exp == 0xF and man == 0x7:
            vals[code] = np.nan
            continue
        if exp == 0:
            mag = man * 2.0 ** -9
        else:
            mag = (1.0 + man / 8.0) * 2.0 ** (exp - 7)
        vals[code] = sign * mag
    return vals


E2M1_VALUES = e2m1_decode_table()
E4M3_VALUES = e4m3_decode_table()

# Non-negative grids in code order (codes 0..7 and 0..126); both increase with
# the code, so a code's magnitude index is its position in the grid.
_E2M1_GRID = E2M1_VALUES[:8].copy()
_E4M3_GRID = E4M3_VALUES[:127].copy()


def _round_to_grid(v, grid: np.ndarray) -> np.ndarray:
    """Magnitude code of the nearest grid point to |v|, ties to the even code.

    ``grid`` holds the non-negative values of codes 0..len-1 in increasing
    order.  Values beyond the last grid point saturate to it.  Works on any
    real array; the comparisons are exact in float64 for float32 inputs.
    """
    a = np.abs(np.asarray(v, dtype=np.float64))
    if np.isnan(a).any():
        raise ValueError("NaN input is outside the rounding contract")
    top = len(grid) - 1
    hi = np.searchsorted(grid, a, side="left")  # grid[hi] >= a (or hi == len)
    hi = np.minimum(hi, top)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    pick_hi = d_hi < d_lo
    tie = d_hi == d_lo
    pick_hi = np.where(tie, (hi % 2) == 0, pick_hi)
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= grid[top], top, code)  # saturation (satfinite)
    code = np.where(a <= grid[0], 0, code)
    return code.astype(np.uint8)


def e2m1_rne(v) -> np.ndarray:
    """4-bit E2M1 code (uint8 0..15) of each value; see the module docstring."""
    v = np.asarray(v, dtype=np.float64)
    mag = _round_to_grid(v, _E2M1_GRID)
    sign = np.signbit(v).astype(np.uint8) << 3
    return (mag | sign).astype(np.uint8)


def e4m3_rne(v) -> np.ndarray:
    """E4M3FN byte of each value (satfinite, RNE, sign kept)."""
    v = np.asarray(v, dtype=np.float64)
    mag = _round_to_grid(v, _E4M3_GRID)
    sign = np.signbit(v).astype(np.uint8) << 7
    return (mag | sign).astype(np.uint8)


def e2m1_value(codes) -> np.ndarray:
    return E2M1_VALUES[np.asarray(codes, dtype=np.int64)]


def e4m3_value(codes) -> np.ndarray:
    return E4M3_VALUES[np.asarray(codes, dtype=np.int64)]


def is_bf16_valued(x: np.ndarray) -> bool:
    """True when every float32 value is exactly representable in bfloat16."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return bool(np.all((bits & 0xFFFF) == 0))


def bf16_rne(x) -> np.ndarray:
    """Round float64/float32 values to the nearest bfloat16 (ties to even).

    Returned as float32 holding bf16 values.  bfloat16 keeps 8 significant
    bits, exponents down to 2^-126 for normals and a fixed quantum of 2^-133
    below; the rounding is done once, from the float64 value.  Used only to
    state what a bf16 output of the exact result is; the method's outputs are
    compared by tolerance, not through this.
    """
    v = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(v)  # v = m * 2^e, 0.5 <= |m| < 1
    quantum_exp = np.maximum(e - 8, -133)  # 8 significant bits, then subnormal
    q = np.ldexp(np.rint(np.ldexp(v, -quantum_exp)), quantum_exp)  # rint: ties to even
    q = np.where(np.abs(q) > 3.3895313892515355e38, np.copysign(np.inf, v), q)
    return q.astype(np.float32)

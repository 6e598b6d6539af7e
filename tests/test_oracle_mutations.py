"""Plant plausible mistakes in the oracle (on the CPU, via monkeypatch) and check
that at least one pin catches each of them."""

import numpy as np
import pytest

import oracle.formats as formats
import oracle.fp8 as fp8
import oracle.linear as linear
import oracle.nvfp4 as nvfp4

from . import test_oracle_formats as tf
from . import test_oracle_fp8 as t8
from . import test_oracle_linear as tl
from . import test_oracle_nvfp4 as tn


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_tie_away_from_zero_is_caught(monkeypatch):
    def bad_round(v, grid):
        a = np.abs(np.asarray(v, np.float64))
        hi = np.minimum(np.searchsorted(grid, a, side="left"), len(grid) - 1)
        lo = np.maximum(hi - 1, 0)
        pick_hi = (grid[hi] - a) <= (a - grid[lo])  # ties up, not to even
        code = np.where(pick_hi, hi, lo)
        code = np.where(a >= grid[-1], len(grid) - 1, code)
        return np.where(a <= grid[0], 0, code).astype(np.uint8)

    monkeypatch.setattr(formats, "_round_to_grid", bad_round)
    _fails(tf.test_e2m1_golden)
    _fails(tf.test_e4m3_golden)


def test_wrong_tensor_scale_constant_is_caught(monkeypatch, rng):
    monkeypatch.setattr(nvfp4, "TENSOR_SCALE_DIVISOR", np.float32(448.0))
    _fails(tn.test_grid_survival, rng)


def test_swapped_nibbles_are_caught(monkeypatch):
    monkeypatch.setattr(nvfp4, "pack_nibbles", lambda c: (c[..., 1::2] | (c[..., 0::2] << 4)).astype(np.uint8))
    _fails(tn.test_nibble_order)


def test_missing_block_scale_in_divisor_is_caught(monkeypatch, rng):
    monkeypatch.setattr(nvfp4, "block_divisor", lambda sb, s_t: np.full(sb.shape, np.float32(s_t) * 64, np.float32))
    _fails(tn.test_grid_survival, rng)


def test_wrong_lora_scale_is_caught(monkeypatch, rng):
    orig = linear.lora_down
    monkeypatch.setattr(linear, "lora_down", lambda x, a: 2.0 * orig(x, a))
    _fails(tl.test_against_naive_loops, rng)


def test_fp8_scale_without_448_is_caught(monkeypatch, rng):
    monkeypatch.setattr(fp8, "FP8_MAX", np.float32(240.0))
    _fails(t8.test_a1x128_matches_library, rng)


def test_swapped_weight_scale_rows_are_caught(monkeypatch, rng):
    orig = fp8.gemm_blockwise
    monkeypatch.setattr(fp8, "gemm_blockwise", lambda qa, sa, qw, sw: orig(qa, sa, qw, np.asarray(sw)[::-1].copy()))
    _fails(t8.test_gemm_against_naive_loops, rng)

"""GPU parity of the power-of-two FP8 GEMM, which runs on the native
block-scaled MMA (tcgen05.mma kind::mxf8f6f4, UE8M0 scale bytes), against the
float64 oracle: exact-integer cases (the bf16 output must equal the rounding
of the exact result), ragged shapes, K lengths that wrap the scale ring, and
scales below or above the UE8M0 byte's reach, which the kernel carries by
shifting a K block's activation and weight exponents against each other.
The full 8B-class shapes in this mode are in test_gpu_fp8_8b.py."""

import numpy as np
import pytest
import torch

import oracle
from quantized_rl_rollout_gb300 import inputs

from .conftest import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
POW2 = 1


@pytest.fixture(scope="module")
def q():
    from quantized_rl_rollout_gb300 import build, qrr

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qrr.lib()
    return qrr


def _gemm(q, x, W, st=None):
    qa, sa = q.quantize_fp8_a1x128(x, POW2)
    qw, sw = q.quantize_fp8_w128x128(W, POW2)
    y = q.gemm_fp8_blockwise(qa, sa, qw, sw, POW2, dev_status=st)
    torch.cuda.synchronize()
    y_ref = oracle.fp8.gemm_blockwise(qa.cpu().numpy(), sa.cpu().numpy(), qw.cpu().numpy(), sw.cpu().numpy())
    return y, y_ref


@pytest.mark.parametrize("m,n,k", [(32, 256, 256), (130, 384, 640), (256, 512, 4608), (1, 128, 128)])
def test_exact_integers(q, m, n, k):
    """Small integers, power-of-two scales: every block sum and the total are
    exact in fp32, so the output must be the bf16 rounding of the exact
    result bit for bit.  K = 4608 has 36 K blocks, wrapping the 8-group ring
    of scale columns; 130 tokens and 384 weight rows leave ragged tiles."""
    a = ((torch.arange(m * k, device=DEV).reshape(m, k) * 7 % 13) - 6).to(torch.bfloat16)
    w = ((torch.arange(n * k, device=DEV).reshape(n, k) * 5 % 11) - 5).to(torch.bfloat16)
    # vary the scales from block to block: scale row blocks and weight tiles by powers of two
    a = a * (2.0 ** (torch.arange(k, device=DEV) // 128 % 5 - 2)).to(torch.bfloat16)
    w = w * (2.0 ** (torch.arange(n, device=DEV) // 128 % 3 - 1)).to(torch.bfloat16)[:, None]
    y, y_ref = _gemm(q, a, w)
    assert np.array_equal(to_np(y), oracle.formats.bf16_rne(y_ref))


@pytest.mark.parametrize("m,n,k", [(96, 384, 512), (200, 256, 1152), (64, 1024, 4096)])
def test_random_shapes(q, m, n, k):
    x = inputs.activations(m, k, inputs.derive_seed(0, "mx", m, n, k, "x"), device=DEV, channel_outlier_frac=0.01)
    W = inputs.weight(n, k, inputs.derive_seed(0, "mx", m, n, k, "W"), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, y_ref = _gemm(q, x, W, st)
    assert q.get_last_device_status(st) == 0
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(y), y_ref)
    assert ok, f"normwise {nerr:.3e}, worst element ratio {worst:.3f}"


@pytest.mark.parametrize("xs,ws", [(1e-37, 1e30), (1e30, 1e-37), (1e-38, 1e25)])
def test_scales_beyond_the_byte(q, xs, ws):
    """Activation or weight magnitudes whose power-of-two scales lie below
    2^-127 (bf16 reaches down to 2^-133), paired with large magnitudes on the
    other operand so the products stay in fp32's normal range: the kernel
    shifts each K block's exponents so every product sa * sw is still applied
    exactly."""
    m, n, k = 64, 256, 512
    x = (inputs.activations(m, k, 31, device=DEV).float() * xs).to(torch.bfloat16)
    W = (inputs.weight(n, k, 32, device=DEV).float() * ws).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, y_ref = _gemm(q, x, W, st)
    assert q.get_last_device_status(st) == 0
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(y), y_ref)
    assert ok, f"normwise {nerr:.3e}, worst element ratio {worst:.3f}"


def test_mixed_magnitude_rows(q):
    """Rows of one tile whose scales differ by ~2^127 within the same K block,
    the small ones below the byte's reach: still one exact shift per block."""
    m, n, k = 128, 256, 512
    x = inputs.activations(m, k, 41, device=DEV).float()
    x[::2] *= 1e-38
    x = x.to(torch.bfloat16)
    W = (inputs.weight(n, k, 42, device=DEV).float() * 1e30).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, y_ref = _gemm(q, x, W, st)
    assert q.get_last_device_status(st) == 0
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(y[1::2]), y_ref[1::2])
    assert ok, f"large rows: normwise {nerr:.3e}"
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(y[::2]), y_ref[::2])
    assert ok, f"tiny rows: normwise {nerr:.3e}"


def test_zero_blocks(q):
    m, n, k = 64, 256, 512
    x = inputs.activations(m, k, 51, device=DEV)
    x[:, 128:256] = 0  # a zero activation block column: scale 0
    W = inputs.weight(n, k, 52, device=DEV)
    W[128:, 384:] = 0  # a zero weight tile
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, y_ref = _gemm(q, x, W, st)
    assert q.get_last_device_status(st) == 0
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(y), y_ref)
    assert ok, f"normwise {nerr:.3e}"
    zx = torch.zeros(m, k, dtype=torch.bfloat16, device=DEV)
    y0, _ = _gemm(q, zx, W)
    assert not y0.float().abs().max().item()


def test_broken_power_of_two_promise_is_flagged(q):
    m, n, k = 32, 256, 256
    x = inputs.activations(m, k, 61, device=DEV)
    W = inputs.weight(n, k, 62, device=DEV)
    qa, sa = q.quantize_fp8_a1x128(x, POW2)
    qw, sw = q.quantize_fp8_w128x128(W, POW2)
    sa[3, 1] *= 1.5  # not a power of two
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.gemm_fp8_blockwise(qa, sa, qw, sw, POW2, dev_status=st)
    assert q.get_last_device_status(st) & q.DEV_SCALE_RANGE

"""GPU parity of the LoRA backward through the frozen NVFP4 weight against the
float64 oracle: dX (bf16) and the adapter gradients dA, dB (fp32), within the
acceptance tolerance of the linear (normwise <= 5e-3, per element <= 1e-2
(|ref| + rms(ref))), on ragged shapes, with and without an adapter, on
closed forms, and on the full 8B-class layer set at 4096 tokens (dX on token
rows touching every 128-row tile, dA and dB in full)."""

import numpy as np
import pytest
import torch

import oracle
from oracle import lora_backward as lb
from quantized_rl_rollout_gb300 import configs, inputs

from .conftest import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def q():
    from quantized_rl_rollout_gb300 import build, qrr

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qrr.lib()
    return qrr


def _layer(q, m, n, k, r, tag):
    W = inputs.weight(n, k, inputs.derive_seed(0, "bwd", tag, "W"), device=DEV)
    codes, scales, ts = q.quantize_nvfp4(W)
    A, B, alpha = inputs.lora(r, k, n, inputs.derive_seed(0, "bwd", tag, "lora"), device=DEV) if r else (None, None, 0.0)
    x = inputs.activations(m, k, inputs.derive_seed(0, "bwd", tag, "x"), device=DEV, channel_outlier_frac=0.01)
    dy = inputs.activations(m, n, inputs.derive_seed(0, "bwd", tag, "dy"), device=DEV)
    return dy, x, codes, scales, ts, A, B, alpha


def _close(got, ref, what):
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(got), ref)
    assert ok, f"{what}: normwise {nerr:.3e}, worst element ratio {worst:.3f}"


@pytest.mark.parametrize("m,n,k,r", [(16, 128, 256, 8), (300, 384, 512, 32), (1, 256, 1024, 64), (64, 512, 256, 0),
                                     (130, 256, 768, 16), (257, 1024, 2048, 32)])
def test_shapes(q, m, n, k, r):
    dy, x, codes, scales, ts, A, B, alpha = _layer(q, m, n, k, r, f"{m}-{n}-{k}-{r}")
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dx, dA, dB = q.lora_backward_nvfp4(dy, x, codes, scales, ts, A, B, alpha, dev_status=st)
    assert q.get_last_device_status(st) == 0
    rdx, rda, rdb = lb.lora_backward(to_np(dy), to_np(x), codes.cpu().numpy(), scales.cpu().numpy(),
                                     np.float32(ts.item()), None if A is None else to_np(A),
                                     None if B is None else to_np(B), alpha)
    _close(dx, rdx, "dX")
    if r:
        _close(dA, rda, "dA")
        _close(dB, rdb, "dB")
    else:
        assert dA is None and dB is None


def test_closed_forms(q):
    m, n, k, r = 40, 256, 512, 16
    dy, x, codes, scales, ts, A, B, alpha = _layer(q, m, n, k, r, "closed")
    dx, dA, dB = q.lora_backward_nvfp4(torch.zeros_like(dy), x, codes, scales, ts, A, B, alpha)
    torch.cuda.synchronize()
    assert not dx.float().abs().max().item() and not dA.abs().max().item() and not dB.abs().max().item()
    dx, dA, dB = q.lora_backward_nvfp4(dy, x, codes, scales, ts, A, B, 0.0)
    torch.cuda.synchronize()
    assert not dA.abs().max().item() and not dB.abs().max().item()
    rdx, _, _ = lb.lora_backward(to_np(dy), to_np(x), codes.cpu().numpy(), scales.cpu().numpy(),
                                 np.float32(ts.item()), None, None, 0.0)
    _close(dx, rdx, "dX alpha=0")
    # W = 0: dX is the adapter term only
    zc, zs, zt = q.quantize_nvfp4(torch.zeros(n, k, dtype=torch.bfloat16, device=DEV))
    dx, dA, dB = q.lora_backward_nvfp4(dy, x, zc, zs, zt, A, B, alpha)
    torch.cuda.synchronize()
    rdx, rda, rdb = lb.lora_backward(to_np(dy), to_np(x), zc.cpu().numpy(), zs.cpu().numpy(), np.float32(0.0),
                                     to_np(A), to_np(B), alpha)
    _close(dx, rdx, "dX W=0")
    _close(dA, rda, "dA W=0")
    _close(dB, rdb, "dB W=0")


def test_no_tokens(q):
    n, k, r = 256, 512, 8
    _, _, codes, scales, ts, A, B, alpha = _layer(q, 1, n, k, r, "empty")
    dy = torch.empty(0, n, dtype=torch.bfloat16, device=DEV)
    x = torch.empty(0, k, dtype=torch.bfloat16, device=DEV)
    dA = torch.full((r, k), 7.0, device=DEV)
    dB = torch.full((n, r), 7.0, device=DEV)
    dx, dA, dB = q.lora_backward_nvfp4(dy, x, codes, scales, ts, A, B, alpha, dA=dA, dB=dB)
    torch.cuda.synchronize()
    assert dx.shape == (0, k) and not dA.abs().max().item() and not dB.abs().max().item()


@pytest.mark.parametrize("li", range(7))
def test_8b_layer_at_4096_tokens(q, li):
    layer = configs.LAYERS_8B[li]
    m, r = 4096, 32
    W = inputs.weight(layer.n, layer.k, inputs.derive_seed(0, "8b", layer.name, "W"), device=DEV)
    codes, scales, ts = q.quantize_nvfp4(W)
    A, B, alpha = inputs.lora(r, layer.k, layer.n, inputs.derive_seed(0, "8b", layer.name, "lora"), device=DEV)
    x = inputs.activations(m, layer.k, inputs.derive_seed(0, "8b", layer.name, "xp"), device=DEV,
                           channel_outlier_frac=0.01)
    dy = inputs.activations(m, layer.n, inputs.derive_seed(0, "8b", layer.name, "dy"), device=DEV)
    dx, dA, dB = q.lora_backward_nvfp4(dy, x, codes, scales, ts, A, B, alpha)
    torch.cuda.synchronize()
    g = np.random.default_rng(40 + li)
    tiles = np.arange(0, m, 128)
    rows = np.unique(np.concatenate([[0, m - 1], tiles + g.integers(0, 128, tiles.size)]))
    rt = torch.from_numpy(rows).to(DEV)
    w_hat = oracle.nvfp4.dequantize(codes.cpu().numpy(), scales.cpu().numpy(), np.float32(ts.item()))
    _close(dx[rt], lb.lora_backward_dx_rows(to_np(dy[rt]), w_hat, to_np(A), to_np(B), alpha), f"dX {layer.name}")
    dy64, x64 = to_np(dy).astype(np.float64), to_np(x).astype(np.float64)
    a64, b64 = to_np(A).astype(np.float64), to_np(B).astype(np.float64)
    c = alpha / r
    _close(dA, c * ((dy64 @ b64).T @ x64), f"dA {layer.name}")
    _close(dB, c * (dy64.T @ (x64 @ a64.T)), f"dB {layer.name}")

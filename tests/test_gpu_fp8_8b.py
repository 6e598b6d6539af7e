"""GPU parity of the FP8 path at the full 8B-class shapes, in both scale
modes, against the float64 oracle: the blockwise-scaled GEMM on every one of
the seven layers at 4096 tokens (the launches the benchmark times), and the
re-quantization of the whole bf16 layer set to 128x128 E4M3 tiles.

Sampling: the GEMM is checked on token rows that touch every 128-row tile of
the 4096 tokens (one random row per tile plus the first and last row), across
all N output columns; the re-quantization is checked on every tile scale and,
bit for bit, on the codes of four 128-row tile bands per layer (the first, the
last and two random ones).  Also: the non-finite flag of both FP8 quantizers
and of the decode prologue."""

import numpy as np
import pytest
import torch

import oracle
from quantized_rl_rollout_gb300 import configs, inputs

from .conftest import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
M = 4096


@pytest.fixture(scope="module")
def q():
    from quantized_rl_rollout_gb300 import build, qrr

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qrr.lib()
    return qrr


def _rows_every_tile(g, m):
    tiles = np.arange(0, m, 128)
    return np.unique(np.concatenate([[0, m - 1], tiles + g.integers(0, 128, tiles.size)]))


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("li", range(7))
def test_fp8_gemm_8b_layer(q, mode, li):
    layer = configs.LAYERS_8B[li]
    g = np.random.default_rng(100 + li)
    W = inputs.weight(layer.n, layer.k, inputs.derive_seed(0, "8b", layer.name, "W"), device=DEV)
    x = inputs.activations(M, layer.k, inputs.derive_seed(0, "8b", layer.name, "xp"), device=DEV,
                           channel_outlier_frac=0.01)
    qa, sa = q.quantize_fp8_a1x128(x, mode)
    qw, sw = q.quantize_fp8_w128x128(W, mode)
    y = q.gemm_fp8_blockwise(qa, sa, qw, sw, mode)
    torch.cuda.synchronize()
    rows = _rows_every_tile(g, M)
    rt = torch.from_numpy(rows).to(DEV)
    y_ref = oracle.fp8.gemm_blockwise(qa[rt].cpu().numpy(), sa[rt].cpu().numpy(), qw.cpu().numpy(),
                                      sw.cpu().numpy())
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(y[rt]), y_ref)
    assert ok, f"{layer.name} mode {mode}: normwise {nerr:.3e}, worst element ratio {worst:.3f}"


@pytest.mark.parametrize("mode", [0, 1])
def test_fp8_requant_8b_layer_set(q, mode):
    """The benchmark's FP8 re-quantization (one grouped call over the seven
    updated bf16 weights): every tile scale exact, sampled tile bands bit-exact."""
    L = configs.LAYERS_8B
    g = np.random.default_rng(7 + mode)
    Ws = [inputs.updated(inputs.weight(l.n, l.k, inputs.derive_seed(0, "8b", l.name, "W"), device=DEV),
                         inputs.derive_seed(0, "8b", l.name, "update")) for l in L]
    outs = [(torch.empty(l.n, l.k, dtype=torch.uint8, device=DEV),
             torch.empty((l.n + 127) // 128, l.k // 128, dtype=torch.float32, device=DEV)) for l in L]
    q.requantize_weights(Ws, outs, q.FORMAT_FP8_W128, mode)
    torch.cuda.synchronize()
    for l, w, (qc, sc) in zip(L, Ws, outs):
        nt, kt = (l.n + 127) // 128, l.k // 128
        # tile absmax by its definition (max |w| over the 128 x 128 tile), then the oracle's scale rule
        amax = w.float().abs().reshape(nt, 128, kt, 128).amax(dim=(1, 3)).cpu().numpy()
        assert np.array_equal(sc.cpu().numpy(), oracle.fp8.scale_of(amax, mode)), l.name
        bands = np.unique(np.concatenate([[0, nt - 1], g.integers(0, nt, 2)]))
        for b in bands:
            rq, rs = oracle.fp8.quantize_w128x128(to_np(w[b * 128:(b + 1) * 128]), mode)
            assert np.array_equal(rs[0], sc[b].cpu().numpy()), (l.name, b)
            assert np.array_equal(rq, qc[b * 128:(b + 1) * 128].cpu().numpy()), (l.name, b)


@pytest.mark.parametrize("mode", [0, 1])
def test_fp8_quantizers_flag_nonfinite(q, mode):
    for bad in (float("inf"), float("nan"), float("-inf")):
        x = torch.randn(16, 512, device=DEV).to(torch.bfloat16)
        x[5, 300] = bad
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        q.quantize_fp8_a1x128(x, mode, dev_status=st)
        assert q.get_last_device_status(st) & q.DEV_NONFINITE, ("a1x128", bad)
        W = torch.randn(256, 384, device=DEV).to(torch.bfloat16)
        W[200, 17] = bad
        st.zero_()
        q.quantize_fp8_w128x128(W, mode, dev_status=st)
        assert q.get_last_device_status(st) & q.DEV_NONFINITE, ("w128", bad)
        st.zero_()
        outs = [(torch.empty(256, 384, dtype=torch.uint8, device=DEV),
                 torch.empty(2, 3, dtype=torch.float32, device=DEV))]
        q.requantize_weights([W], outs, q.FORMAT_FP8_W128, mode, dev_status=st)
        assert q.get_last_device_status(st) & q.DEV_NONFINITE, ("requant", bad)
    ok = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.quantize_fp8_a1x128(torch.randn(16, 512, device=DEV).to(torch.bfloat16), mode, dev_status=ok)
    q.quantize_fp8_w128x128(torch.randn(256, 384, device=DEV).to(torch.bfloat16), mode, dev_status=ok)
    assert q.get_last_device_status(ok) == 0


@pytest.mark.parametrize("m", [1, 8, 64])
def test_decode_prologue_flags_nonfinite(q, m):
    """The decode path's prologue (which forms the f16 image of x) flags a
    non-finite token value; finite tokens leave the word at zero."""
    n, k, r = 256, 1024, 16
    W = inputs.weight(n, k, inputs.derive_seed(0, "nf-dec", "W"), device=DEV)
    codes, scales, ts = q.quantize_nvfp4(W)
    A, B, alpha = inputs.lora(r, k, n, inputs.derive_seed(0, "nf-dec", "lora"), device=DEV)
    x = inputs.activations(m, k, inputs.derive_seed(0, "nf-dec", "x", m), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha, dev_status=st)
    assert q.get_last_device_status(st) == 0
    for bad in (float("inf"), float("nan")):
        xb = x.clone()
        xb[m - 1, k // 3] = bad
        st.zero_()
        q.linear_nvfp4_lora(xb, codes, scales, ts, A, B, alpha, dev_status=st)
        assert q.get_last_device_status(st) & q.DEV_NONFINITE, bad

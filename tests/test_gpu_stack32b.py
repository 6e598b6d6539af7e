"""The 32B-class decode stack at full size: 64 decoder layers of hidden 5120
(q/o 5120x5120, k/v 1024x5120, gate/up 27648x5120, down 5120x27648), NVFP4
weights with LoRA r = 64, 64 tokens.

Every layer's bf16 master weights receive a trainer update and are
re-quantized with the batched requant call (the whole stack: 31.2 G
elements); every tensor scale must be exact and sampled rows of codes and
block scales bit-exact.  Then each layer runs as one grouped decode call (the
bench's launch configuration) and sampled output columns of every 128-row
tile neighbourhood must meet the output tolerance against the float64
oracle."""

import numpy as np
import pytest
import torch

import oracle
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


def _assert_close(y, y_ref, what):
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(y), y_ref)
    assert ok, f"{what}: normwise {nerr:.3e}, worst element ratio {worst:.3f}"


def test_stack32b_requant_and_decode(q):
    c = configs.DECODE_32B
    r, m, depth = c["r"], c["tokens"], c["depth"]
    g = np.random.default_rng(32)
    stack = []
    for li in range(depth):
        masters, outs = [], []
        for lay in configs.LAYERS_32B:
            W = inputs.weight(lay.n, lay.k, inputs.derive_seed(0, "32b", li, lay.name, "W"), device=DEV)
            masters.append(inputs.updated(W, inputs.derive_seed(0, "32b", li, lay.name, "dW")))
            del W
            outs.append((torch.empty(lay.n, lay.k // 2, dtype=torch.uint8, device=DEV),
                         torch.empty(lay.n, lay.k // 16, dtype=torch.uint8, device=DEV),
                         torch.empty(1, dtype=torch.float32, device=DEV)))
        q.requantize_weights(masters, outs, q.FORMAT_NVFP4)
        torch.cuda.synchronize()
        entries = []
        for lay, Wn, (codes, scales, ts) in zip(configs.LAYERS_32B, masters, outs):
            rt = oracle.nvfp4.tensor_scale(Wn.abs().max().float().item())
            assert ts.item() == float(rt), f"layer {li} {lay.name}: tensor scale"
            rows = np.unique(np.concatenate([[0, lay.n - 1] if li == 0 else [], g.integers(0, lay.n, 2)])).astype(np.int64)
            rows_t = torch.from_numpy(rows).to(DEV)
            rc, rs = oracle.nvfp4.quantize_rows(to_np(Wn[rows_t]), rt)
            assert np.array_equal(codes[rows_t].cpu().numpy(), rc), f"layer {li} {lay.name}: codes"
            assert np.array_equal(scales[rows_t].cpu().numpy(), rs), f"layer {li} {lay.name}: block scales"
            A, B, alpha = inputs.lora(r, lay.k, lay.n, inputs.derive_seed(0, "32b", li, lay.name, "lora"), device=DEV)
            x = inputs.activations(m, lay.k, inputs.derive_seed(0, "32b", li, lay.name, "x"), device=DEV)
            entries.append(dict(x=x, codes=codes, scales=scales, tensor_scale=ts, lora_A=A, lora_B=B, alpha=alpha))
        del masters
        stack.append(entries)

    ys = [q.linear_nvfp4_lora_grouped(entries) for entries in stack]
    torch.cuda.synchronize()
    for li, (entries, outs) in enumerate(zip(stack, ys)):
        for lay, d, y in zip(configs.LAYERS_32B, entries, outs):
            tiles = np.arange(0, lay.n // 128, 4) * 128
            rows = np.unique(np.concatenate([tiles + g.integers(0, 128, tiles.size), g.integers(0, lay.n, 8)]))
            rows_t = torch.from_numpy(rows.astype(np.int64)).to(DEV)
            w_hat = oracle.nvfp4.dequantize(d["codes"][rows_t].cpu().numpy(), d["scales"][rows_t].cpu().numpy(),
                                            np.float32(d["tensor_scale"].item()))
            y_ref = oracle.linear.linear_rows(to_np(d["x"]), w_hat, to_np(d["lora_A"]), to_np(d["lora_B"][rows_t]),
                                              d["alpha"])
            _assert_close(y[:, rows_t], y_ref, f"32B layer {li} {lay.name}")

"""GPU parity of the W4A16 + LoRA linear and the blockwise FP8 GEMM against the
float64 oracle, within the acceptance tolerance (normwise <= 5e-3, per
element <= 1e-2 (|y| + rms(y))), plus re-quantization of a layer set."""

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


def _layer(q, n, k, r, tag, outliers=True):
    W = inputs.weight(n, k, inputs.derive_seed(0, tag, "W"), device=DEV, outlier_frac=1e-3 if outliers else 0.0)
    codes, scales, ts = q.quantize_nvfp4(W)
    A, B, alpha = inputs.lora(r, k, n, inputs.derive_seed(0, tag, "lora"), device=DEV) if r else (None, None, 0.0)
    return W, codes, scales, ts, A, B, alpha


def _ref(x, codes, scales, ts, A, B, alpha, rows=None):
    c = codes.cpu().numpy()
    s = scales.cpu().numpy()
    t = np.float32(ts.item())
    a = None if A is None else to_np(A)
    b = None if B is None else to_np(B)
    if rows is None:
        return oracle.linear.linear_nvfp4_lora(to_np(x), c, s, t, a, b, alpha)
    w_hat = oracle.nvfp4.dequantize(c[rows], s[rows], t)
    return oracle.linear.linear_rows(to_np(x), w_hat, a, None if b is None else b[rows], alpha)


def _assert_close(y, y_ref, what):
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(y), y_ref)
    assert ok, f"{what}: normwise {nerr:.3e}, worst element ratio {worst:.3f}"


def test_tiny_config(q):
    c = configs.TINY
    W = inputs.weight(c["n"], c["k"], inputs.derive_seed(0, "tiny", "W"), device=DEV)
    x = inputs.activations(c["m"], c["k"], inputs.derive_seed(0, "tiny", "x"), device=DEV)
    A, B, _ = inputs.lora(c["r"], c["k"], c["n"], inputs.derive_seed(0, "tiny", "lora"), device=DEV)
    codes, scales, ts = q.quantize_nvfp4(W)
    y = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, c["alpha"])
    torch.cuda.synchronize()
    _assert_close(y, _ref(x, codes, scales, ts, A, B, c["alpha"]), "tiny")


@pytest.mark.parametrize("m", [1, 3, 8, 17, 64, 65, 256])
@pytest.mark.parametrize("r", [0, 8, 32, 64])
def test_token_counts_and_ranks(q, m, r):
    n, k = 384, 1024
    W, codes, scales, ts, A, B, alpha = _layer(q, n, k, r, f"mr{r}")
    x = inputs.activations(m, k, inputs.derive_seed(0, "x", m, r), device=DEV)
    y = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha)
    torch.cuda.synchronize()
    _assert_close(y, _ref(x, codes, scales, ts, A, B, alpha), f"m={m} r={r}")


def test_closed_forms(q):
    n, k, r = 256, 512, 16
    W, codes, scales, ts, A, B, alpha = _layer(q, n, k, r, "closed")
    x = torch.zeros(5, k, dtype=torch.bfloat16, device=DEV)
    y = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha)
    torch.cuda.synchronize()
    assert not y.float().abs().max().item()
    # one-hot token -> column k0 of W_hat plus the adapter column
    k0 = 301
    x[2, k0] = 1.0
    y = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha)
    torch.cuda.synchronize()
    _assert_close(y, _ref(x, codes, scales, ts, A, B, alpha), "one-hot")
    # alpha = 0 equals no adapter
    xr = inputs.activations(9, k, 5, device=DEV)
    y0 = q.linear_nvfp4_lora(xr, codes, scales, ts, A, B, 0.0)
    y1 = q.linear_nvfp4_lora(xr, codes, scales, ts, None, None, 0.0)
    torch.cuda.synchronize()
    _assert_close(y0, _ref(xr, codes, scales, ts, None, None, 0.0), "alpha=0")
    _assert_close(y1, _ref(xr, codes, scales, ts, None, None, 0.0), "no adapter")
    # W = 0 -> adapter term only
    Z = torch.zeros(n, k, dtype=torch.bfloat16, device=DEV)
    zc, zs, zt = q.quantize_nvfp4(Z)
    y = q.linear_nvfp4_lora(xr, zc, zs, zt, A, B, alpha)
    torch.cuda.synchronize()
    _assert_close(y, _ref(xr, zc, zs, zt, A, B, alpha), "W=0")


@pytest.mark.parametrize("n", [384, 512])
@pytest.mark.parametrize("m", [1, 8, 64, 100, 300])
def test_one_hot_tokens_bit_exact(q, m, n):
    """Token m is +-e_{k_m}: y[m] is then +-W_hat[:, k_m] scaled once by s_t
    in fp32 and rounded to bf16, with no sum to round, so every output is
    fixed to the bit (the E2M1-plane decode at 1 and 8 tokens, where +-1
    scales to the single digit +-4, the f16 decode tiles at 64 tokens, the
    bf16 prefill tiles of 128 and 256 tokens with a ragged last tile, on
    single CTAs for an odd number of 128-row tiles and on CTA pairs for an
    even one)."""
    k = 2048
    W, codes, scales, ts, _, _, _ = _layer(q, n, k, 0, "onehot")
    g = np.random.default_rng(m)
    cols = g.choice(k, m, replace=False)
    sign = np.where(g.random(m) < 0.5, -1.0, 1.0)
    xh = np.zeros((m, k), np.float32)
    xh[np.arange(m), cols] = sign
    x = torch.from_numpy(xh).to(torch.bfloat16).to(DEV)
    y = q.linear_nvfp4_lora(x, codes, scales, ts, None, None, 0.0)
    torch.cuda.synchronize()
    w_hat = oracle.nvfp4.dequantize(codes.cpu().numpy(), scales.cpu().numpy(), np.float32(ts.item()))
    want = oracle.formats.bf16_rne(np.float32(w_hat[:, cols].T * sign[:, None]))
    got = y.float().cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} outputs differ, first {bad[:3].tolist()}"


def test_empty_tokens(q):
    W, codes, scales, ts, A, B, alpha = _layer(q, 128, 256, 8, "empty")
    x = torch.zeros(0, 256, dtype=torch.bfloat16, device=DEV)
    y = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha)
    torch.cuda.synchronize()
    assert y.shape == (0, 128)


@pytest.mark.parametrize("m", [1, 8, 64])
def test_decode_8b_layer_set_sampled(q, m):
    """Every layer of the 8B-class set at decode sizes; 256 sampled output
    columns per layer (all tokens) against the oracle."""
    g = np.random.default_rng(m)
    r = configs.DECODE_8B["r"]
    for layer in configs.LAYERS_8B:
        tag = f"dec8b/{layer.name}"
        W, codes, scales, ts, A, B, alpha = _layer(q, layer.n, layer.k, r, tag)
        x = inputs.activations(m, layer.k, inputs.derive_seed(0, tag, "x", m), device=DEV)
        y = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha)
        torch.cuda.synchronize()
        rows = np.unique(np.concatenate([[0, layer.n - 1], g.integers(0, layer.n, 254)]))
        y_ref = _ref(x, codes, scales, ts, A, B, alpha, rows=rows)
        _assert_close(y[:, torch.from_numpy(rows).to(DEV)], y_ref, f"{layer.name} m={m}")
        del W, codes, scales


@pytest.mark.parametrize("m", [1, 8, 64, 200, 300])
def test_grouped_layer_set(q, m):
    """The grouped call over a mixed layer set (different N, K, ranks, one
    layer without adapter) matches the oracle layer by layer."""
    shapes = [(384, 1024, 32), (128, 256, 8), (256, 2048, 0), (512, 768, 64)]
    if m == 200:  # an even tile count in every layer: the prefill tiles run on CTA pairs
        shapes = [(256, 1024, 32), (512, 256, 8), (256, 2048, 0), (768, 768, 64)]
    layers = []
    for i, (n, k, r) in enumerate(shapes):
        W, codes, scales, ts, A, B, alpha = _layer(q, n, k, r, f"grp{i}")
        x = inputs.activations(m, k, inputs.derive_seed(0, "grp-x", i, m), device=DEV)
        layers.append(dict(x=x, codes=codes, scales=scales, tensor_scale=ts, lora_A=A, lora_B=B, alpha=alpha))
    ys = q.linear_nvfp4_lora_grouped(layers)
    torch.cuda.synchronize()
    for i, d in enumerate(layers):
        _assert_close(ys[i], _ref(d["x"], d["codes"], d["scales"], d["tensor_scale"], d["lora_A"], d["lora_B"],
                                  d["alpha"]), f"grouped layer {i} m={m}")


@pytest.mark.parametrize("m", [1, 8, 64])
def test_grouped_call_in_cuda_graph(q, m):
    """The grouped call captured in a CUDA graph (workspace and outputs
    supplied, so the call allocates nothing) replays to the same bits as a
    direct call, also after the captured x buffers are refilled."""
    shapes = [(384, 1024, 32), (256, 2048, 0), (512, 768, 64)]
    layers = []
    for i, (n, k, r) in enumerate(shapes):
        W, codes, scales, ts, A, B, alpha = _layer(q, n, k, r, f"graph{i}")
        x = inputs.activations(m, k, inputs.derive_seed(0, "graph-x", i, m), device=DEV)
        y = torch.empty(m, n, dtype=torch.bfloat16, device=DEV)
        layers.append(dict(x=x, codes=codes, scales=scales, tensor_scale=ts, lora_A=A, lora_B=B, alpha=alpha, y=y))
    ws = torch.empty(q.linear_nvfp4_lora_grouped_workspace_bytes(layers), dtype=torch.uint8, device=DEV)
    q.linear_nvfp4_lora_grouped(layers, workspace=ws)
    torch.cuda.synchronize()
    direct = [d["y"].clone() for d in layers]
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        q.linear_nvfp4_lora_grouped(layers, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        q.linear_nvfp4_lora_grouped(layers, workspace=ws)
    for d in layers:
        d["y"].zero_()
    graph.replay()
    torch.cuda.synchronize()
    for i, d in enumerate(layers):
        assert torch.equal(d["y"], direct[i]), f"replay differs, layer {i}"
    for i, d in enumerate(layers):
        d["x"].copy_(inputs.activations(m, d["x"].shape[1], inputs.derive_seed(1, "graph-x", i, m), device=DEV))
    graph.replay()
    torch.cuda.synchronize()
    for i, d in enumerate(layers):
        _assert_close(d["y"], _ref(d["x"], d["codes"], d["scales"], d["tensor_scale"], d["lora_A"], d["lora_B"],
                                   d["alpha"]), f"graph replay, new x, layer {i} m={m}")


@pytest.mark.parametrize("m", [1, 8, 64])
def test_grouped_8b_decode_sampled(q, m):
    """The 8B-class layer set in one grouped call, the bench's launch
    configuration: every CTA runs several units, so accumulator reuse, issuer
    alternation across unit boundaries and split-K tickets all take part;
    sampled columns of every 128-row tile."""
    g = np.random.default_rng(9)
    r = configs.DECODE_8B["r"]
    layers = []
    for layer in configs.LAYERS_8B:
        W, codes, scales, ts, A, B, alpha = _layer(q, layer.n, layer.k, r, f"g8b/{layer.name}")
        x = inputs.activations(m, layer.k, inputs.derive_seed(0, "g8b-x", layer.name, m), device=DEV)
        layers.append(dict(x=x, codes=codes, scales=scales, tensor_scale=ts, lora_A=A, lora_B=B, alpha=alpha))
        del W
    ys = q.linear_nvfp4_lora_grouped(layers)
    torch.cuda.synchronize()
    for layer, d, y in zip(configs.LAYERS_8B, layers, ys):
        tiles = np.arange(layer.n // 128) * 128
        rows = np.unique(np.concatenate([[0, layer.n - 1], tiles + g.integers(0, 128, tiles.size),
                                         g.integers(0, layer.n, 64)]))
        y_ref = _ref(d["x"], d["codes"], d["scales"], d["tensor_scale"], d["lora_A"], d["lora_B"], d["alpha"],
                     rows=rows)
        _assert_close(y[:, torch.from_numpy(rows).to(DEV)], y_ref, f"grouped 8B {layer.name} m={m}")


def test_grouped_8b_prefill_sampled(q):
    """The 8B-class layer set at 4096 tokens in one grouped call, the bench's
    prefill launch (256-token tiles on CTA pairs, LoRA r = 32): all 4096
    tokens of sampled output columns, at least one column in every 128-row
    tile, so both CTAs of every pair and every token tile are checked."""
    c = configs.PREFILL_8B
    m, r = c["tokens"], c["r"]
    g = np.random.default_rng(10)
    layers = []
    for layer in configs.LAYERS_8B:
        W, codes, scales, ts, A, B, alpha = _layer(q, layer.n, layer.k, r, f"p8b/{layer.name}")
        x = inputs.activations(m, layer.k, inputs.derive_seed(0, "p8b-x", layer.name), device=DEV)
        layers.append(dict(x=x, codes=codes, scales=scales, tensor_scale=ts, lora_A=A, lora_B=B, alpha=alpha))
        del W
    ys = q.linear_nvfp4_lora_grouped(layers)
    torch.cuda.synchronize()
    for layer, d, y in zip(configs.LAYERS_8B, layers, ys):
        tiles = np.arange(layer.n // 128) * 128
        rows = np.unique(np.concatenate([[0, layer.n - 1], tiles + g.integers(0, 128, tiles.size)]))
        y_ref = _ref(d["x"], d["codes"], d["scales"], d["tensor_scale"], d["lora_A"], d["lora_B"], d["alpha"],
                     rows=rows)
        _assert_close(y[:, torch.from_numpy(rows).to(DEV)], y_ref, f"grouped 8B prefill {layer.name}")


@pytest.mark.parametrize("mode", [0, 1])
def test_fp8_gemm_small(q, mode):
    m, n, k = 96, 384, 512
    x = inputs.activations(m, k, 11, device=DEV, channel_outlier_frac=0.01)
    W = inputs.weight(n, k, 12, device=DEV)
    qa, sa = q.quantize_fp8_a1x128(x, mode)
    qw, sw = q.quantize_fp8_w128x128(W, mode)
    y = q.gemm_fp8_blockwise(qa, sa, qw, sw, mode)
    torch.cuda.synchronize()
    y_ref = oracle.fp8.gemm_blockwise(qa.cpu().numpy(), sa.cpu().numpy(), qw.cpu().numpy(), sw.cpu().numpy())
    _assert_close(y, y_ref, f"fp8 mode {mode}")


def test_fp8_gemm_exact_integers(q):
    """Small integers with power-of-two scales: the exact result is
    representable, so the bf16 output must equal its rounding."""
    m, n, k = 32, 256, 256
    a = ((torch.arange(m * k, device=DEV).reshape(m, k) % 7) - 3).to(torch.bfloat16)
    w = ((torch.arange(n * k, device=DEV).reshape(n, k) % 5) - 2).to(torch.bfloat16)
    qa, sa = q.quantize_fp8_a1x128(a, 1)
    qw, sw = q.quantize_fp8_w128x128(w, 1)
    y = q.gemm_fp8_blockwise(qa, sa, qw, sw, 1)
    torch.cuda.synchronize()
    y_ref = oracle.fp8.gemm_blockwise(qa.cpu().numpy(), sa.cpu().numpy(), qw.cpu().numpy(), sw.cpu().numpy())
    assert np.array_equal(to_np(y), oracle.formats.bf16_rne(y_ref))


def test_fp8_gemm_8b_sampled(q):
    """FP8 path on an 8B-class layer at 4096 tokens; 64 sampled token rows."""
    g = np.random.default_rng(5)
    layer = configs.LAYERS_8B[4]  # gate 14336 x 4096
    x = inputs.activations(4096, layer.k, 21, device=DEV, channel_outlier_frac=0.01)
    W = inputs.weight(layer.n, layer.k, 22, device=DEV)
    qa, sa = q.quantize_fp8_a1x128(x)
    qw, sw = q.quantize_fp8_w128x128(W)
    y = q.gemm_fp8_blockwise(qa, sa, qw, sw)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 4095], g.integers(0, 4096, 62)]))
    rt = torch.from_numpy(rows).to(DEV)
    y_ref = oracle.fp8.gemm_blockwise(qa[rt].cpu().numpy(), sa[rt].cpu().numpy(), qw.cpu().numpy(), sw.cpu().numpy())
    _assert_close(y[rt], y_ref, "fp8 8B gate")


def test_requantize_nvfp4_matches_single_calls(q):
    shapes = [(512, 256), (1024, 4096), (96, 1024), (128, 32), (0, 64)]
    Ws = [inputs.weight(n, k, inputs.derive_seed(0, "rq", i), device=DEV) for i, (n, k) in enumerate(shapes)]
    Wu = [inputs.updated(w, inputs.derive_seed(0, "rq-upd", i)) for i, w in enumerate(Ws)]
    outs = [(torch.empty(n, k // 2, dtype=torch.uint8, device=DEV), torch.empty(n, k // 16, dtype=torch.uint8, device=DEV),
             torch.empty(1, dtype=torch.float32, device=DEV)) for n, k in shapes]
    q.requantize_weights(Wu, outs, q.FORMAT_NVFP4)
    torch.cuda.synchronize()
    for w, (c, s, t) in zip(Wu, outs):
        rc, rs, rt = oracle.nvfp4.quantize(to_np(w))
        assert t.item() == float(rt)
        assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("mode", [0, 1])
def test_requantize_fp8(q, mode):
    shapes = [(512, 256), (200, 1024), (1024, 128)]
    Ws = [inputs.updated(inputs.weight(n, k, i, device=DEV), 100 + i) for i, (n, k) in enumerate(shapes)]
    outs = [(torch.empty(n, k, dtype=torch.uint8, device=DEV),
             torch.empty((n + 127) // 128, k // 128, dtype=torch.float32, device=DEV)) for n, k in shapes]
    q.requantize_weights(Ws, outs, q.FORMAT_FP8_W128, mode)
    torch.cuda.synchronize()
    for w, (c, s) in zip(Ws, outs):
        rc, rs = oracle.fp8.quantize_w128x128(to_np(w), mode)
        assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(c.cpu().numpy(), rc)


def test_requantize_many_tensors_grouping(q):
    """More descriptors than one grouped launch holds (the library splits them)."""
    Ws = [inputs.weight(32 + i, 64, 500 + i, device=DEV) for i in range(60)]
    outs = [(torch.empty(w.shape[0], 32, dtype=torch.uint8, device=DEV),
             torch.empty(w.shape[0], 4, dtype=torch.uint8, device=DEV),
             torch.empty(1, dtype=torch.float32, device=DEV)) for w in Ws]
    q.requantize_weights(Ws, outs, q.FORMAT_NVFP4)
    torch.cuda.synchronize()
    for w, (c, s, t) in zip(Ws, outs):
        rc, rs, rt = oracle.nvfp4.quantize(to_np(w))
        assert t.item() == float(rt) and np.array_equal(c.cpu().numpy(), rc) and np.array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("m", [4, 40])
def test_decode_token_max_in_one_slice(q, m):
    """Each token's largest |x| sits in a different part of K (first, middle
    and last 64-wide steps): the per-token power of two of the f16 operand
    comes from the maximum over the whole row, which the decode prologue
    forms from its K slices, so every token still matches the oracle."""
    n, k, r = 256, 2048, 16
    W, codes, scales, ts, A, B, alpha = _layer(q, n, k, r, "slicemax")
    x = inputs.activations(m, k, inputs.derive_seed(0, "slicemax", m), device=DEV).float()
    x[0, k - 5] = 3.0e4
    x[1, 3] = -5.0e3
    x[2] *= 1e-6
    x[2, 1000] = 1.0
    x[3, 700] = 1.0e-30
    x = x.to(torch.bfloat16)
    y = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha)
    torch.cuda.synchronize()
    _assert_close(y, _ref(x, codes, scales, ts, A, B, alpha), f"m={m}")


def test_decode_nonfinite_x_flagged(q):
    """An infinite activation at decode sizes raises the non-finite status bit."""
    W, codes, scales, ts, A, B, alpha = _layer(q, 256, 1024, 16, "nonfin")
    x = inputs.activations(3, 1024, 11, device=DEV)
    x[1, 517] = float("inf")
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha, dev_status=st)
    torch.cuda.synchronize()
    assert q.get_last_device_status(st) & q.DEV_NONFINITE


@pytest.mark.parametrize("m", [1, 64])
def test_prepared_grouped_call(q, m):
    """A GroupedLinear prepared once gives the bits of the one-shot grouped
    call, and follows new tokens written into its x buffers in place."""
    shapes = [(384, 1024, 32), (256, 2048, 0), (512, 768, 64)]
    layers, ref_layers = [], []
    for i, (n, k, r) in enumerate(shapes):
        W, codes, scales, ts, A, B, alpha = _layer(q, n, k, r, f"prep{i}")
        x = inputs.activations(m, k, inputs.derive_seed(0, "prep-x", i, m), device=DEV)
        layers.append(dict(x=x, codes=codes, scales=scales, tensor_scale=ts, lora_A=A, lora_B=B, alpha=alpha))
        ref_layers.append(dict(layers[-1]))
    prep = q.GroupedLinear(layers)
    for step in range(2):
        if step:
            for i, d in enumerate(layers):
                d["x"].copy_(inputs.activations(m, d["x"].shape[1], inputs.derive_seed(1, "prep-x", i, m), device=DEV))
        ys = prep.run()
        for d, r in zip(layers, ref_layers):
            r["x"] = d["x"].clone()
            r["y"] = None
        ref = q.linear_nvfp4_lora_grouped(ref_layers)
        torch.cuda.synchronize()
        for a, b in zip(ys, ref):
            assert torch.equal(a, b)


@pytest.mark.parametrize("m", [1, 3, 8])
def test_decode_planes_wide_range(q, m):
    """The plane decode (up to 8 tokens) on activations spanning 2^-40 to
    2^20 within a token, with exact E2M1 values, values just off the
    rounding midpoints of every plane and a token of subnormal-sized
    values: the six digit planes leave less than 6^-5 of each token's
    largest value unrepresented, so the output stays within tolerance."""
    n, k, r = 384, 2048, 16
    W, codes, scales, ts, A, B, alpha = _layer(q, n, k, r, "planes-wide")
    g = np.random.default_rng(7 + m)
    xh = g.standard_normal((m, k)).astype(np.float32)
    xh *= np.exp2(g.integers(-40, 21, size=(m, k))).astype(np.float32)
    xh[0, :8] = [6.0, -4.0, 0.25, 0.75, 1.25, 2.5, 5.0, -3.5]  # on the E2M1 grid and its midpoints
    if m > 1:
        xh[1] = (g.standard_normal(k) * 1e-39).astype(np.float32)  # bf16 subnormals
    x = torch.from_numpy(xh).to(torch.bfloat16).to(DEV)
    y = q.linear_nvfp4_lora(x, codes, scales, ts, A, B, alpha)
    torch.cuda.synchronize()
    _assert_close(y, _ref(x, codes, scales, ts, A, B, alpha), f"m={m}")

"""GPU parity of the quantizers against the CPU oracle: rounding primitive,
NVFP4 and FP8 codes/scales bit-exact, on small, ragged, degenerate and
full-size inputs."""

import numpy as np
import pytest
import torch

import oracle
from oracle import formats
from quantized_rl_rollout_gb300 import configs, inputs

from .conftest import to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    from quantized_rl_rollout_gb300 import build, qrr

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qrr.lib()
    return qrr


DEV = "cuda"


def _probe_inputs(seed=0):
    g = np.random.default_rng(seed)
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    structured = (hi[:, None] | lows[None, :]).reshape(-1).view(np.float32)
    rnd = g.integers(0, 2**32, 1 << 22, dtype=np.uint64).astype(np.uint32).view(np.float32)
    pts = []
    for grid in (formats.E2M1_VALUES[:8], formats.E4M3_VALUES[:127]):
        mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
        for m in np.concatenate([mids, grid.astype(np.float32)]):
            f = np.float32(m)
            pts += [f, np.nextafter(f, np.float32(1e30)), np.nextafter(f, np.float32(-1e30))]
    pts = np.array(pts, np.float32)
    v = np.concatenate([structured, rnd, pts, -pts])
    return v[~np.isnan(v)]


@pytest.mark.parametrize("fmt", [0, 1])
def test_rounding_primitive(q, fmt):
    v = _probe_inputs()
    got = q.round_probe(torch.from_numpy(v).to(DEV), fmt).cpu().numpy()
    want = formats.e2m1_rne(v) if fmt == 0 else formats.e4m3_rne(v)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches, e.g. {v[bad[:5]]} -> {got[bad[:5]]} want {want[bad[:5]]}"


def _check_nvfp4(q, W):
    codes, scales, ts = q.quantize_nvfp4(W)
    torch.cuda.synchronize()
    rc, rs, rt = oracle.nvfp4.quantize(to_np(W))
    assert ts.item() == float(rt)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_nvfp4_tiny(q):
    c = configs.TINY
    W = inputs.weight(c["n"], c["k"], inputs.derive_seed(0, "tiny", "W"), device=DEV)
    _check_nvfp4(q, W)


@pytest.mark.parametrize("n,k", [(1, 32), (37, 96), (300, 4096), (4096, 1024 + 32), (129, 64)])
def test_nvfp4_shapes(q, n, k):
    W = inputs.weight(n, k, inputs.derive_seed(1, "shape", n, k), device=DEV)
    _check_nvfp4(q, W)


def test_nvfp4_degenerate(q):
    # all zero (s_t = 0), a single negative entry, negative zeros, a block far
    # below the tensor absmax (block scale underflows to 0), bf16 subnormals
    W = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
    _check_nvfp4(q, W)
    W[2, 33] = -3.0
    W[1, 5] = -0.0
    _check_nvfp4(q, W)
    W[0, 0] = 1000.0
    W[3, 16:32] = 1e-6
    W[3, 48:64] = 1e-39  # bf16 subnormal
    _check_nvfp4(q, W)
    tiny = torch.full((2, 32), 1e-39, dtype=torch.bfloat16, device=DEV)  # subnormal tensor scale
    tiny[1, 3] = -2e-39
    _check_nvfp4(q, tiny)
    empty = torch.zeros(0, 64, dtype=torch.bfloat16, device=DEV)
    codes, scales, ts = q.quantize_nvfp4(empty)
    torch.cuda.synchronize()
    assert ts.item() == 0.0


def test_nvfp4_grid_survival(q):
    """Entries planted on the NVFP4 grid decode back to themselves."""
    g = np.random.default_rng(7)
    n, k, f = 16, 128, -2
    codes = g.integers(0, 16, (n, k)).astype(np.uint8)
    blk = codes.reshape(n, k // 16, 16)
    blk[:, :, 0] = 7
    S = 2.0 ** g.integers(-7, 6, (n, k // 16)).astype(np.float64)
    S[0, 0] = 448.0 * 2.0 ** f
    w = (formats.e2m1_value(blk) * S[..., None]).reshape(n, k).astype(np.float32)
    W = torch.from_numpy(w).to(torch.bfloat16).to(DEV)
    c, s, t = q.quantize_nvfp4(W)
    torch.cuda.synchronize()
    assert t.item() == 2.0 ** f
    assert np.array_equal(oracle.nvfp4.unpack_nibbles(c.cpu().numpy()), codes)


def test_nvfp4_nonfinite_flag(q):
    W = torch.randn(8, 64, device=DEV).to(torch.bfloat16)
    W[3, 7] = float("inf")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.quantize_nvfp4(W, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & q.DEV_NONFINITE
    ok = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.quantize_nvfp4(torch.randn(8, 64, device=DEV).to(torch.bfloat16), dev_status=ok)
    torch.cuda.synchronize()
    assert ok.item() == 0


def test_nvfp4_8b_layer_set_sampled(q):
    """Full 8B-class layer set: exact tensor scale, sampled rows bit-exact."""
    g = np.random.default_rng(3)
    for layer in configs.LAYERS_8B:
        W = inputs.weight(layer.n, layer.k, inputs.derive_seed(0, "decode8b", layer.name, "W"), device=DEV)
        codes, scales, ts = q.quantize_nvfp4(W)
        torch.cuda.synchronize()
        amax = W.abs().max().float().item()
        rt = oracle.nvfp4.tensor_scale(amax)
        assert ts.item() == float(rt), layer.name
        rows = np.unique(np.concatenate([[0, layer.n - 1], g.integers(0, layer.n, 48)]))
        rows_t = torch.from_numpy(rows).to(DEV)
        rc, rs = oracle.nvfp4.quantize_rows(to_np(W[rows_t]), rt)
        assert np.array_equal(codes[rows_t].cpu().numpy(), rc), layer.name
        assert np.array_equal(scales[rows_t].cpu().numpy(), rs), layer.name


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("m,k", [(1, 128), (33, 512), (4096, 4096)])
def test_fp8_a1x128(q, mode, m, k):
    x = inputs.activations(m, k, inputs.derive_seed(0, "fp8a", m, k), device=DEV, channel_outlier_frac=0.01)
    qa, sa = q.quantize_fp8_a1x128(x, mode)
    torch.cuda.synchronize()
    rq, rs = oracle.fp8.quantize_a1x128(to_np(x), mode)
    assert np.array_equal(sa.cpu().numpy(), rs)
    assert np.array_equal(qa.cpu().numpy(), rq)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("n,k", [(128, 128), (200, 256), (1024, 4096), (1, 384)])
def test_fp8_w128(q, mode, n, k):
    W = inputs.weight(n, k, inputs.derive_seed(0, "fp8w", n, k), device=DEV)
    qw, sw = q.quantize_fp8_w128x128(W, mode)
    torch.cuda.synchronize()
    rq, rs = oracle.fp8.quantize_w128x128(to_np(W), mode)
    assert np.array_equal(sw.cpu().numpy(), rs)
    assert np.array_equal(qw.cpu().numpy(), rq)


def test_fp8_degenerate(q):
    x = torch.zeros(3, 256, dtype=torch.bfloat16, device=DEV)
    x[1, 130] = -2.5
    x[2, :128] = 1e-39
    for mode in (0, 1):
        qa, sa = q.quantize_fp8_a1x128(x, mode)
        torch.cuda.synchronize()
        rq, rs = oracle.fp8.quantize_a1x128(to_np(x), mode)
        assert np.array_equal(sa.cpu().numpy(), rs) and np.array_equal(qa.cpu().numpy(), rq)


def _bf16_neighbours(v):
    """bf16 values at, just below and just above each float in v."""
    b = torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16)
    bits = b.view(torch.int16).to(torch.int32)
    out = [bits, bits + 1, bits - 1]
    return torch.cat(out).to(torch.int16).view(torch.bfloat16).float().numpy()


def test_fp8_quotients_at_midpoints(q):
    """Elements placed on bf16 neighbours of every E4M3 midpoint times the
    block scale: the division and the tie rule decide every code."""
    g = np.random.default_rng(11)
    grid = formats.E4M3_VALUES[:127]
    mids = (grid[1:] + grid[:-1]) / 2
    rows = []
    for _ in range(64):
        c = float(torch.tensor(g.uniform(0.01, 100.0), dtype=torch.bfloat16).float())  # block scale s = c
        vals = _bf16_neighbours(mids * c)
        vals = vals[np.abs(vals) < 448 * c]
        sgn = np.where(g.random(vals.size) < 0.5, -1.0, 1.0)
        row = np.concatenate([[448 * c], vals * sgn]).astype(np.float32)
        row = np.resize(row, 128 * ((row.size + 127) // 128))
        row[0::128] = 448 * c  # every 1x128 block keeps its absmax, so s = c exactly
        rows.append(row[:512])
    x = torch.from_numpy(np.stack(rows)).to(torch.bfloat16).to(DEV)
    qa, sa = q.quantize_fp8_a1x128(x, 0)
    torch.cuda.synchronize()
    rq, rs = oracle.fp8.quantize_a1x128(to_np(x), 0)
    assert np.array_equal(sa.cpu().numpy(), rs)
    assert np.array_equal(qa.cpu().numpy(), rq)


def test_nvfp4_quotients_at_midpoints(q):
    """Blocks whose elements sit on bf16 neighbours of E2M1 midpoints times
    the block's own divisor d_b (absmax kept, so s_t and d_b do not move)."""
    g = np.random.default_rng(12)
    W0 = inputs.weight(256, 512, 99, device=DEV)
    w0 = to_np(W0)
    c0, s0, t0 = oracle.nvfp4.quantize(w0)
    d = formats.e4m3_value(s0) * np.float64(t0)  # [256, 32]
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    w1 = w0.copy().reshape(256, 32, 16)
    amax_pos = np.argmax(np.abs(w1), axis=-1)
    for n in range(256):
        for b in range(32):
            cand = _bf16_neighbours(mids * d[n, b])
            picks = g.choice(cand, 16) * np.where(g.random(16) < 0.5, -1.0, 1.0)
            keep = w1[n, b, amax_pos[n, b]]
            picks = np.where(np.abs(picks) < abs(keep), picks, 0.0)
            w1[n, b] = picks
            w1[n, b, amax_pos[n, b]] = keep
    W1 = torch.from_numpy(w1.reshape(256, 512).astype(np.float32)).to(torch.bfloat16).to(DEV)
    _check_nvfp4(q, W1)

"""GPU parity of adaptive quantization noise against the oracle: the noise
itself bit for bit (its generator is integer arithmetic and single fp32
roundings on both sides), and the re-quantization of noisy masters -- codes,
block and tensor scales bit-exact -- for NVFP4 and both FP8 scale modes, on
tiny, ragged, grouped and full 8B-class inputs."""

import numpy as np
import pytest
import torch

import oracle
from oracle import aqn
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


@pytest.mark.parametrize("seed,tensor,step,start,n", [(0, 0, 0, 0, 2), (0x1234567890ABCDEF, 5, 77, 0, 1 << 20),
                                                      (7, 300, 3, (1 << 33) + 1, 4097)])
def test_noise_bit_exact(q, seed, tensor, step, start, n):
    z = q.aqn_noise_probe(n, seed, tensor, step, start=start)
    torch.cuda.synchronize()
    assert np.array_equal(z.cpu().numpy(), aqn.noise(n, seed, tensor, step, start=start))


def test_sigma_schedule_matches(q):
    for s, S, a, b in [(0, 100, 1e-2, 5e-4), (37, 100, 1e-2, 5e-4), (99, 100, 1e-2, 5e-4), (3, 1, 1e-2, 1e-3)]:
        assert abs(q.aqn_sigma(s, S, a, b) - float(aqn.sigma_at(s, S, a, b))) <= 1e-6 * float(aqn.sigma_at(s, S, a, b))


def _nv_out(n, k):
    return (torch.empty(n, k // 2, dtype=torch.uint8, device=DEV), torch.empty(n, k // 16, dtype=torch.uint8, device=DEV),
            torch.empty(1, dtype=torch.float32, device=DEV))


@pytest.mark.parametrize("sigma", [0.0, 1e-3, 2e-2])
def test_nvfp4_noisy_requant(q, sigma):
    shapes = [(512, 256), (37, 96), (1024, 4096), (0, 64), (129, 64)]
    Ws = [inputs.weight(n, k, inputs.derive_seed(0, "aqn", i), device=DEV) for i, (n, k) in enumerate(shapes)]
    outs = [_nv_out(n, k) for n, k in shapes]
    s32 = np.float32(sigma)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.requantize_weights_aqn(Ws, outs, float(s32), 99, 12, dev_status=st)
    assert q.get_last_device_status(st) == 0
    ref = aqn.requantize_aqn([to_np(w) for w in Ws], s32, 99, 12)
    for (c, s, t), (rc, rs, rt), w in zip(outs, ref, Ws):
        assert t.item() == float(rt)
        assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(s.cpu().numpy(), rs)
    if sigma:  # the noise reached the codes
        plain = oracle.nvfp4.quantize(to_np(Ws[2]))[0]
        assert not np.array_equal(ref[2][0], plain)


@pytest.mark.parametrize("sigma", [1e-4, 3e-3, 5e-2, 1.0])
def test_nvfp4_noisy_absmax_near_ties(q, sigma):
    """The absmax pass draws noise only for values that can still hold a
    tensor's largest |W'| (within fp32(sigma) zmax of the largest |W| of a
    warp's share, by a bound that rounding cannot break).  Many near-ties
    around the maximum, in both signs, one tensor whose largest |W| sits in a
    single 8-value vector, and one spread evenly: the tensor scales and codes
    must still equal the oracle's for small, moderate and overwhelming noise."""
    g = np.random.default_rng(int(sigma * 1e6) + 3)
    a = (g.standard_normal((256, 512)) * 0.02).astype(np.float32)
    idx = g.choice(a.size, 300, replace=False)
    a.flat[idx] = np.where(g.random(300) < 0.5, -1.0, 1.0) * (0.5 - g.random(300) * 0.01)
    b = (g.standard_normal((128, 1024)) * 0.02).astype(np.float32)
    b[77, 8:16] = np.float32(0.25)
    c = np.full((64, 256), 0.125, np.float32) * np.where(g.random((64, 256)) < 0.5, -1.0, 1.0).astype(np.float32)
    Ws = [torch.from_numpy(x).to(torch.bfloat16).to(DEV) for x in (a, b, c)]
    outs = [_nv_out(w.shape[0], w.shape[1]) for w in Ws]
    s32 = np.float32(sigma)
    q.requantize_weights_aqn(Ws, outs, float(s32), 4242, 9)
    torch.cuda.synchronize()
    ref = aqn.requantize_aqn([to_np(w) for w in Ws], s32, 4242, 9)
    for (cd, sc, t), (rc, rs, rt) in zip(outs, ref):
        assert t.item() == float(rt)
        assert np.array_equal(sc.cpu().numpy(), rs) and np.array_equal(cd.cpu().numpy(), rc)


@pytest.mark.parametrize("mode", [0, 1])
def test_fp8_noisy_requant(q, mode):
    shapes = [(512, 256), (200, 1024), (1024, 128)]
    Ws = [inputs.weight(n, k, inputs.derive_seed(1, "aqn", i), device=DEV) for i, (n, k) in enumerate(shapes)]
    outs = [(torch.empty(n, k, dtype=torch.uint8, device=DEV),
             torch.empty((n + 127) // 128, k // 128, dtype=torch.float32, device=DEV)) for n, k in shapes]
    s32 = np.float32(5e-3)
    q.requantize_weights_aqn(Ws, outs, float(s32), 3, 4, fmt=q.FORMAT_FP8_W128, mode=mode)
    torch.cuda.synchronize()
    ref = aqn.requantize_aqn([to_np(w) for w in Ws], s32, 3, 4, fmt="fp8", mode=mode)
    for (c, s), (rc, rs) in zip(outs, ref):
        assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(c.cpu().numpy(), rc)


def test_many_descriptors_keep_their_stream(q):
    """More descriptors than one grouped launch holds: descriptor j keeps the
    noise stream of index j across the library's launch groups."""
    Ws = [inputs.weight(32, 64, 900 + i, device=DEV) for i in range(60)]
    outs = [_nv_out(32, 64) for _ in Ws]
    s32 = np.float32(1e-2)
    q.requantize_weights_aqn(Ws, outs, float(s32), 5, 1)
    torch.cuda.synchronize()
    ref = aqn.requantize_aqn([to_np(w) for w in Ws], s32, 5, 1)
    for (c, s, t), (rc, rs, rt) in zip(outs, ref):
        assert t.item() == float(rt) and np.array_equal(c.cpu().numpy(), rc) and np.array_equal(s.cpu().numpy(), rs)


def test_full_8b_layer_set_sampled(q):
    """The noisy re-quantization of the 8B-class set: every tensor scale exact
    (the absmax of the noisy tensor, found among the elements that can reach
    it: the noise is bounded by 2 sqrt 3 sigma), sampled rows bit-exact."""
    g = np.random.default_rng(8)
    L = configs.LAYERS_8B
    Ws = [inputs.weight(l.n, l.k, inputs.derive_seed(0, "8b", l.name, "W"), device=DEV) for l in L]
    outs = [_nv_out(l.n, l.k) for l in L]
    s32 = np.float32(aqn.sigma_at(10, 100, 1e-2, 5e-4))
    seed, step = 2024, 10
    q.requantize_weights_aqn(Ws, outs, float(s32), seed, step)
    torch.cuda.synchronize()
    reach = 2.0 * 2.0 * np.sqrt(3.0) * float(s32) * 1.01 + 1e-6
    for j, (l, w, (c, s, t)) in enumerate(zip(L, Ws, outs)):
        wa = w.float().abs()
        top = float(wa.max().item())
        cand = torch.nonzero(wa.reshape(-1) >= top - reach).reshape(-1).cpu().numpy()
        flat = w.reshape(-1)
        amax = max(abs(float(_noisy_at(flat, int(i), s32, seed, j, step))) for i in cand)
        rt = np.float32(t.item())
        assert rt == oracle.nvfp4.tensor_scale(amax), l.name
        rows = np.unique(np.concatenate([[0, l.n - 1], g.integers(0, l.n, 30)]))
        wn_rows = np.stack([_noisy_row(w, int(r), s32, seed, j, step) for r in rows])
        rc, rs = oracle.nvfp4.quantize_rows(wn_rows, rt)
        rows_t = torch.from_numpy(rows).to(DEV)
        assert np.array_equal(c[rows_t].cpu().numpy(), rc), l.name
        assert np.array_equal(s[rows_t].cpu().numpy(), rs), l.name


def _noisy_row(w, r, sigma, seed, j, step):
    k = w.shape[1]
    x = to_np(w[r])
    z = aqn.noise(k, seed, j, step, start=r * k)
    return oracle.formats.bf16_rne((x + (np.float32(sigma) * z).astype(np.float32)).astype(np.float32))


def _noisy_at(flat, i, sigma, seed, j, step):
    x = np.float32(flat[i].float().item())
    z = aqn.noise(1, seed, j, step, start=i)[0]
    return oracle.formats.bf16_rne(np.array([x + np.float32(np.float32(sigma) * z)], np.float32))[0]


@pytest.mark.parametrize("bad", [float("inf"), float("-inf"), float("nan")])
def test_nvfp4_noisy_absmax_flags_nonfinite(q, bad):
    """A non-finite master takes the noisy absmax sweep's fallback (every
    vector drawn): the device status still reports it, and a clean tensor
    in the same call raises nothing on its own."""
    W = (torch.randn(256, 512, device=DEV) * 0.02).to(torch.bfloat16)
    W[100, 37] = bad
    outs = [_nv_out(256, 512)]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.requantize_weights_aqn([W], outs, 1e-3, 7, 3, dev_status=st)
    torch.cuda.synchronize()
    assert q.get_last_device_status(st) & q.DEV_NONFINITE
    ok = torch.zeros(1, dtype=torch.int32, device=DEV)
    clean = (torch.randn(256, 512, device=DEV) * 0.02).to(torch.bfloat16)
    q.requantize_weights_aqn([clean], [_nv_out(256, 512)], 1e-3, 7, 3, dev_status=ok)
    torch.cuda.synchronize()
    assert q.get_last_device_status(ok) == 0

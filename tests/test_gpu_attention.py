"""GPU parity of the FP8 key/value cache and decode attention against the
oracle: cache rows bit-exact against the 1x128 rule (both scale modes), and
attention outputs within the acceptance tolerance (normwise <= 5e-3, per
element <= 1e-2 (|ref| + rms(ref))), on ragged sequence lengths, every
grouped-query ratio, the closed forms, and the 8B-class decode batch the
benchmark times (64 sequences up to 4096 cached tokens, 32 query / 8 KV heads)."""

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as att
from quantized_rl_rollout_gb300 import inputs

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


def _empty_cache(b, hkv, lmax):
    return (torch.zeros(b, hkv, lmax, 128, dtype=torch.uint8, device=DEV), torch.zeros(b, hkv, lmax, device=DEV),
            torch.zeros(b, hkv, lmax, 128, dtype=torch.uint8, device=DEV), torch.zeros(b, hkv, lmax, device=DEV))


def _fill(q, b, hkv, lmax, lens, mode, seed):
    """Fill the caches step by step through the append call."""
    kc, ks, vc, vs = _empty_cache(b, hkv, lmax)
    kr = inputs.activations(lmax * b * hkv, 128, inputs.derive_seed(0, "kv", seed, "k"), device=DEV).reshape(
        lmax, b, hkv, 128)
    vr = inputs.activations(lmax * b * hkv, 128, inputs.derive_seed(0, "kv", seed, "v"), device=DEV).reshape(
        lmax, b, hkv, 128)
    for t in range(int(max(lens))):
        pos = torch.full((b,), t, dtype=torch.int32, device=DEV)
        q.kv_append_fp8(kr[t].contiguous(), vr[t].contiguous(), pos, kc, ks, vc, vs, mode)
    return kc, ks, vc, vs, kr, vr


@pytest.mark.parametrize("mode", [0, 1])
def test_append_rows_bit_exact(q, mode):
    b, hkv, lmax = 3, 2, 8
    kc, ks, vc, vs, kr, vr = _fill(q, b, hkv, lmax, [lmax], mode, 1)
    torch.cuda.synchronize()
    for cache, scales, rows in ((kc, ks, kr), (vc, vs, vr)):
        ref_q, ref_s = att.kv_quantize(to_np(rows.permute(1, 2, 0, 3)), mode)
        assert np.array_equal(cache.cpu().numpy(), ref_q) and np.array_equal(scales.cpu().numpy(), ref_s)


def test_append_flags(q):
    b, hkv, lmax = 2, 1, 4
    kc, ks, vc, vs = _empty_cache(b, hkv, lmax)
    k = torch.randn(b, hkv, 128, device=DEV).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    q.kv_append_fp8(k, k, torch.tensor([1, 4], dtype=torch.int32, device=DEV), kc, ks, vc, vs, dev_status=st)
    assert q.get_last_device_status(st) & q.DEV_BAD_INDEX
    assert not kc[1].any()  # the out-of-range slot wrote nothing
    k[0, 0, 3] = float("nan")
    st.zero_()
    q.kv_append_fp8(k, k, torch.tensor([0, 0], dtype=torch.int32, device=DEV), kc, ks, vc, vs, dev_status=st)
    assert q.get_last_device_status(st) & q.DEV_NONFINITE


def _check(q, b, hq, hkv, lmax, lens, seed, mode=0):
    kc, ks, vc, vs, _, _ = _fill(q, b, hkv, lmax, lens, mode, seed)
    qq = inputs.activations(b * hq, 128, inputs.derive_seed(0, "kv", seed, "q"), device=DEV).reshape(b, hq, 128)
    lt = torch.tensor(lens, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = q.attention_decode_fp8(qq, kc, ks, vc, vs, lt, dev_status=st)
    assert q.get_last_device_status(st) == 0
    ref = att.attention_decode(to_np(qq), kc.cpu().numpy(), ks.cpu().numpy(), vc.cpu().numpy(), vs.cpu().numpy(),
                               np.array(lens))
    ok, nerr, worst = oracle.linear.within_tolerance(to_np(o), ref)
    assert ok, f"normwise {nerr:.3e}, worst element ratio {worst:.3f}"


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (32, 8), (16, 2)])
def test_group_ratios(q, hq, hkv):
    _check(q, 3, hq, hkv, 300, [1, 300, 257], 2)


@pytest.mark.parametrize("lens", [[5, 0, 511, 512, 513], [256, 255, 1, 700, 64]])
def test_ragged_lengths(q, lens):
    _check(q, len(lens), 8, 2, 704, lens, 3, mode=1)


def test_single_token_returns_value_row(q):
    b, hq, hkv, lmax = 2, 8, 2, 4
    kc, ks, vc, vs, _, vr = _fill(q, b, hkv, lmax, [1, 1], 0, 4)
    qq = torch.randn(b, hq, 128, device=DEV).to(torch.bfloat16)
    o = q.attention_decode_fp8(qq, kc, ks, vc, vs, torch.ones(b, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    v0 = att.kv_dequantize(vc[:, :, 0].cpu().numpy(), vs[:, :, 0].cpu().numpy())
    ref = np.repeat(v0, hq // hkv, axis=1)
    assert np.array_equal(to_np(o), oracle.formats.bf16_rne(ref.astype(np.float32)))


def test_8b_decode_batch_sampled(q):
    """64 sequences, lengths 2048..4096, 32 query / 8 KV heads: every
    sequence's outputs for two sampled query heads checked."""
    b, hq, hkv, lmax = 64, 32, 8, 4096
    g = np.random.default_rng(9)
    lens = g.integers(lmax // 2, lmax + 1, b)
    kr = inputs.activations(b * hkv * lmax, 128, inputs.derive_seed(0, "kv8b", "k"), device=DEV)
    vr = inputs.activations(b * hkv * lmax, 128, inputs.derive_seed(0, "kv8b", "v"), device=DEV)
    kq, ks = q.quantize_fp8_a1x128(kr)
    vq, vs = q.quantize_fp8_a1x128(vr)
    kc, vc = kq.view(b, hkv, lmax, 128), vq.view(b, hkv, lmax, 128)
    ksc, vsc = ks.view(b, hkv, lmax), vs.view(b, hkv, lmax)
    qq = inputs.activations(b * hq, 128, inputs.derive_seed(0, "kv8b", "q"), device=DEV).reshape(b, hq, 128)
    o = q.attention_decode_fp8(qq, kc, ksc, vc, vsc, torch.from_numpy(lens.astype(np.int32)).to(DEV))
    torch.cuda.synchronize()
    heads = [0, 13]
    for bi in range(0, b, 7):
        ref = att.attention_decode(to_np(qq[bi:bi + 1, heads[0]:heads[0] + 4]), kc[bi:bi + 1, 0:1].cpu().numpy(),
                                   ksc[bi:bi + 1, 0:1].cpu().numpy(), vc[bi:bi + 1, 0:1].cpu().numpy(),
                                   vsc[bi:bi + 1, 0:1].cpu().numpy(), lens[bi:bi + 1])
        ok, nerr, worst = oracle.linear.within_tolerance(to_np(o[bi:bi + 1, 0:4]), ref)
        assert ok, f"seq {bi}: normwise {nerr:.3e}, worst {worst:.3f}"
        g3 = heads[1] // 4
        ref = att.attention_decode(to_np(qq[bi:bi + 1, 4 * g3:4 * g3 + 4]), kc[bi:bi + 1, g3:g3 + 1].cpu().numpy(),
                                   ksc[bi:bi + 1, g3:g3 + 1].cpu().numpy(), vc[bi:bi + 1, g3:g3 + 1].cpu().numpy(),
                                   vsc[bi:bi + 1, g3:g3 + 1].cpu().numpy(), lens[bi:bi + 1])
        ok, nerr, worst = oracle.linear.within_tolerance(to_np(o[bi:bi + 1, 4 * g3:4 * g3 + 4]), ref)
        assert ok, f"seq {bi} group {g3}: normwise {nerr:.3e}, worst {worst:.3f}"

"""GPU parity of the token log-probabilities and importance-sampling weights
against the float64 oracle.

Tolerances (derived from the arithmetic): the kernel sums exp(x - max) in
fp32 over each thread's share (about V / 256 terms in sequence, then a tree),
so the relative error of the sum is at most a few hundred units of 2^-24, and
exp / log are hardware approximations with relative error about 2^-22.  The
log-probability is then within 1e-4 absolute (plus 1e-6 relative for the
final fp32 subtraction); a weight exp(d) inherits that as a relative error, so
weights are checked within 2e-4 relative."""

import numpy as np
import pytest
import torch

import oracle
from oracle import rollout_is as ris
from quantized_rl_rollout_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
LP_REL, LP_ABS = 1e-6, 1e-4
W_REL, W_ABS = 2e-4, 1e-30


@pytest.fixture(scope="module")
def q():
    from quantized_rl_rollout_gb300 import build, qrr

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    qrr.lib()
    return qrr


def _case(t, v, seed, pad_every=0):
    lg = inputs.logits(t, v, inputs.derive_seed(0, "is", t, v, seed), device=DEV)
    tok = inputs.sampled_tokens(lg, inputs.derive_seed(0, "is-tok", t, v, seed))
    if pad_every:
        tok[::pad_every] = -1
    return lg, tok


def _check(q, lg, tok, cap=0.0):
    ref_lp = ris.token_logprobs(lg.float().cpu().numpy(), tok.cpu().numpy())
    # the rollout engine's log-probabilities: the same numbers, slightly off
    rollout = inputs.jitter(torch.from_numpy(ref_lp).to(DEV), 7, 0.02)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lp, w = q.token_logprobs_is(lg, tok, rollout, cap, dev_status=st)
    assert q.get_last_device_status(st) == 0
    ok, worst = ris.within(lp.cpu().numpy(), ref_lp, LP_REL, LP_ABS)
    assert ok, f"logp worst ratio {worst:.3f}"
    ref_w = ris.is_weights(ref_lp, rollout.cpu().numpy(), tok.cpu().numpy(), cap)
    ok, worst = ris.within(w.cpu().numpy(), ref_w, W_REL, W_ABS)
    assert ok, f"w worst ratio {worst:.3f}"


@pytest.mark.parametrize("t,v", [(1, 1), (5, 7), (33, 1000), (64, 4096), (300, 32000), (7, 8195)])
def test_shapes(q, t, v):
    lg, tok = _case(t, v, 1, pad_every=5 if t > 5 else 0)
    _check(q, lg, tok)
    _check(q, lg, tok, cap=2.0)


def test_full_vocabulary_sampled_rows(q):
    """4096 tokens over a 128256-entry vocabulary (an 8B-class model's), the
    benchmark's launch; 64 rows checked against the oracle."""
    t, v = 4096, 128256
    lg, tok = _case(t, v, 2)
    rollout = inputs.jitter(torch.zeros(t, device=DEV), 3, 1.0)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lp, w = q.token_logprobs_is(lg, tok, rollout, 5.0, dev_status=st)
    assert q.get_last_device_status(st) == 0
    rows = np.unique(np.concatenate([[0, t - 1], np.random.default_rng(4).integers(0, t, 62)]))
    rt = torch.from_numpy(rows).to(DEV)
    ref_lp = ris.token_logprobs(lg[rt].float().cpu().numpy(), tok[rt].cpu().numpy())
    ok, worst = ris.within(lp[rt].cpu().numpy(), ref_lp, LP_REL, LP_ABS)
    assert ok, f"logp worst ratio {worst:.3f}"
    ref_w = ris.is_weights(ref_lp, rollout[rt].cpu().numpy(), tok[rt].cpu().numpy(), 5.0)
    ok, worst = ris.within(w[rt].cpu().numpy(), ref_w, W_REL, W_ABS)
    assert ok, f"w worst ratio {worst:.3f}"


def test_closed_forms(q):
    v = 1000
    lg = torch.full((4, v), 3.0, dtype=torch.bfloat16, device=DEV)
    tok = torch.tensor([0, 999, -1, 500], dtype=torch.int32, device=DEV)
    lp = q.token_logprobs_is(lg, tok)
    assert np.allclose(lp.cpu().numpy(), [-np.log(v), -np.log(v), 0.0, -np.log(v)], atol=LP_ABS)
    # masked vocabulary entries (-inf) take no probability
    lg[:, 1:] = float("-inf")
    lp = q.token_logprobs_is(lg, torch.tensor([0, 0, 0, 0], dtype=torch.int32, device=DEV))
    assert np.allclose(lp.cpu().numpy(), 0.0, atol=LP_ABS)
    # equal log-probabilities give weight 1, and the cap truncates
    lp, w = q.token_logprobs_is(lg, torch.zeros(4, dtype=torch.int32, device=DEV),
                                torch.full((4,), -np.log(8.0), device=DEV), 3.0)
    assert np.allclose(w.cpu().numpy(), 3.0, rtol=W_REL)


def test_flags(q):
    lg, tok = _case(8, 512, 9)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    tok2 = tok.clone()
    tok2[3] = 512  # out of the vocabulary
    lp = q.token_logprobs_is(lg, tok2, dev_status=st)
    assert q.get_last_device_status(st) & q.DEV_BAD_INDEX
    assert lp[3].item() == 0.0
    for bad in (float("nan"), float("inf")):
        lg2 = lg.clone()
        lg2[5, 100] = bad
        st.zero_()
        q.token_logprobs_is(lg2, tok, dev_status=st)
        assert q.get_last_device_status(st) & q.DEV_NONFINITE, bad


def test_nan_beside_masked_entries(q):
    """A NaN in a stretch of -inf logits (which the block max skips) is still reported."""
    lg = torch.full((2, 1024), float("-inf"), dtype=torch.bfloat16, device=DEV)
    lg[:, 900] = 1.0
    lg[1, 40] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lp = q.token_logprobs_is(lg, torch.tensor([900, 900], dtype=torch.int32, device=DEV), dev_status=st)
    assert q.get_last_device_status(st) & q.DEV_NONFINITE
    assert abs(lp[0].item()) <= LP_ABS

"""Pins of the oracle's token log-probabilities and importance-sampling
weights against things other than itself: closed forms (uniform rows, two-way
rows as a softplus), brute force in plain Python on tiny rows, the
normalisation invariant, shift invariance, overflow-free extremes, masked
vocabulary entries, and planted mistakes that a pin must catch."""

import math

import numpy as np
import pytest

import oracle
from oracle import rollout_is as ris


def test_uniform_row_is_minus_log_v():
    for v in (1, 2, 7, 128256):
        lp = ris.token_logprobs(np.full((3, v), 2.5, np.float32), np.array([0, v - 1, v // 2]))
        assert np.allclose(lp, -math.log(v), rtol=0, atol=1e-12)


def test_two_way_row_is_softplus():
    g = np.random.default_rng(0)
    for _ in range(50):
        a, b = g.normal(0, 20, 2)
        lp = ris.token_logprobs(np.array([[a, b]]), np.array([0]))[0]
        # log(e^a / (e^a + e^b)) = -log(1 + e^(b - a)), written the stable way round
        d = b - a
        ref = -(d + math.log1p(math.exp(-d))) if d > 0 else -math.log1p(math.exp(d))
        assert abs(lp - ref) <= 1e-12 * max(1.0, abs(ref))


def test_brute_force_tiny_rows():
    g = np.random.default_rng(1)
    logits = g.normal(0, 3, (5, 9))
    toks = g.integers(0, 9, 5)
    lp = ris.token_logprobs(logits, toks)
    for t in range(5):
        z = sum(math.exp(float(x)) for x in logits[t])
        ref = float(logits[t, toks[t]]) - math.log(z)
        assert abs(lp[t] - ref) <= 1e-12


def test_probabilities_sum_to_one_and_shift_invariance():
    g = np.random.default_rng(2)
    row = g.normal(0, 5, 300)
    all_lp = ris.token_logprobs(np.tile(row, (300, 1)), np.arange(300))
    assert abs(np.exp(all_lp).sum() - 1.0) <= 1e-12
    shifted = ris.token_logprobs(np.tile(row + 1024.0, (300, 1)), np.arange(300))
    assert np.allclose(all_lp, shifted, rtol=0, atol=1e-9)


def test_extremes_and_masked_vocabulary():
    lp = ris.token_logprobs(np.array([[1e30, 0.0], [1e30, 0.0]]), np.array([0, 1]))
    assert lp[0] == 0.0 and lp[1] == -1e30
    row = np.array([[0.0, -np.inf, 0.0, -np.inf]])
    assert abs(ris.token_logprobs(row, np.array([2]))[0] + math.log(2)) <= 1e-15


def test_padding_tokens():
    lp = ris.token_logprobs(np.zeros((3, 4)), np.array([1, -1, 3]))
    assert lp[1] == 0.0 and lp[0] == -math.log(4)
    w = ris.is_weights(np.array([-1.0, -1.0, -2.0]), np.array([-1.0, 0.0, -2.0]), np.array([1, -1, 3]))
    assert w[1] == 0.0 and w[0] == 1.0 and w[2] == 1.0


def test_weights_closed_forms_and_cap():
    d = np.array([0.0, math.log(5.0), -math.log(4.0), 3.0])
    w = ris.is_weights(d, np.zeros(4), np.zeros(4, np.int64))
    assert np.allclose(w, [1.0, 5.0, 0.25, math.exp(3.0)], rtol=1e-15, atol=0)
    wc = ris.is_weights(d, np.zeros(4), np.zeros(4, np.int64), cap=2.0)
    assert np.allclose(wc, [1.0, 2.0, 0.25, 2.0], rtol=1e-15, atol=0)


def test_within_gate():
    ref = np.array([-1.0, -2.0, -300.0])
    assert ris.within(ref + 1e-7, ref, 1e-6, 1e-6)[0]
    assert not ris.within(ref + np.array([0, 0, 1e-2]), ref, 1e-6, 1e-6)[0]
    assert not ris.within(np.array([-1.0, np.nan, -300.0]), ref, 1e-6, 1e-6)[0]


@pytest.mark.parametrize("mutation", ["no_lse", "sign", "cap_max"])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    """A plausible mistake planted in the oracle fails one of the pins."""
    if mutation == "no_lse":
        monkeypatch.setattr(ris, "token_logprobs",
                            lambda logits, tokens: np.asarray(logits, np.float64)[np.arange(len(tokens)), tokens])
        with pytest.raises(AssertionError):
            test_uniform_row_is_minus_log_v()
    elif mutation == "sign":
        orig = ris.is_weights
        monkeypatch.setattr(ris, "is_weights", lambda a, b, t, cap=0.0: orig(b, a, t, cap))
        with pytest.raises(AssertionError):
            test_weights_closed_forms_and_cap()
    else:
        def bad(a, b, t, cap=0.0):
            w = np.exp(np.asarray(a, np.float64) - b)
            return np.maximum(w, cap) if cap > 0 else w
        monkeypatch.setattr(ris, "is_weights", bad)
        with pytest.raises(AssertionError):
            test_weights_closed_forms_and_cap()


def test_package_exports_module():
    assert oracle.rollout_is is ris

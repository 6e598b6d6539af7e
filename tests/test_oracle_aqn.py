"""Pins of the AQN oracle: the generator against its published known-answer
vectors, the first noise values derived by hand from them, the noise's
moments (mean 0, variance 1, the Irwin-Hall kurtosis 2.7) and independence
across elements, tensors, steps and seeds, the schedule's closed form, the
sigma = 0 identity, the bf16 rounding bound of the noisy weight, and planted
mistakes."""

import os

import numpy as np
import pytest

from oracle import aqn, fp8, nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_philox_known_answers():
    for row in _rows("philox4x32_10_kat.txt"):
        w = [int(x, 16) for x in row]
        out = aqn.philox4x32_10(*w[:6])
        assert [int(x) for x in out] == w[6:], row


def test_first_noise_values_by_hand():
    z = aqn.noise(4, seed=0, tensor=0, step=0)
    for e, centred in _rows("aqn_noise_first_elements.txt"):
        ref = np.float32(np.float32(int(centred) / 256.0) * np.float32(np.sqrt(3.0)))
        assert z[int(e)] == ref, e


def test_noise_moments():
    n = 4_000_000
    z = aqn.noise(n, seed=7, tensor=3, step=11).astype(np.float64)
    assert abs(z.mean()) < 5 / np.sqrt(n)
    assert abs(z.var() - 65535 / 65536) < 5 * np.sqrt(2.0 / n) * 1.0
    kurt = ((z - z.mean()) ** 4).mean() / z.var() ** 2
    assert abs(kurt - 2.7) < 0.02  # Irwin-Hall(4): 3 - 6 / (5 * 4)
    assert z.max() <= 2 * np.sqrt(3) and z.min() >= -2 * np.sqrt(3)


def test_streams_are_independent():
    n = 1_000_000
    base = aqn.noise(n, 1, 0, 0).astype(np.float64)
    quads = base.reshape(-1, 4)
    for a, b in ((0, 1), (0, 2), (1, 3), (2, 3)):  # the elements that share a generator call
        assert abs(np.corrcoef(quads[:, a], quads[:, b])[0, 1]) < 5 / np.sqrt(n / 4)
    for other in (aqn.noise(n, 2, 0, 0), aqn.noise(n, 1, 1, 0), aqn.noise(n, 1, 0, 1)):
        assert abs(np.corrcoef(base, other.astype(np.float64))[0, 1]) < 5 / np.sqrt(n)
    # an offset window reads the same stream
    assert np.array_equal(aqn.noise(10, 1, 0, 0, start=5), base[5:15].astype(np.float32))


def test_schedule():
    assert aqn.sigma_at(0, 100, 1e-2, 5e-4) == np.float32(1e-2)
    assert aqn.sigma_at(99, 100, 1e-2, 5e-4) == np.float32(5e-4)
    assert aqn.sigma_at(500, 100, 1e-2, 5e-4) == np.float32(5e-4)
    mid = aqn.sigma_at(50, 101, 1e-2, 1e-4)  # geometric: the midpoint is the geometric mean
    assert abs(float(mid) - 1e-3) < 1e-3 * 1e-6
    s = [float(aqn.sigma_at(i, 10, 1e-2, 1e-3)) for i in range(10)]
    assert all(a > b for a, b in zip(s, s[1:]))


def test_noisy_weight_rounding_and_identity():
    g = np.random.default_rng(0)
    w = (g.standard_normal((64, 256)) * 0.02).astype(np.float32)
    from oracle.formats import bf16_rne

    w = bf16_rne(w)
    assert np.array_equal(aqn.noisy_weight(w, 0.0, 1, 0, 0), w)
    sig = np.float32(1e-3)
    wn = aqn.noisy_weight(w, sig, 1, 0, 0)
    exact = w.astype(np.float64) + (sig * aqn.noise(w.size, 1, 0, 0).reshape(w.shape)).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert np.all(np.abs(wn - exact) <= 0.5 * ulp * (1 + 1e-6) + 2.0 ** -133)
    assert not np.array_equal(wn, w)


def test_zero_sigma_requant_is_plain_requant():
    g = np.random.default_rng(1)
    from oracle.formats import bf16_rne

    ws = [bf16_rne((g.standard_normal((32, 128)) * 0.02).astype(np.float32)) for _ in range(3)]
    for (c, s, t), w in zip(aqn.requantize_aqn(ws, 0.0, 5, 9), ws):
        rc, rs, rt = nvfp4.quantize(w)
        assert np.array_equal(c, rc) and np.array_equal(s, rs) and t == rt
    for (q, s), w in zip(aqn.requantize_aqn(ws, 0.0, 5, 9, fmt="fp8", mode=1), ws):
        rq, rs = fp8.quantize_w128x128(w, 1)
        assert np.array_equal(q, rq) and np.array_equal(s, rs)


@pytest.mark.parametrize("mutation", ["odd_half", "no_centre", "swap_rounds"])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    if mutation == "odd_half":
        orig = aqn.philox4x32_10

        def same_words(*a):  # elements of a call share words
            r = orig(*a)
            return [r[0], r[1], r[0], r[1]]

        monkeypatch.setattr(aqn, "philox4x32_10", same_words)
        with pytest.raises(AssertionError):
            test_first_noise_values_by_hand()
    elif mutation == "no_centre":
        orig = aqn.noise
        monkeypatch.setattr(aqn, "noise", lambda n, *a, **k: orig(n, *a, **k) + np.float32(0.05))
        with pytest.raises(AssertionError):
            test_noise_moments()
    else:
        monkeypatch.setattr(aqn, "M0", 0xCD9E8D57)
        monkeypatch.setattr(aqn, "M1", 0xD2511F53)
        with pytest.raises(AssertionError):
            test_philox_known_answers()

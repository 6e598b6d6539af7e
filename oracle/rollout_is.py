"""Token-level importance-sampling correction between the rollout engine's
policy and the trainer's policy.

Test infrastructure only (see the package docstring).

What it follows.  NVIDIA's FP8 recipe for RL ("NVIDIA NeMo RL behaalt 48%
snelheidswinst met end-to-end FP8-precisietraining", the paragraph on the
importance-sampling technique in "Waarom dit belangrijk is voor
AI-economie") keeps accuracy while generation and training run at different
precision by correcting, token by token, the shift between the distribution
the generation engine sampled from and the one the trainer computes.  The
page gives no formula; the readings taken here:

* a token's log-probability under a policy is its logit minus the
  log-sum-exp of the row of logits over the whole vocabulary:
  ``logp[t] = logits[t, tok[t]] - log(sum_v exp(logits[t, v]))``;
* the correction weight of a token is the likelihood ratio of the trainer's
  policy to the rollout policy, ``w[t] = exp(logp_train[t] - logp_rollout[t])``,
  optionally truncated from above at ``cap`` (``cap <= 0``: no truncation);
* a token id below zero marks padding: its log-probability and weight are 0.

Everything is float64 on the bf16-valued logits.
"""

import numpy as np


def log_softmax_rows(logits: np.ndarray) -> np.ndarray:
    """float64 log-softmax of each row (max-shifted log-sum-exp)."""
    x = np.asarray(logits, dtype=np.float64)
    mx = np.max(x, axis=-1, keepdims=True)
    lse = mx + np.log(np.sum(np.exp(x - mx), axis=-1, keepdims=True))
    return x - lse


def token_logprobs(logits: np.ndarray, tokens: np.ndarray) -> np.ndarray:
    """logp[t] of token tokens[t] under row t of logits [T, V]; 0 where tokens[t] < 0."""
    logits = np.asarray(logits, dtype=np.float64)
    tokens = np.asarray(tokens, dtype=np.int64)
    t = logits.shape[0]
    out = np.zeros(t, dtype=np.float64)
    live = np.nonzero(tokens >= 0)[0]
    if live.size:
        rows = logits[live]
        mx = np.max(rows, axis=-1)
        lse = mx + np.log(np.sum(np.exp(rows - mx[:, None]), axis=-1))
        out[live] = rows[np.arange(live.size), tokens[live]] - lse
    return out


def is_weights(logp_train: np.ndarray, logp_rollout: np.ndarray, tokens: np.ndarray, cap: float = 0.0) -> np.ndarray:
    """w[t] = min(exp(logp_train - logp_rollout), cap) (no cap when cap <= 0); 0 on padding."""
    d = np.asarray(logp_train, np.float64) - np.asarray(logp_rollout, np.float64)
    w = np.exp(d)
    if cap > 0:
        w = np.minimum(w, float(cap))
    return np.where(np.asarray(tokens) >= 0, w, 0.0)


def within(got: np.ndarray, ref: np.ndarray, rel: float, abs_: float) -> tuple:
    """Per-element |got - ref| <= abs_ + rel |ref|; returns (ok, worst ratio)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if got.shape != ref.shape:
        return False, float("inf")
    if not np.all(np.isfinite(got)):
        return False, float("inf")
    bound = abs_ + rel * np.abs(ref)
    ratio = np.abs(got - ref) / bound
    return bool(np.all(ratio <= 1.0)), float(ratio.max(initial=0.0))

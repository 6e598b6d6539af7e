"""Backward pass of the W4A16 + LoRA linear through the frozen NVFP4 weight,
in float64.

Test infrastructure only (see the package docstring).

What it follows.  QeRL trains only the LoRA adapter while the policy's
weights stay in NVFP4, and keeps the gradient computation in higher precision
("NVIDIA and MIT Collaborate on QeRL", Key Features, "Stable Backpropagation";
"QeRL: Beyond Efficiency", abstract).  Jet-RL keeps the backward pass in BF16
because 8-bit gradients collapse ("Jet-RL: Enabling On-Policy FP8 RL with
Unified Training and Rollout Precision Flow", Quick Overview).  For the
forward ``y = x . W_hat^T + (alpha / r) (x . A^T) . B^T`` and an upstream
gradient dY = dL/dy [M, N], the chain rule gives (W_hat frozen: no dW):

    dX = dY . W_hat + (alpha / r) (dY . B) . A        [M, K]
    dA = (alpha / r) (dY . B)^T . x                   [r, K]
    dB = (alpha / r) dY^T . (x . A^T)                 [N, r]

Readings: dX is returned to the layer below in bf16 (Jet-RL's BF16 backward),
dA and dB in fp32 (the adapter's gradients, summed over every token, are kept
at the precision the optimizer works in); here everything is float64 with no
intermediate rounding.
"""

import numpy as np

from . import nvfp4


def lora_backward(dy, x, codes, scales, s_t, a, b, alpha: float):
    """(dX [M, K], dA [r, K], dB [N, r]) in float64."""
    dy = np.asarray(dy, np.float64)
    x = np.asarray(x, np.float64)
    w_hat = nvfp4.dequantize(codes, scales, s_t)
    dx = dy @ w_hat
    if a is None or b is None or np.asarray(a).shape[0] == 0:
        return dx, None, None
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    c = float(alpha) / a.shape[0]
    u = dy @ b  # [M, r]
    dx = dx + c * (u @ a)
    da = c * (u.T @ x)
    db = c * (dy.T @ (x @ a.T))
    return dx, da, db


def lora_backward_dx_rows(dy_rows, w_hat, a, b, alpha: float):
    """dX for the given dY rows (full W_hat; for sampled checks of large layers)."""
    dy = np.asarray(dy_rows, np.float64)
    dx = dy @ np.asarray(w_hat, np.float64)
    if a is not None and b is not None and np.asarray(a).shape[0] > 0:
        a64 = np.asarray(a, np.float64)
        dx = dx + (float(alpha) / a64.shape[0]) * ((dy @ np.asarray(b, np.float64)) @ a64)
    return dx

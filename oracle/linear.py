"""The W4A16 + LoRA linear layer, in float64.

Test infrastructure only (see the package docstring).

What it follows.  QeRL runs the policy with NVFP4 weights and a LoRA adapter,
keeping activations, logits and gradients in higher precision ("NVIDIA and MIT
Collaborate on QeRL", Key Features, "Stable Backpropagation", and the
paragraph after them; "QeRL: Beyond Efficiency", abstract: NVFP4 combined with
LoRA).  With nn.Linear orientation (W is [N = out, K = in]) and the usual LoRA
orientation (A is [r, K], B is [N, r]) the layer is

    y = x . W_hat^T + (alpha / r) . (x . A^T) . B^T

where W_hat is the dequantized NVFP4 weight.  Everything here is float64 with
no intermediate rounding; a GPU result in bf16 is compared to it by tolerance.
"""

import numpy as np

from . import nvfp4


def lora_down(x: np.ndarray, a: np.ndarray) -> np.ndarray:
    """t = x . A^T  ([M, r], float64)."""
    return np.asarray(x, np.float64) @ np.asarray(a, np.float64).T


def linear_nvfp4_lora(x, codes, scales, s_t, a=None, b=None, alpha: float = 0.0):
    """y [M, N] float64 for bf16-valued x [M, K] and an NVFP4 weight.

    ``a``/``b`` may be None (no adapter); ``alpha / r`` multiplies the
    adapter term, r being the adapter rank (rows of ``a``).
    """
    x64 = np.asarray(x, np.float64)
    w_hat = nvfp4.dequantize(codes, scales, s_t)
    y = x64 @ w_hat.T
    if a is not None and b is not None and np.asarray(a).shape[0] > 0:
        r = np.asarray(a).shape[0]
        y = y + (float(alpha) / r) * (lora_down(x64, a) @ np.asarray(b, np.float64).T)
    return y


def linear_rows(x_rows, w_hat_rows, a=None, b_rows=None, alpha: float = 0.0):
    """Sampled outputs: y[m, n] for the given x rows and dequantized W rows.

    Same formula as ``linear_nvfp4_lora``; the caller passes the rows of
    W_hat (and of B) it wants, so large layers can be checked on a sample.
    """
    x64 = np.asarray(x_rows, np.float64)
    y = x64 @ np.asarray(w_hat_rows, np.float64).T
    if a is not None and b_rows is not None and np.asarray(a).shape[0] > 0:
        r = np.asarray(a).shape[0]
        y = y + (float(alpha) / r) * (lora_down(x64, a) @ np.asarray(b_rows, np.float64).T)
    return y


def within_tolerance(y, y_ref, norm_tol: float = 5e-3, elem_tol: float = 1e-2):
    """The acceptance test for a bf16 output against the float64 result.

    Normwise ``||y - y_ref||_F / ||y_ref||_F <= norm_tol`` and per element
    ``|y - y_ref| <= elem_tol * (|y_ref| + rms(y_ref))``.  Returns
    ``(ok, normwise_error, worst_element_ratio)``.
    """
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    if y_ref.size == 0:
        return True, 0.0, 0.0
    ref_norm = np.linalg.norm(y_ref)
    err = np.abs(y - y_ref)
    norm_err = float(np.linalg.norm(err) / ref_norm) if ref_norm > 0 else float(np.linalg.norm(err))
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    bound = elem_tol * (np.abs(y_ref) + rms)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err > 0, np.inf, 0.0))
    worst = float(np.max(ratio))
    ok = bool(np.all(np.isfinite(y))) and norm_err <= norm_tol and worst <= 1.0
    return ok, norm_err, worst

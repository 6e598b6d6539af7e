"""Seeded synthetic inputs for the linear-layer path (data only, no arithmetic
of the method).

Both the tests (for the CPU oracle) and the benchmark draw their tensors from
here, so the oracle and the CUDA path see the same bytes.  This module only
draws random numbers and rounds them to bf16; it quantizes nothing.

Recipe (workload shapes follow an 8B-class and a 32B-class decoder layer set):

* weights: ``N(0, 0.02)``; then 0.1% of the entries (positions drawn
  uniformly; the rare duplicate draw just hits the same entry once) are
  multiplied by 20 to make outliers; then rounded to bf16;
* decode activations: ``N(0, 1)`` in bf16;
* prefill / FP8 activations: ``N(0, 1)`` with 1% of the K channels (columns)
  multiplied by 10, in bf16;
* LoRA factors: A [r, K] and B [N, r] ``N(0, 0.01)`` in bf16, alpha = 2 r;
* weight update after a training step: ``W' = bf16(W + N(0, 1e-4))``;
* logits of a vocabulary row: ``N(0, 2)`` in bf16; the sampled token of a row
  by the Gumbel-max rule; the rollout engine's log-probabilities as the
  trainer's plus ``N(0, 0.02)`` (a second engine's numbers).

Every tensor has its own stream: ``torch.Generator`` seeded with
``derive_seed(seed, *labels)``.  Draws are made on the device the tensor is
wanted on, so the same seed gives different (but fixed) numbers on the CPU
and on a GPU; a test that compares the two always hands the oracle a host
copy of the very tensor the GPU used.
"""

import zlib

import torch


def derive_seed(seed: int, *labels) -> int:
    """A 63-bit seed from a base seed and labels (config, layer, tensor kind)."""
    text = "/".join([str(int(seed))] + [str(x) for x in labels])
    return (zlib.crc32(text.encode()) * 0x9E3779B1 + int(seed)) & 0x7FFFFFFFFFFFFFFF


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def weight(n: int, k: int, seed: int, device="cpu", std: float = 0.02,
           outlier_frac: float = 1e-3, outlier_mult: float = 20.0) -> torch.Tensor:
    """bf16 [n, k] weight with a sprinkling of x20 outliers."""
    g = _gen(device, seed)
    w = torch.randn(n, k, generator=g, device=device, dtype=torch.float32)
    w.mul_(std)
    count = int(round(outlier_frac * n * k))
    if count:
        idx = torch.randint(0, n * k, (count,), generator=g, device=device)
        flat = w.view(-1)
        flat[idx] = flat[idx] * outlier_mult
    return w.to(torch.bfloat16)


def activations(m: int, k: int, seed: int, device="cpu", channel_outlier_frac: float = 0.0,
                channel_mult: float = 10.0) -> torch.Tensor:
    """bf16 [m, k] activations ~N(0,1), optionally with scaled outlier channels."""
    g = _gen(device, seed)
    x = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
    count = int(round(channel_outlier_frac * k))
    if count:
        cols = torch.randperm(k, generator=g, device=device)[:count]
        x[:, cols] *= channel_mult
    return x.to(torch.bfloat16)


def lora(r: int, k: int, n: int, seed: int, device="cpu", std: float = 0.01):
    """(A bf16 [r, k], B bf16 [n, r], alpha = 2 r)."""
    g = _gen(device, seed)
    a = (torch.randn(r, k, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    b = (torch.randn(n, r, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return a, b, float(2 * r)


def logits(t: int, v: int, seed: int, device="cpu", std: float = 2.0) -> torch.Tensor:
    """bf16 [t, v] logits ~N(0, std)."""
    g = _gen(device, seed)
    return (torch.randn(t, v, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def sampled_tokens(lg: torch.Tensor, seed: int) -> torch.Tensor:
    """int32 [t]: one token per row drawn from softmax(row) by the Gumbel-max
    rule (the token a sampling rollout would emit)."""
    g = _gen(lg.device, seed)
    u = torch.rand(lg.shape, generator=g, device=lg.device, dtype=torch.float32).clamp_(1e-20, 1.0)
    return (lg.float() - torch.log(-torch.log(u))).argmax(dim=-1).to(torch.int32)


def jitter(x: torch.Tensor, seed: int, std: float) -> torch.Tensor:
    """x + N(0, std) in fp32 (a second engine's slightly different numbers)."""
    g = _gen(x.device, seed)
    return x.float() + torch.randn(x.shape, generator=g, device=x.device, dtype=torch.float32) * std


def updated(w: torch.Tensor, seed: int, std: float = 1e-4) -> torch.Tensor:
    """The trainer's update of a bf16 weight: bf16(W + N(0, std))."""
    g = _gen(w.device, seed)
    noise = torch.randn(w.shape, generator=g, device=w.device, dtype=torch.float32) * std
    return (w.float() + noise).to(torch.bfloat16)

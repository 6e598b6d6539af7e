"""Workload shapes of the linear-layer path (nn.Linear orientation: N = out, K = in).

* tiny: one [512, 256] weight, 16 tokens, LoRA r = 8, alpha = 16;
* an 8B-class decoder layer (hidden 4096, 32 query / 8 key-value heads of
  128, MLP 14336): q/o 4096x4096, k/v 1024x4096, gate/up 14336x4096,
  down 4096x14336; decode at 1, 8 and 64 tokens with LoRA r = 32; prefill at
  4096 tokens; FP8 at 4096 tokens;
* a 32B-class stack: 64 layers of hidden 5120 (q/o 5120x5120, k/v
  1024x5120, gate/up 27648x5120, down 5120x27648), decode at 64 tokens with
  LoRA r = 64.
"""

from dataclasses import dataclass


@dataclass(frozen=True)
class Layer:
    name: str
    n: int
    k: int


def decoder_layer(hidden: int, kv: int, mlp: int):
    return (
        Layer("q", hidden, hidden),
        Layer("k", kv, hidden),
        Layer("v", kv, hidden),
        Layer("o", hidden, hidden),
        Layer("gate", mlp, hidden),
        Layer("up", mlp, hidden),
        Layer("down", hidden, mlp),
    )


LAYERS_8B = decoder_layer(4096, 1024, 14336)
LAYERS_32B = decoder_layer(5120, 1024, 27648)
STACK_32B_DEPTH = 64

TINY = dict(n=512, k=256, m=16, r=8, alpha=16.0, seed=0)
DECODE_8B = dict(tokens=(1, 8, 64), r=32, seed=0)
PREFILL_8B = dict(tokens=4096, r=32, seed=0)
FP8_8B = dict(tokens=4096, seed=0)
DECODE_32B = dict(tokens=64, r=64, depth=STACK_32B_DEPTH, seed=0)


def elements(layers) -> int:
    return sum(l.n * l.k for l in layers)

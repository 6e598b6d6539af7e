"""GB300-native low-precision policy-weight linear layer for RL rollout.

NVFP4 W4A16 + BF16 LoRA linear, blockwise FP8 quantize + GEMM and per-step
re-quantization, as hand-written CUDA for sm_103a behind a C ABI
(``include/qrr.h``).  ``quantized_rl_rollout_gb300.qrr`` is the thin ctypes
binding; importing this package loads nothing until a binding function is
first called.
"""

__all__ = ["configs", "inputs"]

"""Re-quantization of every weight after a training step.

Test infrastructure only (see the package docstring).

What it follows.  The FP8 recipe recalibrates the quantization scales after
every training step because RL keeps updating the policy weights ("NVIDIA NeMo
RL behaalt 48% snelheidswinst ...", section "Praktische prestatiewinsten",
second paragraph); QeRL's rollout policy is likewise the NVFP4 image of the
current weights.  Reading: recalibration uses the current step's absmax only
(no scale history, no delayed scaling), so re-quantizing an updated tensor is
the same as quantizing it from scratch.
"""

from . import nvfp4, fp8

FORMAT_NVFP4 = 0
FORMAT_FP8_W128 = 1


def requantize(weights, fmt: int, mode: int = fp8.SCALE_FP32):
    """Quantize each bf16-valued float32 matrix of ``weights`` from scratch."""
    out = []
    for w in weights:
        if fmt == FORMAT_NVFP4:
            out.append(nvfp4.quantize(w))
        elif fmt == FORMAT_FP8_W128:
            out.append(fp8.quantize_w128x128(w, mode))
        else:
            raise ValueError("unknown format")
    return out

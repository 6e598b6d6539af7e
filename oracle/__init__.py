"""CPU oracle for the low-precision policy-weight linear layer of RL rollout.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library under
``quantized_rl_rollout_gb300`` and its Python binding) imports, links or runs
this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may.

It is a plain, slow, obviously-correct restatement of what the layer computes,
written in numpy:

* ``formats``  -- the E2M1 and E4M3 number grids and round-to-nearest-even onto
  them (NVFP4 element codes, NVFP4 block scales and FP8 codes);
* ``nvfp4``    -- NVFP4 weight quantization (per-tensor FP32 scale, one E4M3
  scale per 16 consecutive elements along K, E2M1 codes) and dequantization;
* ``linear``   -- the W4A16 + LoRA linear ``y = x.dequant(Wq)^T +
  (alpha/r).(x.A^T).B^T`` in float64;
* ``fp8``      -- blockwise E4M3 quantization (128x128 weight tiles, 1x128
  activation row blocks; FP32 or power-of-two scales) and the blockwise-scaled
  GEMM in float64;
* ``requant``  -- re-quantization of every weight of a layer set after a
  training step;
* ``rollout_is`` -- token log-probabilities from a row of logits and the
  token-level importance-sampling weights between rollout and trainer;
* ``aqn``      -- adaptive quantization noise: counter-based noise added to the
  masters before re-quantization, with its schedule;
* ``lora_backward`` -- the backward pass of the linear through the frozen
  NVFP4 weight: dX, dA, dB;
* ``attention`` -- decode attention over an E4M3 key/value cache with 1x128
  row scales.

Sources.  The pages describe QeRL ("QeRL: Beyond Efficiency -- Quantization-
enhanced Reinforcement Learning for LLMs", abstract; "NVIDIA and MIT Collaborate
on QeRL", Key Features and the paragraph after them) and NVIDIA's NeMo RL FP8
recipe ("NVIDIA NeMo RL behaalt 48% snelheidswinst met end-to-end
FP8-precisietraining", sections "De technische doorbraak" and "Praktische
prestatiewinsten").  The pages name NVFP4 but never spell out its bit layout;
the layout used here is the standard one (E2M1 codes, E4M3 block scales over 16
elements, one FP32 tensor scale).  Where the pages leave a step open, each
function states the reading it takes.

Every rounding decision is made on an IEEE float32 value, exactly as numpy's
float32 arithmetic (correctly rounded, subnormals kept) produces it; sums of
products are formed in float64.
"""

from . import formats, nvfp4, fp8, linear, requant, rollout_is, aqn, lora_backward, attention  # noqa: F401

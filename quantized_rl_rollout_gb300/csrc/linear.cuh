// Argument block and launchers of the linear-path kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace qrr {

struct LinearArgs {
  const uint16_t* x;      // bf16 [M, K]
  const uint8_t* codes;   // [N, K/2]
  const uint8_t* scales;  // [N, K/16] E4M3
  const float* tensor_scale;
  const uint16_t* A;  // bf16 [r, K] (nullable when r == 0)
  const uint16_t* B;  // bf16 [N, r]
  const float* t;     // fp32 [M, r] LoRA down projection (workspace)
  void* y;            // bf16 [M, N]
  int64_t M, N, K;
  int r;
  float lora_scale;  // alpha / r
};

cudaError_t launch_lora_down_simt(const void* x, const void* A, int64_t M, int64_t K, int r, float* t,
                                  cudaStream_t stream);
cudaError_t launch_linear_simt(const LinearArgs& a, cudaStream_t stream);

struct Fp8GemmArgs {
  const uint8_t* qa;  // [M, K]
  const float* sa;    // [M, K/128]
  const uint8_t* qw;  // [N, K]
  const float* sw;    // [ceil(N/128), K/128]
  void* y;            // bf16 [M, N]
  int64_t M, N, K;
};

cudaError_t launch_fp8_gemm_tc(const Fp8GemmArgs& a, int32_t* status, cudaStream_t stream);

}  // namespace qrr

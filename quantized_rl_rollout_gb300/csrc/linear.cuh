// Argument block and launchers of the linear-path kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda.h>

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

// ---- tensor-core W4A16 linear (linear_tc.cu) ----

constexpr int kMaxW4Layers = 8;

struct W4Layer {
  CUtensorMap tx;      // x (bf16) or its f16 image [M, K], box [BN, 64], 128 B swizzle
  CUtensorMap tcodes;  // packed codes u8 [N, K/2], box [128, 32]
  CUtensorMap tt;      // LoRA t' bf16 [M, 64 * lora_chunks], box [BN, 64], 128 B swizzle
  CUtensorMap tscales;  // block scales u8 [N, K/16], box [128, 16] (256-wide K stages)
  const uint8_t* scales;
  const float* tensor_scale;
  const uint16_t* B;  // LoRA B [N, r], r <= 64
  const int* pexp;    // per-token power-of-two pre-scale (f16 path) or null
  __nv_bfloat16* y;
  float* partial;      // [splits, M, N] when splits > 1
  uint32_t* counters;  // [m_tiles * n_tiles], zero before the launch
  int M, N, K, r, lora_chunks;
  int n_tiles, m_tiles, splits, kcps;  // kcps: pipeline stages (BK-wide K slices) per split
  int first_unit;
};

struct W4Params {
  W4Layer layer[kMaxW4Layers];
  int count;
  int total_units;
  int32_t* status;
};

// Prologue of one layer: x -> f16 rows (f16 path) and the LoRA down
// projection t = x . A^T, split over 512-wide K slices whose fp32 partials
// the last slice of each rank group sums in slice order into t'.
struct PrepArgs {
  const uint16_t* x;  // bf16 [M, K]
  const uint16_t* A;  // bf16 [r, K]
  const float* tensor_scale;
  __half* x16;          // f16 [M, K] (f16 path)
  int* pexp;            // [M] (f16 path)
  __nv_bfloat16* t;     // [M, t_cols]: (high, low) bf16 of (alpha/r) t / g per rank
  float* tpart;         // [ks, M, r] fp32 partials
  uint32_t* tickets;    // [ceil(r/8)], zero before the launch
  int64_t M, K;
  int r, t_cols, ks;
  float lora_scale;
  int32_t* status;
  int first_cta;  // this layer's first CTA in the launch
};

struct PrepBatch {
  PrepArgs a[kMaxW4Layers];
  int count;
};

// Tensor-core LoRA down projection for many tokens (lora_tc.cu).
struct LoraDownLayer {
  CUtensorMap tx;  // x bf16 [M, K], box [128, 64], 128 B swizzle
  CUtensorMap ta;  // LoRA A bf16 [r, K], box [R, 64], 128 B swizzle
  __nv_bfloat16* t;  // [M, t_cols]
  const float* tensor_scale;
  int M, K, r, R, t_cols;  // R: r rounded up to a multiple of 16
  float lora_scale;
  int first_cta;
};

struct LoraDownBatch {
  LoraDownLayer l[kMaxW4Layers];
  int count;
  int32_t* status;
};

cudaError_t launch_lora_down_tc(LoraDownBatch& b, cudaStream_t stream);

int w4_bn_for(int64_t M);
int w4_bk_for(int64_t M);
cudaError_t launch_lora_prep(PrepBatch& b, bool f16, cudaStream_t stream);
cudaError_t launch_w4a16_tc(W4Params& p, int bn, bool f16, cudaStream_t stream);

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

// Job descriptors and host launchers of the quantizer kernels (quant.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "aqn.cuh"
#include "common.cuh"

namespace qrr {

constexpr int kMaxJobs = 48;          // tensors per grouped launch (kernel parameters stay < 4 KB)

struct Nvfp4Job {
  const uint16_t* W;  // bf16 [N, K]
  uint8_t* codes;     // [N, K/2]
  uint8_t* scales;    // [N, K/16]
  float* tensor_scale;
  int64_t N, K;
  int64_t first_amax_chunk, first_encode_chunk;
  uint32_t tensor;  // index of the tensor in its call (the noise stream of adaptive quantization noise)
};

struct Nvfp4Batch {
  Nvfp4Job job[kMaxJobs];
  int count;
  int64_t total_amax_chunks, total_encode_chunks;
  uint32_t* amax_bits;  // workspace: one word per job
  int32_t* status;
  AqnParams aqn;        // sigma 0: no noise
};

struct Fp8WJob {
  const uint16_t* W;  // bf16 [N, K]
  uint8_t* q;         // [N, K]
  float* scales;      // [ceil(N/128), K/128]
  int64_t N, K;
  int64_t first_tile;
  uint32_t tensor;
};

struct Fp8WBatch {
  Fp8WJob job[kMaxJobs];
  int count;
  int mode;
  int64_t total_tiles;
  int32_t* status;
  AqnParams aqn;
};

int grid_for(int64_t work_units, int per_sm);
cudaError_t launch_nvfp4(Nvfp4Batch& batch, cudaStream_t stream);
cudaError_t launch_fp8_a1x128(const void* x, int64_t M, int64_t K, uint8_t* q, float* scales, int mode,
                              int32_t* status, cudaStream_t stream);
cudaError_t launch_fp8_w128(Fp8WBatch& batch, cudaStream_t stream);
cudaError_t launch_round_probe(const float* in, int64_t n, int fmt, uint8_t* out, cudaStream_t stream);
cudaError_t launch_aqn_noise_probe(float* out, int64_t n, int64_t start, uint32_t tensor, const AqnParams& a,
                                   cudaStream_t stream);

}  // namespace qrr

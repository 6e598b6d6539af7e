// CUDA-core blockwise-scaled FP8 GEMM, the device-side correctness baseline:
//   y[m,n] = sum_kb sa[m,kb] sw[n/128,kb] sum_{k in kb} e4m3(qa[m,k]) e4m3(qw[n,k])
// ("NVIDIA NeMo RL behaalt 48% ...", section "De technische doorbraak":
// FP8 linear layers over 1x128 activation and 128x128 weight blocks).
// Each 128-wide block sum is formed in fp32 (the E4M3 products are exact),
// then scaled and added to the fp32 result.
#include "linear.cuh"

namespace qrr {

namespace {
constexpr int TM = 64, TN = 64, TK = 32;
}

// 256 threads, a 64x64 output tile, 4x4 outputs per thread.
__global__ void __launch_bounds__(256) fp8_gemm_simt_kernel(Fp8GemmArgs a) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Ws[TK][TN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TM, n0 = static_cast<int64_t>(blockIdx.x) * TN;
  float acc[4][4] = {}, part[4][4] = {};
  const int64_t kblocks = a.K / 128;
  for (int64_t kb = 0; kb < kblocks; ++kb) {
    for (int kc = 0; kc < 128; kc += TK) {
      // stage a 64 x 32 slice of each operand, decoded to fp32, K-major in smem
      for (int i = threadIdx.x; i < TM * TK; i += 256) {
        const int r = i / TK, k = i % TK;
        const int64_t gm = m0 + r, gn = n0 + r, gk = kb * 128 + kc + k;
        As[k][r] = gm < a.M ? e4m3_to_f32(a.qa[gm * a.K + gk]) : 0.0f;
        Ws[k][r] = gn < a.N ? e4m3_to_f32(a.qw[gn * a.K + gk]) : 0.0f;
      }
      __syncthreads();
#pragma unroll 8
      for (int k = 0; k < TK; ++k) {
        float av[4], wv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = As[k][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) wv[j] = Ws[k][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], wv[j], part[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t gm = m0 + ty * 4 + i;
      const float sa = gm < a.M ? a.sa[gm * kblocks + kb] : 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t gn = n0 + tx * 4 + j;
        const float sw = gn < a.N ? a.sw[(gn / 128) * kblocks + kb] : 0.0f;
        acc[i][j] = fmaf(__fmul_rn(sa, sw), part[i][j], acc[i][j]);
        part[i][j] = 0.0f;
      }
    }
  }
  __nv_bfloat16* y = static_cast<__nv_bfloat16*>(a.y);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + ty * 4 + i;
    if (gm >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t gn = n0 + tx * 4 + j;
      if (gn < a.N) y[gm * a.N + gn] = __float2bfloat16_rn(acc[i][j]);
    }
  }
}

cudaError_t launch_fp8_gemm_simt(const Fp8GemmArgs& a, cudaStream_t stream) {
  if (a.M == 0 || a.N == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((a.N + TN - 1) / TN), static_cast<unsigned>((a.M + TM - 1) / TM));
  fp8_gemm_simt_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace qrr

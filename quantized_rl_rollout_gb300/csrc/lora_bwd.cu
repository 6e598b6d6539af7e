// Backward pass of the W4A16 + LoRA linear through the frozen NVFP4 weight:
// the operand preparation and the adapter gradients.
//
//   dX = dY . W_hat + (alpha/r) (dY . B) . A
//   dA = (alpha/r) (dY . B)^T . x,   dB = (alpha/r) dY^T . (x . A^T)
//
// ("NVIDIA and MIT Collaborate on QeRL", Key Features, "Stable
// Backpropagation": only the adapter is trained and its gradients stay
// precise; "Jet-RL ...", Quick Overview: the backward pass stays in BF16.)
//
// The call runs as
//   1. prep: W_q^T [K, N] in bf16, where W_q = e2m1(code) e4m3(s_b) is exact
//      in bf16 (at most six significant bits) and s_t is left to the GEMM's
//      epilogue; the adapter factors rearranged for the tensor cores: A^T
//      with every column doubled [K, 2r] (against the (high, low) bf16 pairs
//      of the rank-r projections) and B^T [r, N];
//   2. the rank-r projections u' = (alpha/r) (dY . B) / g and
//      t' = (alpha/r) (x . A^T) / g (g = s_t, or 1 when s_t = 0) on the
//      tensor cores (the forward's LoRA-down kernel), as (high, low) pairs;
//   3. dX = g (dY . W_q + u' . A) on the tensor cores (gemm_bf16_tc.cu);
//   4. dA[j, k] = g sum_m u'[m, j] x[m, k] and dB[n, j] = g sum_m dY[m, n] t'[m, j]
//      on the CUDA cores in fp32: token slices in parallel, partials summed
//      in slice order, so the result does not depend on timing.
#include <cuda_bf16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

namespace {

// |e2m1| values by magnitude code
__device__ __forceinline__ float e2m1_value(uint32_t nib) {
  const uint32_t m = nib & 7u;
  const float mag = m < 4 ? 0.5f * static_cast<float>(m) : (m < 6 ? static_cast<float>(m - 2) : (m == 6 ? 4.0f : 6.0f));
  return (nib & 8u) ? -mag : mag;
}

constexpr int kT = 64;  // transpose tile: 64 weight rows x 64 K

int grid_for_elems(int64_t n) {
  int dev = 0, sms = kSMs;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t ctas = (n + 255) / 256, cap = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(ctas < 1 ? 1 : (ctas < cap ? ctas : cap));
}

}  // namespace

// WT[k][n] = e2m1(code[n][k]) e4m3(scale[n][k / 16]) in bf16 (exact).
__global__ void __launch_bounds__(256) nvfp4_transpose_dequant_kernel(const uint8_t* __restrict__ codes,
                                                                      const uint8_t* __restrict__ scales, int N, int K,
                                                                      __nv_bfloat16* __restrict__ wt) {
  __shared__ __nv_bfloat16 tile[kT][kT + 8];  // [k][n], rows padded against bank conflicts
  const int n0 = blockIdx.y * kT, k0 = blockIdx.x * kT;
  // 64 rows x 32 code bytes: thread t takes 8 bytes (16 K values) of row t / 4
  const int t = threadIdx.x;
  const int rn = t >> 2, part = t & 3;
  const int n = n0 + rn;
  if (n < N) {
    const uint2 cw = __ldg(reinterpret_cast<const uint2*>(codes + static_cast<int64_t>(n) * (K / 2) + k0 / 2) + part);
    const float s = e4m3_to_f32(__ldg(scales + static_cast<int64_t>(n) * (K / 16) + k0 / 16 + part));
    const uint32_t w[2] = {cw.x, cw.y};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t nib = (w[i >> 3] >> (4 * (i & 7))) & 0xFu;
      tile[16 * part + i][rn] = __float2bfloat16_rn(e2m1_value(nib) * s);  // exact product
    }
  }
  __syncthreads();
  // 64 output rows (k) of 64 bf16 (128 bytes): thread t writes 16 bytes
  for (int idx = t; idx < kT * 8; idx += 256) {
    const int kl = idx >> 3, seg = idx & 7;
    const int nn = n0 + 8 * seg;
    if (nn >= N) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(&tile[kl][8 * seg]);
    *reinterpret_cast<uint4*>(wt + static_cast<int64_t>(k0 + kl) * N + nn) = v;
  }
}

// AT2[k][c] = A[c / 2][k] for c < 2r, 0 up to t_cols; BT[j][n] = B[n][j].
__global__ void lora_factor_transpose_kernel(const uint16_t* __restrict__ A, const uint16_t* __restrict__ B, int N,
                                             int K, int r, int t_cols, uint16_t* __restrict__ at2,
                                             uint16_t* __restrict__ bt) {
  const int64_t n_at = static_cast<int64_t>(K) * t_cols, n_bt = static_cast<int64_t>(r) * N;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_at + n_bt;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (i < n_at) {
      const int k = static_cast<int>(i / t_cols), c = static_cast<int>(i % t_cols);
      at2[i] = c < 2 * r ? __ldg(A + static_cast<int64_t>(c >> 1) * K + k) : uint16_t(0);
    } else {
      const int64_t e = i - n_at;
      const int j = static_cast<int>(e / N), n = static_cast<int>(e % N);
      bt[e] = __ldg(B + static_cast<int64_t>(n) * r + j);
    }
  }
}

// Adapter gradient partials: for one slice of tokens [m0, m0 + mlen),
//   part[s][j][c] = sum_m X[m][c] (hi + lo)(tp[m][2j], tp[m][2j + 1])
// X bf16 [M][C]; tp the (high, low) bf16 pairs [M][t_cols].  CTA: 128
// columns x all r ranks, staged 32 tokens at a time in shared memory; each
// thread keeps a register tile of 4 columns x 4 ranks (x 2 for r > 32), so
// every pair of 16-byte shared loads feeds 16 (or 32) FMAs.
__global__ void __launch_bounds__(256) lora_grad_partial_kernel(const uint16_t* __restrict__ X,
                                                                const uint16_t* __restrict__ tp, int M, int C, int r,
                                                                int t_cols, int m_per_slice, float* __restrict__ part) {
  __shared__ __align__(16) float xs[32][128];
  __shared__ __align__(16) float us[32][64];
  const int c0 = blockIdx.x * 128, s = blockIdx.y;
  const int m_begin = s * m_per_slice, m_end = min(M, m_begin + m_per_slice);
  const int cg = threadIdx.x & 31, jg = threadIdx.x >> 5;  // columns 4 cg .. 4 cg + 3; ranks 4 jg .. 4 jg + 3 (+ 32)
  const int halves = r > 32 ? 2 : 1;
  float acc[2][4][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[h][a][b] = 0.0f;
  for (int mb = m_begin; mb < m_end; mb += 32) {
    const int mn = min(32, m_end - mb);
    // x chunk: 32 rows x 128 bf16 (16 vectors of 8 per row)
    for (int idx = threadIdx.x; idx < 32 * 16; idx += 256) {
      const int rr = idx >> 4, seg = idx & 15;
      float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (rr < mn && c0 + 8 * seg < C) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(X + static_cast<int64_t>(mb + rr) * C + c0) + seg);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] = bf16_lo(w[e]);
          v[2 * e + 1] = bf16_hi(w[e]);
        }
      }
      *reinterpret_cast<float4*>(&xs[rr][8 * seg]) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(&xs[rr][8 * seg + 4]) = make_float4(v[4], v[5], v[6], v[7]);
    }
    // rank projections: 32 rows x r values (hi + lo), zero past r
    for (int idx = threadIdx.x; idx < 32 * 64; idx += 256) {
      const int rr = idx >> 6, j = idx & 63;
      float u = 0.0f;
      if (rr < mn && j < r) {
        const uint32_t pw = __ldg(reinterpret_cast<const uint32_t*>(tp + static_cast<int64_t>(mb + rr) * t_cols) + j);
        u = bf16_lo(pw) + bf16_hi(pw);
      }
      us[rr][j] = u;
    }
    __syncthreads();
    for (int mm = 0; mm < mn; ++mm) {
      const float4 x4 = *reinterpret_cast<const float4*>(&xs[mm][4 * cg]);
      const float xv[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h < halves) {
          const float4 u4 = *reinterpret_cast<const float4*>(&us[mm][32 * h + 4 * jg]);
          const float uv[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[h][a][b] = fmaf(xv[a], uv[b], acc[h][a][b]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int j = 32 * h + 4 * jg + b;
      if (h < halves && j < r && c0 + 4 * cg < C)
        *reinterpret_cast<float4*>(part + (static_cast<int64_t>(s) * r + j) * C + c0 + 4 * cg) =
            make_float4(acc[h][0][b], acc[h][1][b], acc[h][2][b], acc[h][3][b]);
    }
}

// out = g * sum over slices (in slice order) of part[s][j][c]; layout
// [j][c] (transposed = false: dA [r][K]) or [c][j] (true: dB [N][r]).
__global__ void lora_grad_reduce_kernel(const float* __restrict__ part, int slices, int r, int C,
                                        const float* __restrict__ tensor_scale, bool transposed,
                                        float* __restrict__ out) {
  const float st = *tensor_scale;
  const float g = st > 0.0f ? st : 1.0f;
  const int64_t n = static_cast<int64_t>(r) * C;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float acc = 0.0f;
    for (int s = 0; s < slices; ++s) acc += __ldg(part + static_cast<int64_t>(s) * n + i);
    const int j = static_cast<int>(i / C), c = static_cast<int>(i % C);
    out[transposed ? static_cast<int64_t>(c) * r + j : i] = g * acc;
  }
}

int lora_grad_slices(int64_t M, int64_t C) {
  const int64_t col_ctas = (C + 127) / 128;
  int64_t s = (8 * kSMs + col_ctas - 1) / col_ctas;  // about eight CTAs per SM: their loads cover each other's latency
  s = s < (M + 31) / 32 ? s : (M + 31) / 32;
  return static_cast<int>(s < 1 ? 1 : s);
}

cudaError_t launch_lora_backward_prep(const uint8_t* codes, const uint8_t* scales, const void* A, const void* B,
                                      int N, int K, int r, int t_cols, __nv_bfloat16* wt, uint16_t* at2, uint16_t* bt,
                                      cudaStream_t stream) {
  if (N > 0 && K > 0) {
    const dim3 grid(static_cast<unsigned>(K / kT), static_cast<unsigned>((N + kT - 1) / kT));
    nvfp4_transpose_dequant_kernel<<<grid, 256, 0, stream>>>(codes, scales, N, K, wt);
  }
  if (r > 0) {
    const int64_t n = static_cast<int64_t>(K) * t_cols + static_cast<int64_t>(r) * N;
    lora_factor_transpose_kernel<<<grid_for_elems(n), 256, 0, stream>>>(static_cast<const uint16_t*>(A),
                                                                        static_cast<const uint16_t*>(B), N, K, r,
                                                                        t_cols, at2, bt);
  }
  return cudaGetLastError();
}

cudaError_t launch_lora_grad(const void* X, const uint16_t* tp, int M, int C, int r, int t_cols,
                             const float* tensor_scale, bool transposed, float* part, float* out,
                             cudaStream_t stream) {
  const int slices = lora_grad_slices(M, C);
  const int m_per = (M + slices - 1) / slices;
  const dim3 grid(static_cast<unsigned>((C + 127) / 128), static_cast<unsigned>(slices));
  lora_grad_partial_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(X), tp, M, C, r, t_cols, m_per,
                                                     part);
  lora_grad_reduce_kernel<<<grid_for_elems(static_cast<int64_t>(r) * C), 256, 0, stream>>>(
      part, slices, r, C, tensor_scale, transposed, out);
  return cudaGetLastError();
}

}  // namespace qrr

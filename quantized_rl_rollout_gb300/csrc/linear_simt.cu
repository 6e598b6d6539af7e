// Reference-grade CUDA-core kernels of the linear path: the LoRA down
// projection t = x . A^T (fp32) and a straightforward W4A16 + LoRA linear.
//
// These are the correctness baseline the tensor-core kernels are checked
// against on the device, and the path taken for shapes the tensor-core
// kernels do not cover.  Layer formula ("NVIDIA and MIT Collaborate on QeRL",
// paragraph after Key Features; "QeRL: Beyond Efficiency", abstract):
//   y = s_t * sum_k x[m,k] e2m1(c[n,k]) e4m3(s_b[n,k/16]) + (alpha/r) sum_j t[m,j] B[n,j]
#include "linear.cuh"

namespace qrr {

// t[m, j] = sum_k x[m, k] A[j, k]; one warp per (m, j), 16-byte loads.
__global__ void __launch_bounds__(256) lora_down_simt_kernel(const uint16_t* __restrict__ x,
                                                             const uint16_t* __restrict__ A, int64_t M,
                                                             int64_t K, int r, float* __restrict__ t) {
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= M * r) return;
  const int64_t m = warp / r;
  const int j = static_cast<int>(warp % r);
  const uint4* xr = reinterpret_cast<const uint4*>(x + m * K);
  const uint4* ar = reinterpret_cast<const uint4*>(A + static_cast<int64_t>(j) * K);
  float acc = 0.0f;
  for (int64_t v = lane; v < K / 8; v += 32) {
    const uint4 a = __ldg(ar + v), b = __ldg(xr + v);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc = fmaf(bf16_lo(aw[i]), bf16_lo(bw[i]), acc);
      acc = fmaf(bf16_hi(aw[i]), bf16_hi(bw[i]), acc);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) t[m * r + j] = acc;
}

// One warp per (weight row n, group of 8 tokens).  Lane l covers K elements
// [1024 i + 32 l, +32) in step i: 16 bytes of codes and two block scales.
__global__ void __launch_bounds__(256) linear_simt_kernel(LinearArgs a) {
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t groups = (a.M + 7) / 8;
  if (warp >= a.N * groups) return;
  const int64_t n = warp / groups;
  const int64_t m0 = (warp % groups) * 8;
  const int mcount = static_cast<int>(a.M - m0 < 8 ? a.M - m0 : 8);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  const uint8_t* crow = a.codes + n * (a.K / 2);
  const uint8_t* srow = a.scales + n * (a.K / 16);
  for (int64_t k0 = lane * 32; k0 < a.K; k0 += 1024) {
    const uint4 c = __ldg(reinterpret_cast<const uint4*>(crow + k0 / 2));
    const float s0 = e4m3_to_f32(__ldg(srow + k0 / 16)), s1 = e4m3_to_f32(__ldg(srow + k0 / 16 + 1));
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    float w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t nib = (cw[i >> 3] >> (4 * (i & 7))) & 0xFu;
      const uint32_t mag = nib & 7u;
      const float v = mag < 2 ? 0.5f * static_cast<float>(mag)
                              : __uint_as_float((0x3F000000u + (mag << 22)));  // 1 .. 6
      w[i] = (nib & 8u ? -v : v) * (i < 16 ? s0 : s1);  // exact: <= 6 significant bits
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      if (t >= mcount) break;
      const uint4* xr = reinterpret_cast<const uint4*>(a.x + (m0 + t) * a.K + k0);
      float s = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 xv = __ldg(xr + q);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          s = fmaf(bf16_lo(xw[i]), w[8 * q + 2 * i], s);
          s = fmaf(bf16_hi(xw[i]), w[8 * q + 2 * i + 1], s);
        }
      }
      acc[t] += s;
    }
  }
#pragma unroll
  for (int t = 0; t < 8; ++t) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc[t] += __shfl_xor_sync(0xFFFFFFFFu, acc[t], o);
  }
  if (lane < mcount) {
    float v = 0.0f;
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t == lane) v = acc[t];
    const int64_t m = m0 + lane;
    float y = __fmul_rn(*a.tensor_scale, v);
    if (a.r > 0) {
      float l = 0.0f;
      for (int j = 0; j < a.r; ++j) l = fmaf(a.t[m * a.r + j], bf16bits_to_f32(a.B[n * a.r + j]), l);
      y = fmaf(a.lora_scale, l, y);
    }
    reinterpret_cast<__nv_bfloat16*>(a.y)[m * a.N + n] = __float2bfloat16_rn(y);
  }
}

cudaError_t launch_lora_down_simt(const void* x, const void* A, int64_t M, int64_t K, int r, float* t,
                                  cudaStream_t stream) {
  const int64_t warps = M * r;
  if (warps == 0) return cudaSuccess;
  lora_down_simt_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(
      static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(A), M, K, r, t);
  return cudaGetLastError();
}

cudaError_t launch_linear_simt(const LinearArgs& a, cudaStream_t stream) {
  const int64_t warps = a.N * ((a.M + 7) / 8);
  if (warps == 0) return cudaSuccess;
  linear_simt_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace qrr

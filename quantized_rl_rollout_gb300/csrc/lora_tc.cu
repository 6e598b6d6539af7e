// LoRA down projection for many tokens on the tensor cores:
//
//   t[m, j] = sum_k x[m, k] A[j, k],   t'[m, 2j] = bf16(v), t'[m, 2j+1] = bf16(v - bf16(v)),
//   v = (alpha / r) t[m, j] / g,       g = s_t (or 1 when s_t = 0)
//
// ("NVIDIA and MIT Collaborate on QeRL", Key Features: LoRA keeps the adapter
// path in higher precision; the result feeds the W4A16 GEMM's extra K
// columns.)  One CTA per (layer, 128-token tile) runs the whole K loop:
//   warp 0      TMA: x [128 x 64] and A [R x 64] (R = r rounded up to 16,
//               rows past r read as zeros), 128-byte swizzle, 6-stage ring
//   warp 1      MMA: 4 x tcgen05.mma kind::f16 (M128 x R x K16) per stage
//   warps 2..5  epilogue: thread = token row, t from TMEM -> t' row
#include <cuda_bf16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

namespace {

constexpr int kStages = 6;
constexpr int kXBytes = 128 * 128;  // [128 x 64] bf16
constexpr int kABytes = 64 * 128;   // up to [64 x 64] bf16
constexpr int kStage = kXBytes + kABytes;
constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * kStage + 256;

struct Ctl {
  uint64_t full[kStages], empty[kStages];
  uint64_t d_full;
  uint32_t tmem;
  int abort;
};

}  // namespace

__global__ void __launch_bounds__(192, 1) lora_down_tc_kernel(const __grid_constant__ LoraDownBatch b) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl& sh = *reinterpret_cast<Ctl*>(tiles + kStages * kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &sh.abort;
  int j = 0;
  while (j + 1 < b.count && b.l[j + 1].first_cta <= static_cast<int>(blockIdx.x)) ++j;
  const LoraDownLayer& L = b.l[j];
  const int m0 = (static_cast<int>(blockIdx.x) - L.first_cta) * 128;
  const int kc = L.K / 64;
  const int R = L.R;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.d_full, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  if (warp == 0) {
    if (elect_one()) {
      int issued = 0;
      for (int c = 0; c < kc; ++c) {
        const int s = c % kStages, use = c / kStages;
        if (use > 0 && !mbar_wait(&sh.empty[s], (use - 1) & 1, abort, b.status)) break;
        uint8_t* xs = tiles + s * kStage;
        mbar_arrive_expect_tx(&sh.full[s], kXBytes + R * 128);
        tma_load_2d(&L.tx, &sh.full[s], xs, c * 64, m0);
        tma_load_2d(&L.ta, &sh.full[s], xs + kXBytes, c * 64, 0);
        issued = c + 1;
      }
      volatile int no_abort = 0;
      for (int k = issued - 1; k >= 0 && k >= issued - kStages; --k)
        mbar_wait(&sh.full[k % kStages], (k / kStages) & 1, &no_abort, b.status);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      const uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, 128, static_cast<uint32_t>(R));
      bool ok = true;
      for (int c = 0; c < kc; ++c) {
        const int s = c % kStages;
        if (!mbar_wait(&sh.full[s], (c / kStages) & 1, abort, b.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t xa = smem_u32(tiles + s * kStage), ab = xa + kXBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16_ss(tmem, sw128_desc(xa + 32 * k), sw128_desc(ab + 32 * k), idesc, (c > 0 || k > 0) ? 1u : 0u);
        mma_commit(&sh.empty[s]);
      }
      mma_commit(&sh.d_full);
      volatile int no_abort = 0;
      if (!ok) mbar_wait(&sh.d_full, 0, &no_abort, b.status);
    }
  } else {
    const int q = warp & 3;
    const int m = m0 + 32 * q + lane;
    if (mbar_wait(&sh.d_full, 0, abort, b.status)) {
      tc_fence_after();
      const float st = *L.tensor_scale;
      const float g = st > 0.0f ? st : 1.0f;
      __nv_bfloat16* trow = L.t + static_cast<int64_t>(m) * L.t_cols;
      for (int c0 = 0; c0 < R; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + c0, r);
        tmem_ld_wait();
        if (m < L.M) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int jj = c0 + i;
            if (jj < L.r) {
              const float v = __fdiv_rn(L.lora_scale * __uint_as_float(r[i]), g);
              const __nv_bfloat16 hi = __float2bfloat16_rn(v);
              const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
              trow[2 * jj] = hi;
              trow[2 * jj + 1] = lo;
            }
          }
        }
      }
      if (m < L.M)
        for (int jj = 2 * L.r; jj < L.t_cols; ++jj) trow[jj] = __float2bfloat16_rn(0.0f);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

cudaError_t launch_lora_down_tc(LoraDownBatch& b, cudaStream_t stream) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(lora_down_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  int ctas = 0;
  for (int j = 0; j < b.count; ++j) {
    b.l[j].first_cta = ctas;
    ctas += static_cast<int>((b.l[j].M + 127) / 128);
  }
  if (ctas == 0) return cudaSuccess;
  lora_down_tc_kernel<<<ctas, 192, kSmem, stream>>>(b);
  return cudaGetLastError();
}

}  // namespace qrr

// bf16 GEMM on the 5th-generation tensor cores with an extra contraction
// block, for the backward pass of the W4A16 + LoRA linear:
//
//   y[m, c] = g * ( sum_n A[m, n] B[c, n]  +  sum_j A2[m, j] B2[c, j] )
//
// Both operands are K-major (row-major with the contraction index
// contiguous), y is bf16 [M, C] row-major, g is a device scalar (1 when it is
// 0 or absent).  For dX = dY . W_hat + (alpha/r) (dY . B) . A, A = dY,
// B = (e2m1 x e4m3 part of W_hat)^T, A2 / B2 the LoRA term's factors, g = s_t.
// ("NVIDIA and MIT Collaborate on QeRL", Key Features, "Stable
// Backpropagation": LoRA keeps the gradient path precise; "Jet-RL ...", Quick
// Overview: the backward pass stays in BF16.)
//
// Persistent CTAs, one per SM, take 128 x 256 output tiles in turn:
//   warp 0      TMA: per 64-wide contraction stage, A [128 x 64] and B [256 x 64]
//               bf16 (128-byte swizzle) into a 4-stage ring; the last stages of
//               a tile read A2 / B2
//   warp 1      MMA: 4 x tcgen05.mma kind::f16 (M128 N256 K16) per stage into
//               one of two 256-column TMEM accumulators
//   warps 2..9  epilogue: the finished accumulator scaled by g, rounded to
//               bf16 and stored, while the MMAs fill the other accumulator
#include <cuda_bf16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int THREADS = 10 * 32;
constexpr uint32_t TMEM_COLS = 512;  // two 256-column fp32 accumulators
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256;

struct Params {
  CUtensorMap ta, ta2;  // A [M, K], A2 [M, K2]: box 128 x 64
  CUtensorMap tb, tb2;  // B [C, K], B2 [C, K2]: box 256 x 64
  const float* g;
  __nv_bfloat16* y;
  int M, C, ks_main, ks_extra;  // 64-wide contraction stages of each block
  int32_t* status;
};

struct Shared {
  uint64_t full[STAGES], empty[STAGES];
  uint64_t d_full[2], d_empty[2];
  uint64_t done;
  uint32_t tmem;
  int abort;
};

}  // namespace

__global__ void __launch_bounds__(THREADS, 1) gemm_bf16_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared& sh = *reinterpret_cast<Shared*>(tiles + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c_tiles = (p.C + BN - 1) / BN;
  const int total = c_tiles * ((p.M + BM - 1) / BM);
  const int ks = p.ks_main + p.ks_extra;
  volatile int* abort = &sh.abort;
  // output columns vary fastest, so the CTAs working at once share A rows
  auto tile_of = [&](int t, int& m0, int& c0) {
    m0 = (t / c_tiles) * BM;
    c0 = (t % c_tiles) * BN;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.d_full[b], 1);
      mbar_init(&sh.d_empty[b], 8);
    }
    mbar_init(&sh.done, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (elect_one()) {
      tma_prefetch_desc(&p.ta);
      tma_prefetch_desc(&p.tb);
      int issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int m0, c0;
        tile_of(t, m0, c0);
        for (int k = 0; k < ks; ++k, ++issued) {
          const int s = issued % STAGES, use = issued / STAGES;
          if (issued >= STAGES && !mbar_wait(&sh.empty[s], (use - 1) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh.full[s], STAGE_BYTES);
          uint8_t* a = tiles + s * STAGE_BYTES;
          const bool main = k < p.ks_main;
          const int kx = (main ? k : k - p.ks_main) * BK;
          tma_load_2d(main ? &p.ta : &p.ta2, &sh.full[s], a, kx, m0);
          tma_load_2d(main ? &p.tb : &p.tb2, &sh.full[s], a + A_BYTES, kx, c0);
        }
      }
      volatile int no_abort = 0;
      for (int i = issued - 1; i >= 0 && i >= issued - STAGES; --i)
        mbar_wait(&sh.full[i % STAGES], (i / STAGES) & 1, &no_abort, p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (elect_one()) {
      constexpr uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, BM, BN);
      int stage = 0, tiles_done = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tiles_done) {
        const int b = tiles_done & 1, buse = tiles_done >> 1;
        if (buse > 0 && !mbar_wait(&sh.d_empty[b], (buse - 1) & 1, abort, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + BN * b;
        for (int k = 0; k < ks; ++k, ++stage) {
          const int s = stage % STAGES, use = stage / STAGES;
          if (!mbar_wait(&sh.full[s], use & 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(tiles + s * STAGE_BYTES), bb = a + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16_ss(d, sw128_desc(a + 32 * kk), sw128_desc(bb + 32 * kk), idesc, (k > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&sh.empty[s]);
        }
        if (!ok) break;
        mma_commit(&sh.d_full[b]);
      }
      mma_commit(&sh.done);
      volatile int no_abort = 0;
      mbar_wait(&sh.done, 0, &no_abort, p.status);
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int q = warp & 3, h = (warp - 2) >> 2;  // lane quarter, column half
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const float st = p.g ? *p.g : 0.0f;
    const float g = st > 0.0f ? st : 1.0f;
    int tiles_done = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tiles_done) {
      int m0, c0;
      tile_of(t, m0, c0);
      const int b = tiles_done & 1;
      const int row = m0 + 32 * q + lane;
      const int col0 = c0 + 128 * h;
      if (!mbar_wait(&sh.d_full[b], (tiles_done >> 1) & 1, abort, p.status) || *abort) break;
      tc_fence_after();
      uint32_t packed[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_addr + BN * b + 128 * h + 32 * c, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat162 b2 =
              __floats2bfloat162_rn(__uint_as_float(r[2 * i]) * g, __uint_as_float(r[2 * i + 1]) * g);
          packed[16 * c + i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.d_empty[b]);
      if (row < p.M && col0 < p.C) {
        uint4* dst = reinterpret_cast<uint4*>(p.y + static_cast<int64_t>(row) * p.C + col0);
#pragma unroll
        for (int v = 0; v < 16; ++v)
          dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

cudaError_t launch_gemm_bf16_tc(const Bf16GemmArgs& a, int32_t* status, cudaStream_t stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  Params p{};
  if (!make_tmap_2d(&p.ta, a.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.M, a.K, a.K * 2, BM, BK,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&p.tb, a.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.C, a.K, a.K * 2, BN, BK,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (a.K2 > 0) {
    if (!make_tmap_2d(&p.ta2, a.A2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.M, a.K2, a.K2 * 2, BM, BK,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d(&p.tb2, a.B2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.C, a.K2, a.K2 * 2, BN, BK,
                      CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    p.ta2 = p.ta;  // never read
    p.tb2 = p.tb;
  }
  p.g = a.g;
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.M = static_cast<int>(a.M);
  p.C = static_cast<int>(a.C);
  p.ks_main = static_cast<int>((a.K + BK - 1) / BK);
  p.ks_extra = static_cast<int>((a.K2 + BK - 1) / BK);
  p.status = status;
  const int64_t tiles = ((a.C + BN - 1) / BN) * ((a.M + BM - 1) / BM);
  if (tiles == 0) return cudaSuccess;
  int dev = 0, sms = kSMs;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);
  gemm_bf16_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qrr

// Blockwise-scaled FP8 GEMM on the 5th-generation tensor cores (tcgen05).
//
//   y[m,n] = sum_kb sa[m,kb] sw[n/128,kb] sum_{k in kb} e4m3(qa[m,k]) e4m3(qw[n,k])
//
// ("NVIDIA NeMo RL behaalt 48% ...", section "De technische doorbraak": FP8
// linear layers over 1x128 activation and 128x128 weight blocks.)
//
// One CTA computes a 128 (tokens) x 256 (weight rows) output tile.
//   warp 0      TMA producer: per 128-wide K block, a 128x128 B tile of qa and
//               a 256x128 B tile of qw into a 4-stage ring (128 B swizzle)
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::f8f6f4 (M128 N256 K32) per K
//               block into one of two TMEM partial buffers (256 fp32 columns each)
//   warps 2..9  epilogue: read the finished partial of block kb from TMEM,
//               multiply by sa[m,kb] * sw[n/128,kb] and add into fp32 registers
//               (the "promotion" of each block sum), then store bf16.
// The two partial buffers let the tensor core fill block kb+1 while the
// epilogue promotes block kb.
#include <cuda_bf16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4;
constexpr int A_BYTES = BM * BK;                  // 16 KB
constexpr int B_BYTES = BN * BK;                  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;    // 48 KB
constexpr int THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;  // two 256-column fp32 partials
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256;

struct Params {
  CUtensorMap ta;  // qa [M, K] u8, box 128 x 128
  CUtensorMap tb;  // qw [N, K] u8, box 256 x 128
  const float* sa;
  const float* sw;
  __nv_bfloat16* y;
  int M, N, K;
  int32_t* status;
};

struct Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t done;
  uint32_t tmem;
  int abort;
};

}  // namespace

__global__ void __launch_bounds__(THREADS, 1) fp8_gemm_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared& sh = *reinterpret_cast<Shared*>(tiles + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int kblocks = p.K / BK;
  volatile int* abort = &sh.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.tfull[b], 1);
      mbar_init(&sh.tempty[b], 8);
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
      for (int kb = 0; kb < kblocks; ++kb) {
        const int s = kb % STAGES, use = kb / STAGES;
        if (kb >= STAGES && !mbar_wait(&sh.empty[s], (use - 1) & 1, abort, p.status)) break;
        mbar_arrive_expect_tx(&sh.full[s], STAGE_BYTES);
        uint8_t* a = tiles + s * STAGE_BYTES;
        tma_load_2d(&p.ta, &sh.full[s], a, kb * BK, m0);
        tma_load_2d(&p.tb, &sh.full[s], a + A_BYTES, kb * BK, n0);
        issued = kb + 1;
      }
      // drain: every stage's last load has landed before the CTA may exit
      for (int kb = issued - 1; kb >= 0 && kb >= issued - STAGES; --kb) {
        volatile int no_abort = 0;
        mbar_wait(&sh.full[kb % STAGES], (kb / STAGES) & 1, &no_abort, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (elect_one()) {
      constexpr uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, BM, BN);
      for (int kb = 0; kb < kblocks; ++kb) {
        const int s = kb % STAGES, use = kb / STAGES, buf = kb & 1, buse = kb >> 1;
        if (!mbar_wait(&sh.full[s], use & 1, abort, p.status)) break;
        if (kb >= 2 && !mbar_wait(&sh.tempty[buf], (buse - 1) & 1, abort, p.status)) break;
        tc_fence_after();
        const uint32_t a = smem_u32(tiles + s * STAGE_BYTES), b = a + A_BYTES;
        const uint32_t d = tmem + buf * BN;
#pragma unroll
        for (int k = 0; k < BK / 32; ++k) mma_fp8_ss(d, sw128_desc(a + 32 * k), sw128_desc(b + 32 * k), idesc, k);
        mma_commit(&sh.empty[s]);
        mma_commit(&sh.tfull[buf]);
      }
      // all issued MMAs have finished before TMEM is released
      mma_commit(&sh.done);
      volatile int no_abort = 0;
      mbar_wait(&sh.done, 0, &no_abort, p.status);
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int e = warp - 2, q = warp & 3, h = e >> 2;
    const int row = m0 + 32 * q + lane;
    const int col0 = n0 + 128 * h;
    const bool col_ok = col0 < p.N;
    const int ntile = col0 >> 7;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    float acc[128];
#pragma unroll
    for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
    for (int kb = 0; kb < kblocks; ++kb) {
      const int buf = kb & 1, buse = kb >> 1;
      const float sa = row < p.M ? __ldg(p.sa + static_cast<int64_t>(row) * kblocks + kb) : 0.0f;
      const float sw = col_ok ? __ldg(p.sw + static_cast<int64_t>(ntile) * kblocks + kb) : 0.0f;
      const float f = __fmul_rn(sa, sw);
      if (!mbar_wait(&sh.tfull[buf], buse & 1, abort, p.status)) break;
      tc_fence_after();
      // promotion acc += f P on the paired fp32 pipe (each half an ordinary
      // correctly rounded fp32 FMA), two TMEM loads in flight
      uint64_t f2;
      asm("mov.b64 %0, {%1, %1};" : "=l"(f2) : "f"(f));
#pragma unroll
      for (int c = 0; c < 4; c += 2) {
        uint32_t r[2][32];
        tmem_ld32(tmem + lane_addr + buf * BN + 128 * h + 32 * c, r[0]);
        tmem_ld32(tmem + lane_addr + buf * BN + 128 * h + 32 * (c + 1), r[1]);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float& a0 = acc[32 * (c + u) + j];
            float& a1 = acc[32 * (c + u) + j + 1];
            uint64_t a2, p2;
            asm("mov.b64 %0, {%1, %2};" : "=l"(a2) : "f"(a0), "f"(a1));
            asm("mov.b64 %0, {%1, %2};" : "=l"(p2) : "r"(r[u][j]), "r"(r[u][j + 1]));
            asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a2) : "l"(f2), "l"(p2));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a2));
          }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.tempty[buf]);
    }
    if (row < p.M && col_ok && !*abort) {
      uint4* dst = reinterpret_cast<uint4*>(p.y + static_cast<int64_t>(row) * p.N + col0);
#pragma unroll
      for (int v = 0; v < 16; ++v) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[8 * v + 2 * i], acc[8 * v + 2 * i + 1]);
          w[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
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

cudaError_t launch_fp8_gemm_tc(const Fp8GemmArgs& a, int32_t* status, cudaStream_t stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(fp8_gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  Params p{};
  if (!make_tmap_2d(&p.ta, a.qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.M, a.K, a.K, BM, BK,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&p.tb, a.qw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, a.K, a.K, BN, BK, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  p.sa = a.sa;
  p.sw = a.sw;
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.status = status;
  const dim3 grid(static_cast<unsigned>((a.N + BN - 1) / BN), static_cast<unsigned>((a.M + BM - 1) / BM));
  fp8_gemm_tc_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qrr

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
//      on the tensor cores, with x, dY and the projections read as MN-major
//      operands (no transposes): token slices in parallel, fp32 partials
//      summed in slice order, so the result does not depend on timing.
#include <cuda_bf16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

namespace {

int grid_for_elems(int64_t n) {
  int dev = 0, sms = kSMs;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t ctas = (n + 255) / 256, cap = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(ctas < 1 ? 1 : (ctas < cap ? ctas : cap));
}

}  // namespace

// WT[k][n] = e2m1(code[n][k]) e4m3(scale[n][k / 16]) in bf16 (exact).  A CTA
// takes 64 weight rows x kSub tiles of 128 K.  Every code and scale load of
// its tiles is issued first (one tile alone leaves too few bytes in flight to
// cover HBM latency); each tile then goes through shared memory as [k][n]
// rows of 32-bit (n, n + 1) pairs, which the CTA writes out as 128-byte rows
// of WT.  The 16-byte chunk c of row k is kept at chunk c ^ ((k / 16) mod 8):
// a warp's pair stores (eight rows 16 apart, four pairs each) and its
// 16-byte row reads then each touch every bank once.
constexpr int kTN = 64, kTK = 128;
constexpr int kSub = 1;
__global__ void __launch_bounds__(256) nvfp4_transpose_dequant_kernel(const uint8_t* __restrict__ codes,
                                                                      const uint8_t* __restrict__ scales, int N, int K,
                                                                      __nv_bfloat16* __restrict__ wt) {
  __shared__ uint4 tile[kTK][kTN / 8];
  const int t = threadIdx.x, lane = t & 31;
  const int part = lane & 7;                  // K values [16 part, 16 part + 16) of a tile
  const int pair = (t >> 5) * 4 + (lane >> 3);  // weight rows na, na + 1
  const int n0 = blockIdx.y * kTN, kb = blockIdx.x * kTK * kSub;
  const int na = n0 + 2 * pair;
  const bool rows_in = na + 1 < N;
  uint2 c0[kSub], c1[kSub];
  float s0[kSub], s1[kSub];
#pragma unroll
  for (int u = 0; u < kSub; ++u) {
    const int k0 = kb + u * kTK;
    const bool in = rows_in && k0 < K;
    const uint8_t* cr = codes + static_cast<int64_t>(na) * (K / 2) + k0 / 2 + 8 * part;
    const uint8_t* sr = scales + static_cast<int64_t>(na) * (K / 16) + k0 / 16 + part;
    c0[u] = in ? __ldg(reinterpret_cast<const uint2*>(cr)) : make_uint2(0u, 0u);
    c1[u] = in ? __ldg(reinterpret_cast<const uint2*>(cr + K / 2)) : make_uint2(0u, 0u);
    s0[u] = in ? e4m3_to_f32(__ldg(sr)) : 0.0f;
    s1[u] = in ? e4m3_to_f32(__ldg(sr + K / 16)) : 0.0f;
  }
  uint32_t* tw = reinterpret_cast<uint32_t*>(&tile[0][0]);
  const int col = (((pair >> 2) ^ part) << 2) | (pair & 3);  // word within a row: (k / 16) mod 8 = part
#pragma unroll
  for (int u = 0; u < kSub; ++u) {
    const int k0 = kb + u * kTK;
    if (k0 >= K) break;  // uniform over the CTA
    if (u > 0) __syncthreads();  // the previous tile has been read out
    // the two rows' block scales times 2^112 as one bf16x2 (exact: four
    // significant bits, at most 448 2^112)
    uint32_t s2;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(s2) : "f"(s1[u] * 0x1p112f), "f"(s0[u] * 0x1p112f));
    const uint32_t w0[2] = {c0[u].x, c0[u].y}, w1[2] = {c1[u].x, c1[u].y};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t a[4], b[4];  // f16x2 of K (2q, 2q + 1) of rows na and na + 1
      f16x2x4_from_e2m1x8(w0[h], a);
      f16x2x4_from_e2m1x8(w1[h], b);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t ra = e2m1_f16x2_rebias_bf16x2(a[q]), rb = e2m1_f16x2_rebias_bf16x2(b[q]);
        const int k = 16 * part + 8 * h + 2 * q;
        // (row na, row na + 1) at K k and k + 1, times (s0, s1): exact products
        tw[k * (kTN / 2) + col] = bmul2(__byte_perm(ra, rb, 0x5410), s2);
        tw[(k + 1) * (kTN / 2) + col] = bmul2(__byte_perm(ra, rb, 0x7632), s2);
      }
    }
    __syncthreads();
    // 128 rows of 64 bf16: four 16-byte chunks per thread
#pragma unroll
    for (int idx = t; idx < kTK * 8; idx += 256) {
      const int kl = idx >> 3, seg = idx & 7;
      const int nn = n0 + 8 * seg;
      if (nn >= N) continue;
      *reinterpret_cast<uint4*>(wt + static_cast<int64_t>(k0 + kl) * N + nn) = tile[kl][seg ^ ((kl >> 4) & 7)];
    }
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

// Adapter gradient partials on the tensor cores: for one slice of tokens
//   part[s][j][c] = sum_m X[m][c] (hi + lo)(tp[m][2j], tp[m][2j + 1])
// as D[c][c'] = sum_m X[m][c] tp[m][c'] (M = 128 columns c of X, N = t_cols
// columns of tp, K = the slice's tokens), then column pairs summed.  X and tp
// are token-major in memory, i.e. MN-major operands: TMA stages 64-token
// boxes of 64 columns (128-byte swizzle) and the MMA reads them through
// MN-major descriptors, so nothing is transposed.
//   warp 0  TMA: per 64-token stage, X [64 x 128] (two boxes) and tp [64 x t_cols]
//   warp 1  MMA: 4 x tcgen05.mma kind::f16 (M128 N t_cols K16), A and B MN-major
//   warps 2..5  the 128 x t_cols accumulator out of TMEM, pairs summed, stored
namespace {
constexpr int kGStages = 3;
constexpr int kGPerSm = 2;  // resident CTAs per SM (shared memory and TMEM allow two)
constexpr int kGA = 2 * 64 * 128;      // X stage: 2 boxes of 64 tokens x 64 columns (bf16)
constexpr int kGB = 2 * 64 * 128;      // tp stage: up to 2 boxes
constexpr int kGStage = kGA + kGB;     // 32 KB
constexpr size_t kGSmem = 1024 + kGStages * kGStage + 256;
}  // namespace

struct GradTcParams {
  CUtensorMap tx;  // X [M][C] bf16, box 64 x 64
  CUtensorMap tt;  // tp [M][t_cols] bf16, box 64 x 64
  float* part;
  int M, C, r, t_cols, m_per_slice;
  int32_t* status;
};

__global__ void __launch_bounds__(192, kGPerSm) lora_grad_tc_kernel(const __grid_constant__ GradTcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  struct Ctl {
    uint64_t full[kGStages], empty[kGStages], d_full;
    uint32_t tmem;
    int abort;
  };
  Ctl& sh = *reinterpret_cast<Ctl*>(tiles + kGStages * kGStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 128, s = blockIdx.y;
  const int m_begin = s * p.m_per_slice, m_end = min(p.M, m_begin + p.m_per_slice);
  const int steps = m_end > m_begin ? (m_end - m_begin + 63) / 64 : 0;
  const int nb = p.t_cols / 64;  // tp boxes per stage
  volatile int* abort = &sh.abort;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
    }
    mbar_init(&sh.d_full, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;
  if (warp == 0) {
    if (elect_one()) {
      int issued = 0;
      for (int k = 0; k < steps; ++k) {
        const int st = k % kGStages, use = k / kGStages;
        if (use > 0 && !mbar_wait(&sh.empty[st], (use - 1) & 1, abort, p.status)) break;
        uint8_t* a = tiles + st * kGStage;
        const int m = m_begin + 64 * k;
        mbar_arrive_expect_tx(&sh.full[st], kGA + nb * 8192);
        tma_load_2d(&p.tx, &sh.full[st], a, c0, m);
        tma_load_2d(&p.tx, &sh.full[st], a + 8192, c0 + 64, m);
        for (int b = 0; b < nb; ++b) tma_load_2d(&p.tt, &sh.full[st], a + kGA + 8192 * b, 64 * b, m);
        issued = k + 1;
      }
      volatile int no_abort = 0;
      for (int k = issued - 1; k >= 0 && k >= issued - kGStages; --k)
        mbar_wait(&sh.full[k % kGStages], (k / kGStages) & 1, &no_abort, p.status);
    }
  } else if (warp == 1) {
    if (elect_one()) {
      const uint32_t idesc = make_idesc_major(kFmtBF16, kFmtBF16, 128, static_cast<uint32_t>(p.t_cols), true, true);
      bool ok = true;
      for (int k = 0; k < steps; ++k) {
        const int st = k % kGStages;
        if (!mbar_wait(&sh.full[st], (k / kGStages) & 1, abort, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(tiles + st * kGStage), b = a + kGA;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tmem, sw128_mn_desc(a + 2048 * kk, 8192), sw128_mn_desc(b + 2048 * kk, 8192), idesc,
                      (k > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&sh.empty[st]);
      }
      mma_commit(&sh.d_full);
      volatile int no_abort = 0;
      if (!ok) mbar_wait(&sh.d_full, 0, &no_abort, p.status);
    }
  } else {
    const int q = warp & 3;
    const int c = c0 + 32 * q + lane;
    const bool ok = steps > 0 && mbar_wait(&sh.d_full, 0, abort, p.status) && !*abort;
    tc_fence_after();
    for (int cb = 0; cb < p.t_cols; cb += 32) {
      uint32_t v[32];
      if (ok) {
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + cb, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;  // an empty slice adds nothing
      }
      if (c < p.C)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = cb / 2 + i;
          if (j < p.r)
            p.part[(static_cast<int64_t>(s) * p.r + j) * p.C + c] =
                __uint_as_float(v[2 * i]) + __uint_as_float(v[2 * i + 1]);
        }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
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
  // as many token slices as keep every CTA in one wave of kGPerSm per SM
  // (rounding up would leave a few CTAs to run their whole slice afterwards)
  int64_t s = static_cast<int64_t>(kSMs) * kGPerSm / col_ctas;
  s = s < (M + 255) / 256 ? s : (M + 255) / 256;  // at least 256 tokens per slice
  if (s < 1) s = 1;
  // slices are whole 64-token stages: count only those that get tokens
  const int64_t per = ((M + s - 1) / s + 63) / 64 * 64;
  s = per > 0 ? (M + per - 1) / per : 1;
  return static_cast<int>(s < 1 ? 1 : s);
}

cudaError_t launch_lora_backward_prep(const uint8_t* codes, const uint8_t* scales, const void* A, const void* B,
                                      int N, int K, int r, int t_cols, __nv_bfloat16* wt, uint16_t* at2, uint16_t* bt,
                                      cudaStream_t stream) {
  if (N > 0 && K > 0) {
    const int kc = kTK * kSub;
    const dim3 grid(static_cast<unsigned>((K + kc - 1) / kc), static_cast<unsigned>((N + kTN - 1) / kTN));
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
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(lora_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kGSmem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int slices = lora_grad_slices(M, C);
  GradTcParams p{};
  if (!make_tmap_2d(&p.tx, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, M, C, static_cast<uint64_t>(C) * 2, 64, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&p.tt, tp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, M, t_cols, static_cast<uint64_t>(t_cols) * 2, 64, 64,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  p.part = part;
  p.M = M;
  p.C = C;
  p.r = r;
  p.t_cols = t_cols;
  p.m_per_slice = ((M + slices - 1) / slices + 63) / 64 * 64;  // whole 64-token stages per slice
  p.status = nullptr;
  const dim3 grid(static_cast<unsigned>((C + 127) / 128), static_cast<unsigned>(slices));
  lora_grad_tc_kernel<<<grid, 192, kGSmem, stream>>>(p);
  lora_grad_reduce_kernel<<<grid_for_elems(static_cast<int64_t>(r) * C), 256, 0, stream>>>(
      part, slices, r, C, tensor_scale, transposed, out);
  return cudaGetLastError();
}

}  // namespace qrr

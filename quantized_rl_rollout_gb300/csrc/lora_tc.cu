// Prologue of the W4A16 + LoRA linear: the LoRA down projection on the tensor
// cores, and (decode) the f16 image of x.
//
//   t[m, j] = sum_k x[m, k] A[j, k],   t'[m, 2j] = bf16(v), t'[m, 2j+1] = bf16(v - bf16(v)),
//   v = (alpha / r) t[m, j] / g,       g = s_t (or 1 when s_t = 0)
//
// ("NVIDIA and MIT Collaborate on QeRL", Key Features: LoRA keeps the adapter
// path in higher precision; the result feeds the W4A16 GEMM's extra K
// columns.)  Per layer, CTAs of two kinds in one launch:
//
// LoRA CTAs, one per (128-token tile, K slice):
//   warp 0      TMA: x [128 x 64] and A [R x 64] (R = r rounded up to 16;
//               rows past M or r read as zeros), 128-byte swizzle, 4-stage ring
//   warp 1      MMA: 4 x tcgen05.mma kind::f16 (M128 x R x K16) per stage
//   warps 2..5  epilogue: thread = token row.  With one slice (many tokens)
//               t goes straight from TMEM to t'.  With several (decode, few
//               tokens: the K loop is cut into 512-wide slices so the whole
//               projection runs in one wave) each slice writes fp32 partials,
//               and the last slice of the tile to finish (a ticket) sums them
//               in slice order, so the result does not depend on timing.
// x-row CTAs (decode): p_m so that max|x_m| 2^-p_m is in [2^14, 2^15), and
//   x16 = f16(x 2^-p_m), the GEMM's f16 operand.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

// Development builds (-DQRR_TRACE_BUILD) record global-timer stamps of each
// prologue CTA's phases; ordinary builds compile them away.
#ifdef QRR_TRACE_BUILD
__device__ unsigned long long qrr_ptrace_buf[256][16];
#define QRR_PSTAMP(ev)                                                               \
  do {                                                                               \
    unsigned long long t_;                                                           \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                           \
    if (blockIdx.x < 256) qrr_ptrace_buf[blockIdx.x][ev] = t_;                       \
  } while (0)
#else
#define QRR_PSTAMP(ev) \
  do {                 \
  } while (0)
#endif

namespace {

constexpr int kStages = 4;  // 97 KB: two CTAs per SM, so a decode prologue fits in one wave
constexpr int kXBytes = 128 * 128;  // [128 x 64] bf16
constexpr int kABytes = 64 * 128;   // up to [64 x 64] bf16
constexpr int kStage = kXBytes + kABytes;
constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * kStage + 256;
constexpr int kThreads = 192;
constexpr int kRowsPerCta = kThreads / 32;

struct Ctl {
  uint64_t full[kStages], empty[kStages];
  uint64_t d_full;
  uint32_t tmem;
  int abort;
  int last;
};

// t'[m, 2j], t'[m, 2j + 1] of one rank: v = scale t / g as (high, low) bf16
__device__ __forceinline__ void write_tprime(__nv_bfloat16* trow, int jj, float scale, float t, float g) {
  const float v = __fdiv_rn(scale * t, g);
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
  trow[2 * jj] = hi;
  trow[2 * jj + 1] = lo;
}

// x rows -> f16 with their power-of-two pre-scales.  The CTA's 6 warps take
// `rows` token rows (1, 2, 3 or 6), 6 / rows warps per row, with 8 loads in
// flight per thread; the row maxima meet in shared memory.
// (Layer fields are read once into registers here and in the LoRA CTAs:
// through the parameter reference they would be re-read after every store.)
__device__ void x_rows_f16(const LoraDownLayer& L, int first_row, int warp, int lane, int32_t* status) {
  __shared__ uint32_t rmax[kRowsPerCta];
  const int rows = L.x_rows_per_cta, wpr = kRowsPerCta / rows;
  const int M = L.M, K = L.K;
  const uint16_t* const xg = L.x;
  __half* const x16g = L.x16;
  int* const pexpg = L.pexp;
  const int m = first_row + warp / wpr, sub = warp % wpr;
  const int nvec = K / 8;
  if (threadIdx.x < kRowsPerCta) rmax[threadIdx.x] = 0u;
  if (threadIdx.x == 0) QRR_PSTAMP(0);
  __syncthreads();
  const uint4* xr = reinterpret_cast<const uint4*>(xg + static_cast<int64_t>(m) * K);
  if (m < M) {
    uint32_t mx = 0;
#pragma unroll 8
    for (int v = sub * 32 + lane; v < nvec; v += wpr * 32) mx = max(mx, absmax_bits8(__ldg(xr + v)));
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) atomicMax(&rmax[warp / wpr], mx);
  }
  __syncthreads();
  if (threadIdx.x == 0) QRR_PSTAMP(6);
  if (m >= M) return;
  const uint32_t mx = rmax[warp / wpr];
  int pexp = 0;
  if (mx != 0u) {
    int e;
    frexpf(bf16bits_to_f32(mx), &e);  // amax = f 2^e, 0.5 <= f < 1
    pexp = e - 15;                    // amax 2^-p in [2^14, 2^15)
  }
  if (sub == 0 && lane == 0) {
    if (mx >= 0x7F80u) flag(status, QRR_DEV_NONFINITE);
    pexpg[m] = pexp;
  }
  const Pow2Scaler sc(pexp);
  uint4* x16 = reinterpret_cast<uint4*>(x16g + static_cast<int64_t>(m) * K);
#pragma unroll 8
  for (int v = sub * 32 + lane; v < nvec; v += wpr * 32) {
    const uint4 xv = __ldg(xr + v);
    const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 h = __floats2half2_rn(sc(bf16_lo(w[i])), sc(bf16_hi(w[i])));
      o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    x16[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) QRR_PSTAMP(7);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) lora_down_tc_kernel(const __grid_constant__ LoraDownBatch b) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl& sh = *reinterpret_cast<Ctl*>(tiles + kStages * kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &sh.abort;
  int j = 0;
  while (j + 1 < b.count && b.l[j + 1].first_cta <= static_cast<int>(blockIdx.x)) ++j;
  const LoraDownLayer& L = b.l[j];
  // the GEMM that consumes t' and x16 may be scheduled now: it streams its
  // weights while this runs and waits for this grid before reading them
  griddep_launch_dependents();
  const int local = static_cast<int>(blockIdx.x) - L.first_cta;
  const int m_tiles = (L.M + 127) / 128;
  const int lora_ctas = L.r > 0 ? m_tiles * L.ks : 0;
  if (local >= lora_ctas) {  // uniform per CTA: no TMEM in this branch
    x_rows_f16(L, (local - lora_ctas) * L.x_rows_per_cta, warp, lane, b.status);
    return;
  }
  const int mt = local / L.ks, slice = local % L.ks;
  const int m0 = mt * 128;
  const int kc_all = L.K / 64;
  const int kc0 = slice * L.slice_steps;
  const int kc = min(kc_all, kc0 + L.slice_steps) - kc0;  // 64-wide K steps of this slice
  const int R = L.R;

  if (threadIdx.x == 0) {
    QRR_PSTAMP(0);
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
        tma_load_2d(&L.tx, &sh.full[s], xs, (kc0 + c) * 64, m0);
        tma_load_2d(&L.ta, &sh.full[s], xs + kXBytes, (kc0 + c) * 64, 0);
        issued = c + 1;
      }
      QRR_PSTAMP(1);
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
    const int et = threadIdx.x - 64;  // 0..127 over the epilogue warps
    const int M = L.M, r = L.r, ks = L.ks, t_cols = L.t_cols;
    const int ksp = (ks + 3) & ~3;  // partials of one output: contiguous, 16-byte rows
    const float lscale = L.lora_scale;
    __nv_bfloat16* const t = L.t;
    float* const tpart = L.tpart;
    uint32_t* const tickets = L.tickets;
    const float st = *L.tensor_scale;
    const float g = st > 0.0f ? st : 1.0f;
    bool ok = mbar_wait(&sh.d_full, 0, abort, b.status);
    if (et == 0) QRR_PSTAMP(2);
    if (lane == 0) QRR_PSTAMP(8 + q);
    if (ok) {
      tc_fence_after();
      for (int c0 = 0; c0 < R; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + c0, v);
        tmem_ld_wait();
        if (m < M) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int jj = c0 + i;
            if (jj >= r) continue;
            if (ks == 1)
              write_tprime(t + static_cast<int64_t>(m) * t_cols, jj, lscale, __uint_as_float(v[i]), g);
            else
              tpart[(static_cast<int64_t>(m) * r + jj) * ksp + slice] = __uint_as_float(v[i]);
          }
        }
      }
    }
    if (ks == 1) {
      if (ok && m < M)
        for (int jj = 2 * r; jj < t_cols; ++jj) t[static_cast<int64_t>(m) * t_cols + jj] = __float2bfloat16_rn(0.0f);
    } else {
      // every partial of this slice is written; one thread makes them visible
      // GPU-wide (cumulative over the barrier) and takes the tile's ticket
      if (lane == 0) QRR_PSTAMP(12 + q);
      named_bar(1, 128);
      if (et == 0) {
        QRR_PSTAMP(3);
        __threadfence();
        const uint32_t prev = atomicAdd(tickets + mt, 1u);
        sh.last = ok && prev == static_cast<uint32_t>(ks - 1);
        if (sh.last) __threadfence();
        QRR_PSTAMP(4);
      }
      named_bar(1, 128);
      if (sh.last) {
        // sum each output's slice partials in slice order; four outputs per
        // thread at a time with all their loads in flight
        const int rows = min(128, M - m0), n_out = rows * r, nv = ksp / 4;
        const float4* tp = reinterpret_cast<const float4*>(tpart + static_cast<int64_t>(m0) * r * ksp);
        for (int i0 = et; i0 < n_out; i0 += 512) {
          float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          for (int v0 = 0; v0 < nv; v0 += 4) {
            float4 f[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const int idx = i0 + 128 * u;
                f[u][w] = (idx < n_out && v0 + w < nv) ? __ldcg(tp + static_cast<int64_t>(idx) * nv + v0 + w)
                                                      : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
              }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int w = 0; w < 4; ++w) {
                const int s0 = 4 * (v0 + w);
                if (s0 < ks) acc[u] += f[u][w].x;
                if (s0 + 1 < ks) acc[u] += f[u][w].y;
                if (s0 + 2 < ks) acc[u] += f[u][w].z;
                if (s0 + 3 < ks) acc[u] += f[u][w].w;
              }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int idx = i0 + 128 * u;
            if (idx < n_out)
              write_tprime(t + static_cast<int64_t>(m0 + idx / r) * t_cols, idx % r, lscale, acc[u], g);
          }
        }
        const int pad = t_cols - 2 * r;
        for (int idx = et; idx < rows * pad; idx += 128)
          t[static_cast<int64_t>(m0 + idx / pad) * t_cols + 2 * r + idx % pad] = __float2bfloat16_rn(0.0f);
        if (et == 0) QRR_PSTAMP(5);
      }
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
    LoraDownLayer& L = b.l[j];
    L.first_cta = ctas;
    if (L.r > 0) ctas += ((L.M + 127) / 128) * L.ks;
    if (L.x16) {
      // few tokens: several warps per row; many: a warp per row
      L.x_rows_per_cta = L.M <= 8 ? 1 : L.M <= 32 ? 2 : kRowsPerCta;
      ctas += (L.M + L.x_rows_per_cta - 1) / L.x_rows_per_cta;
    }
  }
  if (ctas == 0) return cudaSuccess;
  lora_down_tc_kernel<<<ctas, kThreads, kSmem, stream>>>(b);
  return cudaGetLastError();
}

}  // namespace qrr

#ifdef QRR_TRACE_BUILD
extern "C" int qrr_ptrace_read(unsigned long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, qrr::qrr_ptrace_buf, sizeof(qrr::qrr_ptrace_buf)));
}
extern "C" int qrr_ptrace_clear(void) {
  static unsigned long long zeros[256 * 16] = {};
  return static_cast<int>(cudaMemcpyToSymbol(qrr::qrr_ptrace_buf, zeros, sizeof(zeros)));
}
#endif

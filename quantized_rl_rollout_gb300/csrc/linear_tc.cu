// W4A16 + LoRA linear on the 5th-generation tensor cores (tcgen05), prefill
// and decode.
//
//   y = x . W_hat^T + (alpha/r) (x . A^T) . B^T,   W_hat = e2m1(code) e4m3(s_b) s_t
//
// ("NVIDIA and MIT Collaborate on QeRL", paragraph after Key Features: NVFP4
// weight path, activations and logits in higher precision; "QeRL: Beyond
// Efficiency", abstract: NVFP4 combined with LoRA.)
//
// Design (swap-AB).  The MMA's A operand is a 128-row slice of the weight,
// dequantized by CUDA cores straight into tensor memory (TMEM); B is a tile of
// BN tokens of x staged by TMA in shared memory; D[n, m] accumulates in TMEM.
// The dequantized operand e2m1 * e4m3 (<= 6 significant bits) is exact in
// bf16 and in f16, so the tensor core forms every product exactly and sums in
// fp32; s_t is applied once in the epilogue.
//
//   warp 0      TMA: per 64-wide K chunk, x [BN x 64] (128 B swizzle) and the
//               packed codes [128 x 32 B] into an S-stage ring
//   warp 1      MMA: 4 x tcgen05.mma (M128 x BN x K16) per chunk, A from TMEM
//   warps 2..5  dequant: thread = weight row (its TMEM lane); codes from
//               shared memory, E4M3 block scales from global, 64 values per
//               chunk stored to a 4-stage TMEM ring; then the epilogue
//
// LoRA is folded into the same accumulator as extra K columns: the prologue
// writes t' = (alpha/r) t / (g 2^p) (t = x . A^T, g = s_t or 1, 2^p the
// per-token pre-scale below) split into a bf16 high part and a bf16 low part;
// the extra A columns hold [B | B].  So y = g 2^p D with no separate pass.
//
// Operand type.  Prefill (many tokens) feeds bf16 x directly and dequantizes
// to bf16.  Decode (<= 64 tokens, HBM-bound) feeds f16: the prologue rescales
// each token row by a power of two 2^-p (max |x| into [2^14, 2^15)) and
// rounds it to f16, which is exact for every element within 2^-29 of the
// row's largest magnitude; the weight dequantizes to f16 with one hardware
// conversion and one packed multiply per two values, half the cost of the
// bf16 route.  The LoRA chunks stay bf16 (their own instruction descriptor).
//
// Split-K (decode): units of (layer, 128-row tile, token tile, K range); each
// split writes an fp32 partial, and the last split to finish (a counter per
// tile) sums the partials in split order and writes y, so the result does not
// depend on timing.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

namespace {

constexpr int kBK = 64;     // K per chunk (one 128-byte bf16/f16 row of x)
constexpr int kAStages = 4;  // TMEM A ring
constexpr int kThreads = 192;

template <int BN>
struct Cfg {
  static constexpr int X_BYTES = BN * 128;
  static constexpr int C_BYTES = 128 * 32;
  static constexpr int STAGE = X_BYTES + C_BYTES;
  static constexpr int STAGES = (200 * 1024) / STAGE > 16 ? 16 : (200 * 1024) / STAGE;
  static constexpr int A_COL = BN < 32 ? 32 : BN;
  static constexpr uint32_t TMEM_COLS = (A_COL + 32 * kAStages) <= 256 ? 256 : 512;
  static constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * STAGE + 512;
};

struct SharedCtl {
  uint64_t full[16], empty[16];
  uint64_t a_full[kAStages], a_empty[kAStages];
  uint64_t d_full, d_empty, done;
  uint32_t tmem;
  int abort;
  int last;
};

__device__ __forceinline__ uint32_t f16x2_from_e2m1x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float f16_lo_to_f32(uint32_t h2) { return __half2float(__ushort_as_half(h2 & 0xFFFFu)); }
__device__ __forceinline__ float f16_hi_to_f32(uint32_t h2) { return __half2float(__ushort_as_half(h2 >> 16)); }

// 64 codes (8 words) + 4 block scales -> 32 words of the MMA A operand.
template <bool F16>
__device__ __forceinline__ void dequant64(const uint32_t (&w)[8], uint32_t scales4, uint32_t (&out)[32]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const float sv = e4m3_to_f32((scales4 >> (8 * g)) & 0xFFu);
    if constexpr (F16) {
      const uint32_t s16 = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(sv)));  // exact
      const uint32_t s2 = s16 | (s16 << 16);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t word = w[2 * g + q];
#pragma unroll
        for (int b = 0; b < 4; ++b) out[8 * g + 4 * q + b] = hmul2(f16x2_from_e2m1x2(word >> (8 * b)), s2);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t word = w[2 * g + q];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint32_t h2 = f16x2_from_e2m1x2(word >> (8 * b));
          out[8 * g + 4 * q + b] = pack_bf16x2(f16_lo_to_f32(h2) * sv, f16_hi_to_f32(h2) * sv);
        }
      }
    }
  }
}

}  // namespace

template <int BN, bool F16>
__global__ void __launch_bounds__(kThreads, 1) w4a16_tc_kernel(const __grid_constant__ W4Params p) {
  using C = Cfg<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SharedCtl& sh = *reinterpret_cast<SharedCtl*>(tiles + C::STAGES * C::STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &sh.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 5);  // MMA commit + 4 dequant warps
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&sh.a_full[s], 4);
      mbar_init(&sh.a_empty[s], 1);
    }
    mbar_init(&sh.d_full, 1);
    mbar_init(&sh.d_empty, 4);
    mbar_init(&sh.done, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  // unit -> (layer, n tile, m tile, split, chunk range)
  auto locate = [&](int u, int& j, int& nt, int& mt, int& sp, int& c0, int& nk, int& nl) {
    j = 0;
    while (j + 1 < p.count && p.layer[j + 1].first_unit <= u) ++j;
    const W4Layer& L = p.layer[j];
    const int local = u - L.first_unit;
    nt = local % L.n_tiles;
    const int rest = local / L.n_tiles;
    mt = rest % L.m_tiles;
    sp = rest / L.m_tiles;
    c0 = sp * L.kcps;
    const int kc = L.K / kBK;
    nk = min(c0 + L.kcps, kc) - c0;
    nl = (L.r > 0 && sp == L.splits - 1) ? L.lora_chunks : 0;
  };

  if (warp == 0) {
    // ------------------------------ TMA ------------------------------
    if (elect_one()) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
        int j, nt, mt, sp, c0, nk, nl;
        locate(u, j, nt, mt, sp, c0, nk, nl);
        const W4Layer& L = p.layer[j];
        for (int c = 0; c < nk + nl; ++c, ++it) {
          const int s = it % C::STAGES;
          const uint32_t use = it / C::STAGES;
          if (use > 0 && !mbar_wait(&sh.empty[s], (use - 1) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          uint8_t* xs = tiles + s * C::STAGE;
          if (c < nk) {
            mbar_arrive_expect_tx(&sh.full[s], C::X_BYTES + C::C_BYTES);
            tma_load_2d(&L.tx, &sh.full[s], xs, (c0 + c) * kBK, mt * BN);
            tma_load_2d(&L.tcodes, &sh.full[s], xs + C::X_BYTES, (c0 + c) * (kBK / 2), nt * 128);
          } else {
            mbar_arrive_expect_tx(&sh.full[s], C::X_BYTES);
            tma_load_2d(&L.tt, &sh.full[s], xs, (c - nk) * kBK, mt * BN);
          }
        }
      }
      // drain: the last load of every stage has landed
      volatile int no_abort = 0;
      for (uint32_t k = 0; k < static_cast<uint32_t>(C::STAGES) && k < it; ++k) {
        const uint32_t i = it - 1 - k;
        mbar_wait(&sh.full[i % C::STAGES], (i / C::STAGES) & 1, &no_abort, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA ------------------------------
    if (elect_one()) {
      constexpr uint32_t id_main = make_idesc(F16 ? kFmtF16 : kFmtBF16, F16 ? kFmtF16 : kFmtBF16, 128, BN);
      constexpr uint32_t id_lora = make_idesc(kFmtBF16, kFmtBF16, 128, BN);
      uint32_t it = 0, units = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x, ++units) {
        int j, nt, mt, sp, c0, nk, nl;
        locate(u, j, nt, mt, sp, c0, nk, nl);
        if (units > 0 && !mbar_wait(&sh.d_empty, (units - 1) & 1, abort, p.status)) break;
        for (int c = 0; c < nk + nl; ++c, ++it) {
          const int s = it % C::STAGES;
          const int sa = it % kAStages;
          if (!mbar_wait(&sh.full[s], (it / C::STAGES) & 1, abort, p.status) ||
              !mbar_wait(&sh.a_full[sa], (it / kAStages) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xb = smem_u32(tiles + s * C::STAGE);
          const uint32_t a0 = tmem + C::A_COL + 32 * sa;
          const uint32_t idesc = c < nk ? id_main : id_lora;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16_ts(tmem, a0 + 8 * k, sw128_desc(xb + 32 * k), idesc, (c > 0 || k > 0) ? 1u : 0u);
          mma_commit(&sh.empty[s]);
          mma_commit(&sh.a_empty[sa]);
        }
        if (!ok) break;
        mma_commit(&sh.d_full);
      }
      mma_commit(&sh.done);
      volatile int no_abort = 0;
      mbar_wait(&sh.done, 0, &no_abort, p.status);
    }
  } else {
    // ------------------------- dequant + epilogue -------------------------
    const int q = warp & 3;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    uint32_t it = 0, units = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x, ++units) {
      int j, nt, mt, sp, c0, nk, nl;
      locate(u, j, nt, mt, sp, c0, nk, nl);
      const W4Layer& L = p.layer[j];
      const int n = nt * 128 + 32 * q + lane;
      const uint8_t* srow = L.scales + static_cast<int64_t>(n) * (L.K / 16);
      uint4 sc = make_uint4(0, 0, 0, 0);
      bool ok = true;
      for (int c = 0; c < nk + nl; ++c, ++it) {
        const int s = it % C::STAGES;
        const int sa = it % kAStages;
        uint32_t out[32];
        if (c < nk) {
          const int kc = c0 + c;
          if ((c & 3) == 0 || c == 0) sc = __ldg(reinterpret_cast<const uint4*>(srow + (kc & ~3) * 4));
          if (!mbar_wait(&sh.full[s], (it / C::STAGES) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          const uint4* crow = reinterpret_cast<const uint4*>(tiles + s * C::STAGE + C::X_BYTES + (32 * q + lane) * 32);
          // the two 16-byte halves are read in lane-dependent order to spread banks
          const int h = (lane >> 2) & 1;
          const uint4 c0v = crow[h], c1v = crow[h ^ 1];
          const uint4 lo = h ? c1v : c0v, hi = h ? c0v : c1v;
          const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
          dequant64<F16>(w, sw[kc & 3], out);
        } else {
          // LoRA chunk: A columns hold [B | B] (bf16), zero past 2r.  The wait
          // on the stage keeps this warp's arrivals on `empty` in phase order.
          if (!mbar_wait(&sh.full[s], (it / C::STAGES) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          const int lc = c - nk;
          const uint16_t* brow = L.B + static_cast<int64_t>(n) * L.r;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int j0 = lc * kBK + 2 * i;
            const uint32_t b0 = j0 < 2 * L.r ? __ldg(brow + (j0 % L.r)) : 0u;
            const uint32_t b1 = j0 + 1 < 2 * L.r ? __ldg(brow + ((j0 + 1) % L.r)) : 0u;
            out[i] = b0 | (b1 << 16);
          }
        }
        if (it >= kAStages && !mbar_wait(&sh.a_empty[sa], ((it / kAStages) - 1) & 1, abort, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st32(tmem + lane_addr + C::A_COL + 32 * sa, out);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sh.a_full[sa]);
          mbar_arrive(&sh.empty[s]);
        }
      }
      if (!ok) break;
      // ------------------------------ epilogue ------------------------------
      if (!mbar_wait(&sh.d_full, units & 1, abort, p.status)) break;
      tc_fence_after();
      const float st = *L.tensor_scale;
      const float g = st > 0.0f ? st : 1.0f;
      const int m0 = mt * BN;
      float* part = L.splits > 1 ? L.partial + static_cast<int64_t>(sp) * L.M * L.N : nullptr;
      // stream D out of TMEM 16 or 32 columns (tokens) at a time
      constexpr int CW = BN == 16 ? 16 : 32;
#pragma unroll 1
      for (int cc = 0; cc < BN / CW; ++cc) {
        uint32_t r[CW];
        if constexpr (CW == 16)
          tmem_ld16(tmem + lane_addr, r);
        else
          tmem_ld32(tmem + lane_addr + 32 * cc, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          const int m = m0 + CW * cc + i;
          if (m < L.M) {
            const float sc2 = L.pexp ? __fmul_rn(g, ldexpf(1.0f, L.pexp[m])) : g;
            const float v = __uint_as_float(r[i]) * sc2;
            if (part)
              part[static_cast<int64_t>(m) * L.N + n] = v;
            else
              L.y[static_cast<int64_t>(m) * L.N + n] = __float2bfloat16_rn(v);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.d_empty);

      if (part) {
        __threadfence();
        named_bar(1, 128);
        if (warp == 2 && lane == 0) {
          uint32_t* cnt = L.counters + mt * L.n_tiles + nt;
          const uint32_t prev = atomicAdd(cnt, 1u);
          sh.last = prev == static_cast<uint32_t>(L.splits - 1);
          if (sh.last) *cnt = 0u;  // ready for the next call
        }
        named_bar(1, 128);
        if (sh.last) {
          __threadfence();
          for (int i = 0; i < BN; ++i) {
            const int m = m0 + i;
            if (m >= L.M) break;
            float sum = 0.0f;
            for (int s2 = 0; s2 < L.splits; ++s2)
              sum += __ldcg(L.partial + (static_cast<int64_t>(s2) * L.M + m) * L.N + n);
            L.y[static_cast<int64_t>(m) * L.N + n] = __float2bfloat16_rn(sum);
          }
        }
        named_bar(1, 128);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Prologue: one CTA per token row m.
//   F16: p_m so that max|x_m| 2^-p_m is in [2^14, 2^15); x16 = f16(x 2^-p_m)
//   LoRA: t_j = sum_k x[m,k] A[j,k] (fp32); v = (alpha/r) t_j / (g 2^p_m);
//         t'[m, j] = bf16(v), t'[m, r + j] = bf16(v - bf16(v)); zero to 64 lc.
template <bool F16>
__global__ void __launch_bounds__(256) lora_prep_kernel(PrepArgs a) {
  __shared__ float red[8][16];
  __shared__ uint32_t amax_s[8];
  const int m = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(m) * a.K);
  const int nvec = static_cast<int>(a.K / 8);
  int pexp = 0;
  if constexpr (F16) {
    uint32_t mx = 0;
    for (int v = threadIdx.x; v < nvec; v += 256) mx = max(mx, absmax_bits8(__ldg(xr + v)));
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) amax_s[warp] = mx;
    __syncthreads();
    mx = amax_s[0];
    for (int i = 1; i < 8; ++i) mx = max(mx, amax_s[i]);
    if (mx >= 0x7F80u && threadIdx.x == 0) flag(a.status, QRR_DEV_NONFINITE);
    if (mx != 0u) {
      const float amax = bf16bits_to_f32(mx);
      int e;
      frexpf(amax, &e);  // amax = f 2^e, 0.5 <= f < 1
      pexp = e - 15;     // amax 2^-p in [2^14, 2^15)
    }
    if (threadIdx.x == 0) a.pexp[m] = pexp;
    const Pow2Scaler sc(pexp);
    uint4* x16 = reinterpret_cast<uint4*>(a.x16 + static_cast<int64_t>(m) * a.K);
    for (int v = threadIdx.x; v < nvec; v += 256) {
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
  }
  if (a.r == 0) return;
  const float st = *a.tensor_scale;
  const float g = st > 0.0f ? st : 1.0f;
  // (alpha/r) / (g 2^p): divide by g first, then scale by the power of two
  const Pow2Scaler unp(pexp);
  for (int j0 = 0; j0 < a.r; j0 += 16) {
    float part[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) part[i] = 0.0f;
    for (int v = threadIdx.x; v < nvec; v += 256) {
      const uint4 xv = __ldg(xr + v);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (j0 + i >= a.r) break;
        const uint4 av = __ldg(reinterpret_cast<const uint4*>(a.A + static_cast<int64_t>(j0 + i) * a.K) + v);
        const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
        float s = part[i];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          s = fmaf(bf16_lo(xw[q]), bf16_lo(aw[q]), s);
          s = fmaf(bf16_hi(xw[q]), bf16_hi(aw[q]), s);
        }
        part[i] = s;
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) part[i] += __shfl_xor_sync(0xFFFFFFFFu, part[i], o);
    }
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < 16; ++i) red[warp][i] = part[i];
    }
    __syncthreads();
    if (threadIdx.x < 16 && j0 + static_cast<int>(threadIdx.x) < a.r) {
      float t = 0.0f;
      for (int w2 = 0; w2 < 8; ++w2) t += red[w2][threadIdx.x];
      const float v = unp(__fdiv_rn(a.lora_scale * t, g));
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      __nv_bfloat16* trow = a.t + static_cast<int64_t>(m) * a.t_cols;
      trow[j0 + threadIdx.x] = hi;
      trow[a.r + j0 + threadIdx.x] = lo;
    }
    __syncthreads();
  }
  __nv_bfloat16* trow = a.t + static_cast<int64_t>(m) * a.t_cols;
  for (int j = 2 * a.r + threadIdx.x; j < a.t_cols; j += 256) trow[j] = __float2bfloat16_rn(0.0f);
}

// ---------------------------------------------------------------------------

namespace {

template <int BN, bool F16>
cudaError_t launch_bn(const W4Params& p, int grid, cudaStream_t stream) {
  using C = Cfg<BN>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(w4a16_tc_kernel<BN, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  w4a16_tc_kernel<BN, F16><<<grid, kThreads, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int w4_bn_for(int64_t M) {
  if (M <= 16) return 16;
  if (M <= 32) return 32;
  if (M <= 64) return 64;
  if (M <= 128) return 128;
  return 256;
}

cudaError_t launch_lora_prep(const PrepArgs& a, bool f16, cudaStream_t stream) {
  if (a.M == 0) return cudaSuccess;
  if (f16)
    lora_prep_kernel<true><<<static_cast<unsigned>(a.M), 256, 0, stream>>>(a);
  else
    lora_prep_kernel<false><<<static_cast<unsigned>(a.M), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_w4a16_tc(W4Params& p, int bn, bool f16, cudaStream_t stream) {
  int units = 0;
  for (int j = 0; j < p.count; ++j) {
    p.layer[j].first_unit = units;
    units += p.layer[j].n_tiles * p.layer[j].m_tiles * p.layer[j].splits;
  }
  p.total_units = units;
  if (units == 0) return cudaSuccess;
  int dev = 0, sms = kSMs;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = units < sms ? units : sms;
  switch (bn) {
    case 16: return f16 ? launch_bn<16, true>(p, grid, stream) : launch_bn<16, false>(p, grid, stream);
    case 32: return f16 ? launch_bn<32, true>(p, grid, stream) : launch_bn<32, false>(p, grid, stream);
    case 64: return f16 ? launch_bn<64, true>(p, grid, stream) : launch_bn<64, false>(p, grid, stream);
    case 128: return launch_bn<128, false>(p, grid, stream);
    default: return launch_bn<256, false>(p, grid, stream);
  }
}

}  // namespace qrr

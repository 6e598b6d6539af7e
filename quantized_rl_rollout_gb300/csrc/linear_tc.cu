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
//   warp 0      TMA: per BK-wide K stage, x [BN x BK] (128 B swizzle, in
//               64-wide sub-tiles), the packed codes [128 x BK/2 B] and, for
//               BK = 256, the block scales [128 x 16 B] into an S-stage ring
//   warp 1      MMA: BK/16 x tcgen05.mma (M128 x BN x K16) per stage, A from TMEM
//   warps 2..5  epilogue: D out of TMEM (double-buffered when it fits), scale,
//               store y or a split-K partial
//   warps 6..   G dequant warpgroups taking the stages in turn: thread = weight
//               row (its TMEM lane); codes and scales from shared memory, BK
//               values per stage stored to a TMEM ring of A stages
//
// LoRA is folded into the same accumulator as extra K columns: the prologue
// writes t' = (alpha/r) t / g (t = x . A^T, g = s_t or 1) as interleaved bf16
// (high, low) pairs, the f16 path scales each token row of that tile by its
// pre-scale 2^-p in shared memory, and the matching A columns hold
// (B_j, B_j).  So y = g 2^p D with no separate pass.
//
// Operand type.  Prefill (many tokens) feeds bf16 x directly and dequantizes
// to bf16.  Decode (<= 64 tokens, HBM-bound) feeds f16: the prologue rescales
// each token row by a power of two 2^-p (max |x| into [2^14, 2^15)) and
// rounds it to f16, which is exact for every element within 2^-29 of the
// row's largest magnitude; the weight then dequantizes with one hardware
// E2M1->f16x2 conversion and one packed multiply per two values.  The LoRA
// stages stay bf16 (their own instruction descriptor).
//
// Split-K (decode): units of (layer, 128-row tile, token tile, K range); each
// split writes an fp32 partial, and the last split to finish (a counter per
// tile) sums the partials in split order and writes y, so the result does not
// depend on timing.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

// Pipeline tracing for development builds: compiled with -DQRR_TRACE_BUILD,
// CTA 0 records SM clock stamps of its pipeline hand-offs into qrr_trace
// (role, event, index); qrr_trace_read copies them out.  Ordinary builds
// compile every stamp away.
#ifdef QRR_TRACE_BUILD
__device__ unsigned long long qrr_trace_buf[8][4][256];
#define QRR_STAMP(role, ev, idx) \
  do {                                                                  \
    if (blockIdx.x == 0 && (idx) < 256) qrr_trace_buf[role][ev][idx] = clock64(); \
  } while (0)
#else
#define QRR_STAMP(role, ev, idx) \
  do {                           \
  } while (0)
#endif

namespace {

template <int BN, int BK, int G>
struct Cfg {
  static constexpr int KSUB = BK / 64;     // 64-wide sub-chunks per stage
  static constexpr int X_SUB = BN * 128;   // one [BN x 64] 128-byte-swizzled sub-tile
  static constexpr int X_BYTES = KSUB * X_SUB;
  static constexpr int C_ROW = BK / 2;     // packed code bytes per weight row per stage
  static constexpr int C_BYTES = 128 * C_ROW;
  static constexpr bool SC_TMA = BK >= 256;  // block scales staged by TMA (16 B per row)
  static constexpr int S_BYTES = SC_TMA ? 128 * (BK / 16) : 0;
  static constexpr int STAGE = X_BYTES + C_BYTES + S_BYTES;
  static constexpr int STAGES_RAW = (200 * 1024) / STAGE;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int DBUF = BN <= 128 ? 2 : 1;  // accumulator buffers in TMEM
  static constexpr int D_COLS = BN < 32 ? 32 : BN;
  static constexpr int A_COL = DBUF * D_COLS;
  // The A operand moves through TMEM in chunks of up to 128 K (64 columns), so
  // a dequant group can fill its next chunk while the MMAs still read its last.
  static constexpr int ACH = BK < 128 ? BK : 128;  // K per A chunk
  static constexpr int ACOLS = ACH / 2;
  static constexpr int CPS = BK / ACH;             // A chunks per stage
  static constexpr int AST_RAW = (512 - A_COL) / ACOLS;
  static constexpr int AST = (AST_RAW > 8 ? 8 : AST_RAW) / G * G;
  static constexpr int THREADS = 32 * (2 + 4 + 4 * G);
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * STAGE + 1024;
  static_assert(STAGES >= 2, "shared memory ring too small");
  static_assert(AST >= 2 * G, "TMEM ring too small");
  static_assert(A_COL + AST * ACOLS <= 512, "TMEM overflow");
};

struct SharedCtl {
  uint64_t full[8], empty[8];
  uint64_t a_full[8], a_empty[8];  // per A chunk slot
  uint64_t d_full[2], d_empty[2];
  uint64_t done;
  uint32_t tmem;
  int abort;
  int last;
};

__device__ __forceinline__ uint32_t f16x2_from_e2m1x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}

// Two E4M3 bytes (low 16 bits) -> f16x2, exactly (every E4M3 value is an f16).
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t two) {
  uint32_t r;
  asm("{\n\t.reg .b16 b;\n\tcvt.u16.u32 b, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, b;\n\t}" : "=r"(r) : "r"(two));
  return r;
}

// Four E4M3 bytes -> two f16x2 (bytes 0,1 and bytes 2,3), one unpack.
__device__ __forceinline__ void f16x2x2_from_e4m3x4(uint32_t four, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\tcvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
}

// Eight E2M1 codes (one word, code k in nibble k) -> four f16x2 (pairs 0-1,
// 2-3, 4-5, 6-7), one byte unpack feeding four hardware conversions.
__device__ __forceinline__ void f16x2x4_from_e2m1x8(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
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

// 64 codes (8 words) + their 4 block scales (one word) -> 32 words of A.
template <bool F16>
__device__ __forceinline__ void dequant64(const uint32_t* w, uint32_t scales4, uint32_t* out) {
  if constexpr (F16) {
    uint32_t s01, s23;
    f16x2x2_from_e4m3x4(scales4, s01, s23);
    const uint32_t sg[4] = {__byte_perm(s01, 0, 0x1010), __byte_perm(s01, 0, 0x3232), __byte_perm(s23, 0, 0x1010),
                            __byte_perm(s23, 0, 0x3232)};
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t h[4];
        f16x2x4_from_e2m1x8(w[2 * g + q], h);
#pragma unroll
        for (int b = 0; b < 4; ++b) out[8 * g + 4 * q + b] = hmul2(h[b], sg[g]);
      }
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float sv = e4m3_to_f32((scales4 >> (8 * g)) & 0xFFu);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t h[4];
        f16x2x4_from_e2m1x8(w[2 * g + q], h);
#pragma unroll
        for (int b = 0; b < 4; ++b)
          out[8 * g + 4 * q + b] = pack_bf16x2(f16_lo_to_f32(h[b]) * sv, f16_hi_to_f32(h[b]) * sv);
      }
    }
  }
}

// ring position: index in [0, R) and the number of completed wraps
struct Ring {
  int idx = 0;
  uint32_t use = 0;
  template <int R>
  __device__ __forceinline__ void next() {
    if (++idx == R) {
      idx = 0;
      ++use;
    }
  }
};

}  // namespace

template <int BN, int BK, bool F16, int G>
__global__ void __launch_bounds__(Cfg<BN, BK, G>::THREADS, 1) w4a16_tc_kernel(const __grid_constant__ W4Params p) {
  using C = Cfg<BN, BK, G>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SharedCtl& sh = *reinterpret_cast<SharedCtl*>(tiles + C::STAGES * C::STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &sh.abort;
  constexpr int KSUB = C::KSUB;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1 + 4 * C::CPS);  // MMA commit + 4 dequant warps per A chunk
    }
    for (int s = 0; s < C::AST; ++s) {
      mbar_init(&sh.a_full[s], 4);
      mbar_init(&sh.a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.d_full[b], 1);
      mbar_init(&sh.d_empty[b], 4);
    }
    mbar_init(&sh.done, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  // unit -> (layer, n tile, m tile, split, stage range, LoRA stages)
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
    const int kc = L.K / BK;
    nk = min(c0 + L.kcps, kc) - c0;
    nl = (L.r > 0 && sp == L.splits - 1) ? (L.lora_chunks + KSUB - 1) / KSUB : 0;
  };

  if (warp == 0) {
    // ------------------------------ TMA ------------------------------
    if (elect_one()) {
      Ring st;
      uint32_t issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
        int j, nt, mt, sp, c0, nk, nl;
        locate(u, j, nt, mt, sp, c0, nk, nl);
        const W4Layer& L = p.layer[j];
        for (int c = 0; c < nk + nl; ++c, st.next<C::STAGES>(), ++issued) {
          if (st.use > 0 && !mbar_wait(&sh.empty[st.idx], (st.use - 1) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          QRR_STAMP(0, 0, issued);
          uint8_t* xs = tiles + st.idx * C::STAGE;
          uint64_t* fb = &sh.full[st.idx];
          if (c < nk) {
            const int kb = (c0 + c) * BK;
            mbar_arrive_expect_tx(fb, C::STAGE);
#pragma unroll
            for (int q = 0; q < KSUB; ++q) tma_load_2d(&L.tx, fb, xs + q * C::X_SUB, kb + 64 * q, mt * BN);
            tma_load_2d(&L.tcodes, fb, xs + C::X_BYTES, kb / 2, nt * 128);
            if constexpr (C::SC_TMA) tma_load_2d(&L.tscales, fb, xs + C::X_BYTES + C::C_BYTES, kb / 16, nt * 128);
          } else {
            // LoRA stage: t' sub-tiles past the tensor's width read as zeros
            const int lsub = (c - nk) * KSUB;
            mbar_arrive_expect_tx(fb, C::X_BYTES);
#pragma unroll
            for (int q = 0; q < KSUB; ++q) tma_load_2d(&L.tt, fb, xs + q * C::X_SUB, (lsub + q) * 64, mt * BN);
          }
        }
      }
      // drain: the last load of every stage has landed before the CTA exits
      volatile int no_abort = 0;
      for (uint32_t k = 0; k < static_cast<uint32_t>(C::STAGES) && k < issued; ++k) {
        const uint32_t i = issued - 1 - k;
        mbar_wait(&sh.full[i % C::STAGES], (i / C::STAGES) & 1, &no_abort, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA ------------------------------
    // A stage sa is ready only after its dequant group saw the stage's TMA
    // data land (it waits on `full` first), so this thread waits on a_full alone.
    if (elect_one()) {
      constexpr uint32_t id_main = make_idesc(F16 ? kFmtF16 : kFmtBF16, F16 ? kFmtF16 : kFmtBF16, 128, BN);
      constexpr uint32_t id_lora = make_idesc(kFmtBF16, kFmtBF16, 128, BN);
      Ring st, at;
      uint32_t units = 0, chunks = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x, ++units) {
        int j, nt, mt, sp, c0, nk, nl;
        locate(u, j, nt, mt, sp, c0, nk, nl);
        const int db = units % C::DBUF;
        const uint32_t duse = units / C::DBUF;
        QRR_STAMP(1, 2, units);
        if (duse > 0 && !mbar_wait(&sh.d_empty[db], (duse - 1) & 1, abort, p.status)) break;
        QRR_STAMP(1, 3, units);
        const uint32_t dcol = tmem + db * C::D_COLS;
        for (int c = 0; c < nk + nl && ok; ++c, st.next<C::STAGES>()) {
          const uint32_t xb = smem_u32(tiles + st.idx * C::STAGE);
          const uint32_t idesc = c < nk ? id_main : id_lora;
#pragma unroll
          for (int hc = 0; hc < C::CPS; ++hc, at.next<C::AST>()) {
            if (!mbar_wait(&sh.a_full[at.idx], at.use & 1, abort, p.status)) {
              ok = false;
              break;
            }
            QRR_STAMP(1, 0, chunks);
            tc_fence_after();
            const uint32_t a0 = tmem + C::A_COL + C::ACOLS * at.idx;
#pragma unroll
            for (int k = 0; k < C::ACH / 16; ++k) {
              const int kk = hc * (C::ACH / 16) + k;  // K16 step within the stage
              mma_bf16_ts(dcol, a0 + 8 * k, sw128_desc(xb + (kk >> 2) * C::X_SUB + 32 * (kk & 3)), idesc,
                          (c > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&sh.a_empty[at.idx]);
            QRR_STAMP(1, 1, chunks);
            ++chunks;
          }
          if (ok) mma_commit(&sh.empty[st.idx]);
        }
        if (!ok) break;
        mma_commit(&sh.d_full[db]);
      }
      mma_commit(&sh.done);
      volatile int no_abort = 0;
      mbar_wait(&sh.done, 0, &no_abort, p.status);
    }
  } else if (warp < 6) {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    uint32_t units = 0;
    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x, ++units) {
      int j, nt, mt, sp, c0, nk, nl;
      locate(u, j, nt, mt, sp, c0, nk, nl);
      const W4Layer& L = p.layer[j];
      const int n = nt * 128 + 32 * q + lane;
      const int db = units % C::DBUF;
      if (warp == 2 && lane == 0) QRR_STAMP(3, 0, units);
      if (!mbar_wait(&sh.d_full[db], (units / C::DBUF) & 1, abort, p.status)) break;
      if (warp == 2 && lane == 0) QRR_STAMP(3, 1, units);
      tc_fence_after();
      const float st = *L.tensor_scale;
      const float g = st > 0.0f ? st : 1.0f;
      const int m0 = mt * BN;
      float* part = L.splits > 1 ? L.partial + static_cast<int64_t>(sp) * L.M * L.N : nullptr;
      constexpr int CW = BN == 16 ? 16 : 32;
#pragma unroll 1
      for (int cc = 0; cc < BN / CW; ++cc) {
        uint32_t r[CW];
        if constexpr (CW == 16)
          tmem_ld16(tmem + lane_addr + db * C::D_COLS, r);
        else
          tmem_ld32(tmem + lane_addr + db * C::D_COLS + 32 * cc, r);
        // the per-token factors of this slab first: y / partial stores may
        // alias the exponent array as far as the compiler knows, so loads
        // interleaved with the stores would run one after another
        float sc2[CW];
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          const int m = m0 + CW * cc + i;
          sc2[i] = (L.pexp && m < L.M) ? __fmul_rn(g, pow2_from_exp(__ldg(L.pexp + m))) : g;
        }
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          const int m = m0 + CW * cc + i;
          if (m < L.M) {
            const float v = __uint_as_float(r[i]) * sc2[i];
            if (part)
              part[static_cast<int64_t>(m) * L.N + n] = v;
            else
              L.y[static_cast<int64_t>(m) * L.N + n] = __float2bfloat16_rn(v);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.d_empty[db]);
      if (warp == 2 && lane == 0) QRR_STAMP(3, 2, units);
      if (part) {
        // all 128 epilogue threads have written their partials; one thread
        // makes them visible GPU-wide (the fence is cumulative over the
        // barrier) and takes a ticket; the last split of the tile sums all
        // partials in split order
        named_bar(1, 128);
        if (warp == 2 && lane == 0) {
          __threadfence();
          uint32_t* cnt = L.counters + mt * L.n_tiles + nt;
          const uint32_t prev = atomicAdd(cnt, 1u);
          sh.last = prev == static_cast<uint32_t>(L.splits - 1);
          if (sh.last) {
            *cnt = 0u;  // ready for the next call
            __threadfence();
          }
        }
        named_bar(1, 128);
        if (sh.last) {
          constexpr int TB = 8, SB = 4;  // tokens per batch; loads of SB splits in flight
          for (int i0 = 0; i0 < BN && m0 + i0 < L.M; i0 += TB) {
            float sum[TB];
#pragma unroll
            for (int i = 0; i < TB; ++i) sum[i] = 0.0f;
            for (int s0 = 0; s0 < L.splits; s0 += SB) {
              float v[SB][TB];
#pragma unroll
              for (int s1 = 0; s1 < SB; ++s1)
#pragma unroll
                for (int i = 0; i < TB; ++i)
                  v[s1][i] = (s0 + s1 < L.splits && m0 + i0 + i < L.M)
                                 ? __ldcg(L.partial + (static_cast<int64_t>(s0 + s1) * L.M + m0 + i0 + i) * L.N + n)
                                 : 0.0f;
#pragma unroll
              for (int s1 = 0; s1 < SB; ++s1)
#pragma unroll
                for (int i = 0; i < TB; ++i) sum[i] += v[s1][i];
            }
#pragma unroll
            for (int i = 0; i < TB; ++i)
              if (m0 + i0 + i < L.M) L.y[static_cast<int64_t>(m0 + i0 + i) * L.N + n] = __float2bfloat16_rn(sum[i]);
          }
        }
        named_bar(1, 128);
      }
      if (warp == 2 && lane == 0) QRR_STAMP(3, 3, units);
    }
  } else {
    // ------------------------------ dequant ------------------------------
    const int grp = (warp - 6) >> 2;
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    // TMA swizzle of the code tile: 16-byte piece p of row r sits at
    // p ^ (r & 7) for 128-byte rows and p ^ ((r >> 2) & 1) for 32-byte rows,
    // which keeps every 8-thread phase of a 16-byte shared load on distinct banks
    const int rot = BK == 256 ? (row & 7) : ((row >> 2) & 1);
    Ring st, at;
    int turn = 0;  // A-chunk counter modulo G
    uint32_t chunk = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
      int j, nt, mt, sp, c0, nk, nl;
      locate(u, j, nt, mt, sp, c0, nk, nl);
      const W4Layer& L = p.layer[j];
      const int n = nt * 128 + row;
      const uint8_t* srow = L.scales + static_cast<int64_t>(n) * (L.K / 16);
      for (int c = 0; c < nk + nl && ok; ++c, st.next<C::STAGES>()) {
#pragma unroll 1
        for (int hc = 0; hc < C::CPS; ++hc, at.next<C::AST>(), turn = turn + 1 == G ? 0 : turn + 1, ++chunk) {
          if (turn != grp) continue;
          if (q == 2 && lane == 0) QRR_STAMP(4, 0, chunk);
          uint32_t scw[C::ACH / 64];
          if constexpr (!C::SC_TMA) {
            if (c < nk) scw[0] = __ldg(reinterpret_cast<const uint32_t*>(srow + (c0 + c) * (BK / 16)));
          }
          if (!mbar_wait(&sh.full[st.idx], st.use & 1, abort, p.status) ||
              (at.use > 0 && !mbar_wait(&sh.a_empty[at.idx], (at.use - 1) & 1, abort, p.status))) {
            ok = false;
            break;
          }
          if (q == 2 && lane == 0) QRR_STAMP(4, 1, chunk);
          tc_fence_after();
          const uint8_t* stage = tiles + st.idx * C::STAGE;
          const uint32_t a_addr = tmem + lane_addr + C::A_COL + C::ACOLS * at.idx;
          if (c < nk) {
            if constexpr (C::SC_TMA) {
              // this chunk's 8 scale bytes of the row's 16 (ACH = 128)
              const uint2 sv =
                  *reinterpret_cast<const uint2*>(stage + C::X_BYTES + C::C_BYTES + row * (BK / 16) + 8 * hc);
              scw[0] = sv.x;
              scw[1] = sv.y;
            }
            const uint4* crow = reinterpret_cast<const uint4*>(stage + C::X_BYTES + row * C::C_ROW);
            // 64 values at a time: convert, then store (the store runs async
            // while the next sub-chunk converts)
#pragma unroll
            for (int h = 0; h < C::ACH / 64; ++h) {
              const int piece0 = 2 * ((C::ACH / 64) * hc + h);
              uint32_t w[8];
#pragma unroll
              for (int pc = 0; pc < 2; ++pc) {
                const uint4 v = crow[(piece0 + pc) ^ rot];
                w[4 * pc] = v.x;
                w[4 * pc + 1] = v.y;
                w[4 * pc + 2] = v.z;
                w[4 * pc + 3] = v.w;
              }
              uint32_t out[32];
              dequant64<F16>(w, scw[h], out);
              tmem_st32(a_addr + 32 * h, out);
            }
          } else {
            if constexpr (F16) {
              // t' holds (alpha/r) t / g; the f16 path's accumulator carries
              // the per-token factor 2^-p_m, so scale this chunk's t' rows by
              // it (exact) before the tensor core reads them
              const int tig = q * 32 + lane;
              constexpr int PIECES = (C::ACH / 64) * BN * 8;
              const int m0 = mt * BN;
              for (int idx = tig; idx < PIECES; idx += 128) {
                const int sub = idx / (BN * 8), rem = idx % (BN * 8), mr = rem >> 3;
                if (m0 + mr >= L.M) continue;
                uint4* pc = reinterpret_cast<uint4*>(const_cast<uint8_t*>(stage) +
                                                     (hc * (C::ACH / 64) + sub) * C::X_SUB + mr * 128 +
                                                     (rem & 7) * 16);
                const Pow2Scaler sc(L.pexp[m0 + mr]);
                uint4 v = *pc;
                uint32_t* wv = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
                for (int e = 0; e < 4; ++e) wv[e] = pack_bf16x2(sc(bf16_lo(wv[e])), sc(bf16_hi(wv[e])));
                *pc = v;
              }
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            // LoRA chunk: A word i holds (B[n, rb+i], B[n, rb+i]) against the
            // (high, low) halves of t'; zero past rank r
            const int rb = (c - nk) * (BK / 2) + hc * (C::ACH / 2);
            const uint16_t* brow = L.B + static_cast<int64_t>(n) * L.r + rb;
#pragma unroll
            for (int h = 0; h < C::ACH / 64; ++h) {
              uint32_t out[32];
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                const int v8 = 4 * h + v4;
                uint4 bv = make_uint4(0, 0, 0, 0);
                if (rb + 8 * v8 < L.r) bv = __ldg(reinterpret_cast<const uint4*>(brow) + v8);
                const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  out[8 * v4 + 2 * e] = (bw[e] & 0xFFFFu) * 0x10001u;
                  out[8 * v4 + 2 * e + 1] = (bw[e] >> 16) * 0x10001u;
                }
              }
              tmem_st32(a_addr + 32 * h, out);
            }
          }
          tmem_st_wait();
          if (q == 2 && lane == 0) QRR_STAMP(4, 2, chunk);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&sh.a_full[at.idx]);
            mbar_arrive(&sh.empty[st.idx]);
          }
        }
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
// Prologue.  Per layer, CTAs of two kinds:
//   x rows (f16 path): p_m so that max|x_m| 2^-p_m is in [2^14, 2^15) and
//     x16 = f16(x 2^-p_m), one CTA per token row;
//   LoRA slices: one CTA per (group of 8 ranks, 512-wide K slice) computes the
//     fp32 partial dot products of every token with its ranks; the last slice
//     of a rank group to finish (a ticket) sums the partials in slice order,
//     t_j = sum_k x[m,k] A[j,k], and writes t'[m, 2j] = bf16(v),
//     t'[m, 2j + 1] = bf16(v - bf16(v)) for v = (alpha/r) t_j / g (g = s_t,
//     or 1 when s_t = 0).  The per-token 2^-p_m of the f16 path is applied to
//     the t' tile inside the GEMM, so the two kinds do not depend on each other.
template <bool F16>
__global__ void __launch_bounds__(256) lora_prep_kernel(const __grid_constant__ PrepBatch batch) {
  __shared__ uint32_t amax_s[8];
  __shared__ int last_s;
  int j = 0;
  while (j + 1 < batch.count && batch.a[j + 1].first_cta <= static_cast<int>(blockIdx.x)) ++j;
  const PrepArgs& a = batch.a[j];
  int local = static_cast<int>(blockIdx.x) - a.first_cta;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = static_cast<int>(a.K / 8);
  const int nx = F16 ? static_cast<int>(a.M) : 0;
  if (local < nx) {
    // ---- x row -> f16 with its power-of-two pre-scale ----
    const int m = local;
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(m) * a.K);
    uint32_t mx = 0;
    for (int v = threadIdx.x; v < nvec; v += 256) mx = max(mx, absmax_bits8(__ldg(xr + v)));
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) amax_s[warp] = mx;
    __syncthreads();
    mx = amax_s[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) mx = max(mx, amax_s[i]);
    int pexp = 0;
    if (mx != 0u) {
      int e;
      frexpf(bf16bits_to_f32(mx), &e);  // amax = f 2^e, 0.5 <= f < 1
      pexp = e - 15;                    // amax 2^-p in [2^14, 2^15)
    }
    if (mx >= 0x7F80u && threadIdx.x == 0) flag(a.status, QRR_DEV_NONFINITE);
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
    return;
  }
  local -= nx;
  // ---- LoRA slice: ranks [8 rg, 8 rg + 8), vectors [64 ks, 64 ks + 64) ----
  const int rg = local / a.ks, kslice = local % a.ks;
  const int j0 = rg * 8, nj = min(8, a.r - j0);
  const int v0 = kslice * 64, v1 = min(nvec, v0 + 64);
  // each lane holds two 8-element vectors of the 8 A rows
  uint4 av[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int v = v0 + lane + 32 * h;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      av[h][i] = (v < v1 && i < nj)
                     ? __ldg(reinterpret_cast<const uint4*>(a.A + static_cast<int64_t>(j0 + i) * a.K) + v)
                     : make_uint4(0, 0, 0, 0);
  }
  for (int m = warp; m < a.M; m += 8) {
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(m) * a.K);
    float d[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = v0 + lane + 32 * h;
      const uint4 xv = v < v1 ? __ldg(xr + v) : make_uint4(0, 0, 0, 0);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t aw[4] = {av[h][i].x, av[h][i].y, av[h][i].z, av[h][i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          d[i] = fmaf(bf16_lo(xw[q]), bf16_lo(aw[q]), d[i]);
          d[i] = fmaf(bf16_hi(xw[q]), bf16_hi(aw[q]), d[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) d[i] += __shfl_xor_sync(0xFFFFFFFFu, d[i], o);
    }
    if (lane < nj) {
      float mine = d[0];
#pragma unroll
      for (int i = 1; i < 8; ++i)
        if (lane == i) mine = d[i];
      a.tpart[(static_cast<int64_t>(kslice) * a.M + m) * a.r + j0 + lane] = mine;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(a.tickets + rg, 1u);
    last_s = prev == static_cast<uint32_t>(a.ks - 1);
    if (last_s) __threadfence();
  }
  __syncthreads();
  if (!last_s) return;
  const float st = *a.tensor_scale;
  const float g = st > 0.0f ? st : 1.0f;
  for (int idx = threadIdx.x; idx < a.M * nj; idx += 256) {
    const int m = idx / nj, i = idx % nj;
    float t = 0.0f;
    for (int s2 = 0; s2 < a.ks; ++s2) t += __ldcg(a.tpart + (static_cast<int64_t>(s2) * a.M + m) * a.r + j0 + i);
    const float v = __fdiv_rn(a.lora_scale * t, g);
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    __nv_bfloat16* trow = a.t + static_cast<int64_t>(m) * a.t_cols;
    trow[2 * (j0 + i)] = hi;
    trow[2 * (j0 + i) + 1] = lo;
  }
  if (rg == 0) {
    const int pad = a.t_cols - 2 * a.r;
    for (int idx = threadIdx.x; idx < a.M * pad; idx += 256)
      a.t[static_cast<int64_t>(idx / pad) * a.t_cols + 2 * a.r + idx % pad] = __float2bfloat16_rn(0.0f);
  }
}

// ---------------------------------------------------------------------------

namespace {

template <int BN, int BK, bool F16, int G>
cudaError_t launch_bn(const W4Params& p, int grid, cudaStream_t stream) {
  using C = Cfg<BN, BK, G>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(w4a16_tc_kernel<BN, BK, F16, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  w4a16_tc_kernel<BN, BK, F16, G><<<grid, C::THREADS, C::SMEM, stream>>>(p);
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

// Decode tiles (<= 64 tokens) stream the weight in 256-wide K stages (block
// scales staged by TMA); prefill tiles use 64-wide stages.
int w4_bk_for(int64_t M) { return M <= 64 ? 256 : 64; }

cudaError_t launch_lora_prep(PrepBatch& b, bool f16, cudaStream_t stream) {
  if (b.count == 0 || b.a[0].M == 0) return cudaSuccess;
  int ctas = 0;
  for (int j = 0; j < b.count; ++j) {
    PrepArgs& a = b.a[j];
    a.first_cta = ctas;
    ctas += (f16 ? static_cast<int>(a.M) : 0) + (a.r > 0 ? ((a.r + 7) / 8) * a.ks : 0);
  }
  if (ctas == 0) return cudaSuccess;
  if (f16)
    lora_prep_kernel<true><<<ctas, 256, 0, stream>>>(b);
  else
    lora_prep_kernel<false><<<ctas, 256, 0, stream>>>(b);
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
  if (f16) {
    switch (bn) {
      case 16: return launch_bn<16, 256, true, 3>(p, grid, stream);
      case 32: return launch_bn<32, 256, true, 3>(p, grid, stream);
      default: return launch_bn<64, 256, true, 3>(p, grid, stream);
    }
  }
  return bn == 128 ? launch_bn<128, 64, false, 2>(p, grid, stream) : launch_bn<256, 64, false, 2>(p, grid, stream);
}

}  // namespace qrr

#ifdef QRR_TRACE_BUILD
extern "C" int qrr_trace_read(unsigned long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, qrr::qrr_trace_buf, sizeof(qrr::qrr_trace_buf)));
}
extern "C" int qrr_trace_clear(void) {
  static unsigned long long zeros[8 * 4 * 256] = {};
  return static_cast<int>(cudaMemcpyToSymbol(qrr::qrr_trace_buf, zeros, sizeof(zeros)));
}
#endif

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
//   warps 2, 3, 4G+4, 4G+5  epilogue: D out of TMEM (double-buffered when it
//               fits), scale, store y or a split-K partial
//   warps 4..4G+3  G dequant warpgroups taking the A chunks in turn: thread =
//               weight row (its TMEM lane); codes and scales from shared
//               memory, stored to a TMEM ring of A chunks
//
// Prefill tiles of 256 tokens run on CTA pairs (2-CTA clusters): the even
// CTA issues cta_group::2 MMAs (M = 256, 128 weight rows in each CTA's TMEM)
// and each CTA stages only its half of the token tile.
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

#include <string.h>

#include <algorithm>
#include <mutex>
#include <type_traits>
#include <vector>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

// Pipeline tracing for development builds: compiled with -DQRR_TRACE_BUILD,
// CTA 0 records SM clock stamps of its pipeline hand-offs into qrr_trace
// (role, event, index); qrr_trace_read copies them out.  Ordinary builds
// compile every stamp away.
#ifdef QRR_TRACE_BUILD
__device__ unsigned long long qrr_trace_buf[8][4][256];
// global-timer stamps per CTA: start, x stream released, first MMA, end
__device__ unsigned long long qrr_gtrace_buf[256][8];
#define QRR_GSTAMP(ev)                                               \
  do {                                                               \
    unsigned long long t_;                                           \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));           \
    if (blockIdx.x < 256) qrr_gtrace_buf[blockIdx.x][ev] = t_;       \
  } while (0)
#define QRR_STAMP(role, ev, idx) \
  do {                                                                  \
    if (blockIdx.x == 0 && (idx) < 256) qrr_trace_buf[role][ev][idx] = clock64(); \
  } while (0)
#else
#define QRR_STAMP(role, ev, idx) \
  do {                           \
  } while (0)
#define QRR_GSTAMP(ev) \
  do {                 \
  } while (0)
#endif

namespace {

template <int BN, int BK, int G, bool PAIR = false>
struct Cfg {
  static constexpr int KSUB = BK / 64;     // 64-wide sub-chunks per stage
  // token rows of x held by this CTA: a CTA pair splits its BN tokens
  static constexpr int BNL = PAIR ? BN / 2 : BN;
  static constexpr int X_SUB = BNL * 128;  // one [BNL x 64] 128-byte-swizzled sub-tile
  static constexpr int X_BYTES = KSUB * X_SUB;
  static constexpr int C_ROW = BK / 2;     // packed code bytes per weight row per stage
  static constexpr int C_BYTES = 128 * C_ROW;
  static constexpr bool SC_TMA = BK >= 256;  // block scales staged by TMA (16 B per row)
  static constexpr int S_BYTES = SC_TMA ? 128 * (BK / 16) : 0;
  static constexpr int STAGE = X_BYTES + C_BYTES + S_BYTES;
  // as many stages as fit in shared memory (227 KB per CTA, less the
  // alignment slack and the control block): the ring is what covers the L2
  // and HBM latency of the x tiles
  static constexpr int STAGES_RAW = (224 * 1024 - 2048) / STAGE;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int DBUF = BN <= 128 ? 2 : 1;  // accumulator buffers in TMEM
  static constexpr int D_COLS = BN < 32 ? 32 : BN;
  static constexpr int A_COL = DBUF * D_COLS;
  // The A operand moves through TMEM in chunks of up to 128 K (64 columns), so
  // a dequant group can fill its next chunk while the MMAs still read its last.
  static constexpr int ACH = BK < 128 ? BK : 128;  // K per A chunk
  static constexpr int ACOLS = ACH / 2;
  static constexpr int CPS = BK / ACH;             // A chunks per stage
  // A slot of chunk c is rewritten for chunk c + AST once the MMAs of chunk c
  // are done.  While the TMEM ring is no deeper than the shared-memory ring,
  // the release of chunk c's stage says so (its barrier phase is still
  // unambiguous, at most STAGES stages back); a deeper TMEM ring gets one
  // release barrier per slot, at the price of a second commit per chunk.
  static constexpr int AST_FIT = (512 - A_COL) / ACOLS;
  // 256-wide decode stages release each A slot per chunk: waiting for the
  // stage's second chunk would hold the slot back by a chunk's dequant time
  static constexpr bool SLOT_BARS = AST_FIT > CPS * STAGES || BK >= 256;
  static constexpr int AST = (AST_FIT > 8 ? 8 : AST_FIT) / G * G;
  static constexpr int THREADS = 32 * (2 + 4 + 4 * G);
  // registers per thread for one resident CTA: each of the SM's four
  // sub-partitions holds 16K registers and ceil(warps / 4) of the warps, in
  // the allocator's steps of 8
  static constexpr int WARPS_PER_SMSP = (THREADS / 32 + 3) / 4;
  static constexpr int REGS_RAW = 16384 / (32 * WARPS_PER_SMSP) / 8 * 8;
  static constexpr int MAXNREG = REGS_RAW > 255 ? 255 : REGS_RAW;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * STAGE + 1024;
  static_assert(STAGES >= 2, "shared memory ring too small");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA exceeded");
  static_assert(AST >= 2 * G, "TMEM ring too small");
  static_assert(A_COL + AST * ACOLS <= 512, "TMEM overflow");
  static_assert(!PAIR || (BN == 256 && !SLOT_BARS), "CTA pairs: 256-token tiles, stage-released A slots");
};

struct SharedCtl {
  uint64_t full[8], full_x[8], empty[8];  // full: codes + scales landed; full_x: x (or t') landed
  uint64_t a_full[8], a_empty[8];  // per A chunk slot (a_empty: only with SLOT_BARS)
  uint64_t d_full[2], d_empty[2];
  uint64_t done;
  uint32_t next_chunk[4];  // next A chunk to take, per TMEM lane quarter
  uint32_t tmem;
  int abort;
  int last;
};

// Four E4M3 bytes -> two f16x2 (bytes 0,1 and bytes 2,3), one unpack.
__device__ __forceinline__ void f16x2x2_from_e4m3x4(uint32_t four, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\tcvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(four));
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
    // The hardware conversion's f16 E2M1 values re-read as bf16 v 2^-112,
    // then one bf16x2 multiply by s_b 2^112 returns v s_b exactly: both
    // factors and the product are normal bf16 numbers, the product has at
    // most six significant bits.
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const float sv = e4m3_to_f32((scales4 >> (8 * g)) & 0xFFu) * 0x1p112f;
      const uint32_t s2 = pack_bf16x2(sv, sv);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t h[4];
        f16x2x4_from_e2m1x8(w[2 * g + q], h);
#pragma unroll
        for (int b = 0; b < 4; ++b)
          out[8 * g + 4 * q + b] = bmul2(e2m1_f16x2_rebias_bf16x2(h[b]), s2);
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

template <int BN, int BK, bool F16, int G, bool PAIR>
__global__ void __maxnreg__((Cfg<BN, BK, G, PAIR>::MAXNREG)) w4a16_tc_kernel(const __grid_constant__ W4Params p) {
  using C = Cfg<BN, BK, G, PAIR>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SharedCtl& sh = *reinterpret_cast<SharedCtl*>(tiles + C::STAGES * C::STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &sh.abort;
  constexpr int KSUB = C::KSUB;
  if (threadIdx.x == 0) QRR_GSTAMP(0);
  // CTA pairs (2-CTA clusters): both CTAs walk the same units, the even one
  // (rank 0) issues the pair's MMAs and holds the barriers the pair meets on
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const int ustart = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ustep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // this CTA's units: its slice of the unit table (decode), round-robin
  // otherwise; unit_at(i) is the i-th of them
  const bool sk = !PAIR && p.use_table;
  const int sk0 = sk ? p.unit_off[blockIdx.x] : 0;
  const int n_my = sk ? p.unit_off[blockIdx.x + 1] - sk0
                      : (ustart < p.total_units ? (p.total_units - 1 - ustart) / ustep + 1 : 0);
  auto unit_at = [&](int i) { return sk ? sk0 + i : ustart + i * ustep; };
  // Every wait acquires at CTA scope, which keeps the SM's L1 contents valid
  // across it: what the peer CTA of a pair hands over through a barrier is
  // tensor-memory state, TMA bytes or tensor-core completion, none of it
  // generic memory.
  auto wait = [&](uint64_t* bar, uint32_t parity) { return mbar_wait(bar, parity, abort, p.status); };
  // arrive on the even CTA's copy of a barrier (this CTA's own when unpaired)
  auto arrive_leader = [&](uint64_t* bar) {
    if (PAIR && rank != 0)
      mbar_arrive_cluster(cluster_addr(bar, 0));
    else
      mbar_arrive(bar);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.full_x[s], 1);
      mbar_init(&sh.empty[s], 1 + 4 * C::CPS);  // MMA commit + 4 dequant warps per A chunk
    }
    for (int s = 0; s < C::AST; ++s) {
      mbar_init(&sh.a_full[s], PAIR ? 8 : 4);  // the dequant warps of both CTAs of a pair
      mbar_init(&sh.a_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.d_full[b], 1);
      mbar_init(&sh.d_empty[b], PAIR ? 8 : 4);
    }
    mbar_init(&sh.done, 1);
    for (int i = 0; i < 4; ++i) sh.next_chunk[i] = 0;
    sh.abort = 0;
    fence_barrier_init();
  }
  // warp roles: the TMA and MMA issuers take the lowest warp numbers, which
  // the schedulers favour on a busy sub-partition (an MMA issuer sharing its
  // sub-partition with three busy dequant warps otherwise slows to about 70
  // cycles per MMA); then two epilogue warps (lane quarters 2, 3), the
  // dequant warpgroups, and the other two epilogue warps (quarters 0, 1).
  // Every warp w that touches TMEM serves lane quarter w % 4.
  constexpr int kTma = 0, kMma = 1, kEpi = 2, kDqEnd = 4 + 4 * G;
  const bool epi_warp = warp == 2 || warp == 3 || warp >= kDqEnd;
  if (warp == kMma) {
    if constexpr (PAIR)
      tmem_alloc_pair(&sh.tmem, C::TMEM_COLS);
    else
      tmem_alloc(&sh.tmem, C::TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the peer's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  // unit -> (layer, n tile, m tile, piece, stage range, LoRA stages); the
  // tile's piece count is unit_pieces(u)
  auto locate = [&](int u, int& j, int& nt, int& mt, int& sp, int& c0, int& nk, int& nl) {
    if (sk) {
      const uint32_t w0 = p.unit[u][0], w1 = p.unit[u][1];
      j = static_cast<int>(w0 & 0xFu);
      mt = static_cast<int>((w0 >> 4) & 0xFu);
      nt = static_cast<int>((w0 >> 8) & 0xFFFFu);
      c0 = static_cast<int>(w1 & 0xFFFu);
      nk = static_cast<int>((w1 >> 12) & 0x7FFu);
      sp = static_cast<int>((w1 >> 23) & 0xFFu);
      nl = static_cast<int>(w1 >> 31);
      return;
    }
    j = 0;
    while (j + 1 < p.count && p.layer[j + 1].first_unit <= u) ++j;
    const W4Layer& L = p.layer[j];
    const int local = u - L.first_unit;
    const int n_units = PAIR ? L.n_tiles / 2 : L.n_tiles;  // a pair takes two adjacent 128-row tiles
    nt = local % n_units;
    const int rest = local / n_units;
    mt = rest % L.m_tiles;
    sp = rest / L.m_tiles;
    c0 = sp * L.kcps;
    const int kc = L.K / BK;
    nk = min(c0 + L.kcps, kc) - c0;
    nl = (L.r > 0 && sp == L.splits - 1) ? (L.lora_chunks + KSUB - 1) / KSUB : 0;
    if constexpr (PAIR) nt = 2 * nt + static_cast<int>(rank);
  };

  auto unit_pieces = [&](int u, int j) { return sk ? static_cast<int>(p.unit[u][0] >> 24) : p.layer[j].splits; };

  if (warp == kTma) {
    // ------------------------------ TMA ------------------------------
    // The weight stream does not depend on the prologue kernel that writes
    // t' (and, on the f16 path, the f16 x): this kernel may start while it
    // runs, as its programmatic dependent.  The first ring of stages gets its
    // codes and scales at once; f16 x waits for the prologue to complete,
    // bf16 x does not, and t' (the LoRA stages) always does.
    if (elect_one()) {
      struct Cursor {
        int i = -1, c = 0, j = 0, nt = 0, mt = 0, sp = 0, c0 = 0, nk = 0, nl = 0;
      };
      auto next = [&](Cursor& k) {  // advance to the next stage of the CTA; false past the last
        if (k.i >= n_my) return false;
        if (k.i >= 0 && ++k.c < k.nk + k.nl) return true;
        k.c = 0;
        for (++k.i; k.i < n_my; ++k.i) {
          locate(unit_at(k.i), k.j, k.nt, k.mt, k.sp, k.c0, k.nk, k.nl);
          if (k.nk + k.nl > 0) return true;
        }
        return false;
      };
      auto issue_w = [&](const Cursor& k, int idx) {
        uint64_t* fb = &sh.full[idx];
        if (k.c < k.nk) {
          const int kb = (k.c0 + k.c) * BK;
          uint8_t* xs = tiles + idx * C::STAGE;
          mbar_arrive_expect_tx(fb, C::C_BYTES + C::S_BYTES);
          tma_load_2d(&p.layer[k.j].tcodes, fb, xs + C::X_BYTES, kb / 2, k.nt * 128);
          if constexpr (C::SC_TMA)
            tma_load_2d(&p.layer[k.j].tscales, fb, xs + C::X_BYTES + C::C_BYTES, kb / 16, k.nt * 128);
        } else if (F16) {
          // LoRA stage: no codes; the adapter's B rows of the tile take
          // their place (r <= 64: at most 16 KB)
          uint8_t* xs = tiles + idx * C::STAGE;
          mbar_arrive_expect_tx(fb, 128u * static_cast<uint32_t>(p.layer[k.j].r) * 2u);
          tma_load_2d(&p.layer[k.j].tb, fb, xs + C::X_BYTES, 0, k.nt * 128);
        } else {
          mbar_arrive(fb);  // LoRA stage: no codes
        }
      };
      // x (or t') rows of this CTA; in a pair each CTA loads its half of the
      // tile's tokens and both halves count on the even CTA's barrier
      auto issue_x = [&](const Cursor& k, int idx) {
        uint64_t* fb = &sh.full_x[idx];
        uint8_t* xs = tiles + idx * C::STAGE;
        const int row0 = k.mt * BN + static_cast<int>(rank) * C::BNL;
        const CUtensorMap* map = k.c < k.nk ? &p.layer[k.j].tx : &p.layer[k.j].tt;
        // column of the first sub-tile: K offset, or the LoRA sub-tile (past
        // the tensor's width reads as zeros)
        const int col0 = k.c < k.nk ? (k.c0 + k.c) * BK : (k.c - k.nk) * KSUB * 64;
        if (!F16 && k.c >= k.nk) griddep_wait();  // t' is the prologue's
        if constexpr (PAIR) {
          if (rank == 0) mbar_arrive_expect_tx(fb, 2 * C::X_BYTES);
          const uint32_t fbc = cluster_addr(fb, 0);
#pragma unroll
          for (int q = 0; q < KSUB; ++q) tma_load_2d_pair(map, fbc, xs + q * C::X_SUB, col0 + 64 * q, row0);
        } else {
          mbar_arrive_expect_tx(fb, C::X_BYTES);
#pragma unroll
          for (int q = 0; q < KSUB; ++q) tma_load_2d(map, fb, xs + q * C::X_SUB, col0 + 64 * q, row0);
        }
      };
      Cursor kw, kx;
      uint32_t nw = 0;  // stages whose weights are issued
      while (nw < static_cast<uint32_t>(C::STAGES) && next(kw)) {
        QRR_STAMP(0, 0, nw);
        issue_w(kw, static_cast<int>(nw));
        ++nw;
      }
      if constexpr (F16) griddep_wait();
      QRR_GSTAMP(1);
      uint32_t nx = 0;
      bool ok = true;
      while (nx < nw) {
        next(kx);
        issue_x(kx, static_cast<int>(nx));
        ++nx;
      }
      while (ok && next(kw)) {
        next(kx);
        const uint32_t idx = nw % C::STAGES, use = nw / C::STAGES;
        if (!wait(&sh.empty[idx], (use - 1) & 1)) {
          ok = false;
          break;
        }
        QRR_STAMP(0, 0, nw);
        issue_w(kw, static_cast<int>(idx));
        issue_x(kx, static_cast<int>(idx));
        ++nw;
      }
      // drain: the last loads of every stage have landed before the CTA exits
      // (a pair's x halves all count on the even CTA, which the odd one
      // waits for at the closing cluster barrier)
      volatile int no_abort = 0;
      for (uint32_t k = 0; k < static_cast<uint32_t>(C::STAGES) && k < nw; ++k) {
        const uint32_t i = nw - 1 - k;
        mbar_wait(&sh.full[i % C::STAGES], (i / C::STAGES) & 1, &no_abort, p.status);
        if (!PAIR || rank == 0) mbar_wait(&sh.full_x[i % C::STAGES], (i / C::STAGES) & 1, &no_abort, p.status);
      }
    }
  } else if (warp == kMma) {
    // ------------------------------ MMA ------------------------------
    // Per stage: the x (or t') tile has landed; per A chunk: its dequant
    // warps have stored it to TMEM.
    // In a CTA pair only the even CTA issues: M = 256 rows (128 in each
    // CTA's TMEM), and every commit reaches the barrier in both CTAs.
    if (elect_one() && (!PAIR || rank == 0)) {
      constexpr uint32_t MM = PAIR ? 256 : 128;
      constexpr uint32_t id_main = make_idesc(F16 ? kFmtF16 : kFmtBF16, F16 ? kFmtF16 : kFmtBF16, MM, BN);
      constexpr uint32_t id_lora = make_idesc(kFmtBF16, kFmtBF16, MM, BN);
      auto commit = [&](uint64_t* bar) {
        if constexpr (PAIR)
          mma_commit_pair(bar, 0x3);
        else
          mma_commit(bar);
      };
      Ring st, at;
      uint32_t units = 0, chunks = 0;
      bool ok = true;
      for (int ui = 0; ui < n_my && ok; ++ui, ++units) {
        int j, nt, mt, sp, c0, nk, nl;
        locate(unit_at(ui), j, nt, mt, sp, c0, nk, nl);
        const int db = units % C::DBUF;
        const uint32_t duse = units / C::DBUF;
        QRR_STAMP(1, 2, units);
        if (duse > 0 && !wait(&sh.d_empty[db], (duse - 1) & 1)) break;
        QRR_STAMP(1, 3, units);
        const uint32_t dcol = tmem + db * C::D_COLS;
        for (int c = 0; c < nk + nl && ok; ++c, st.next<C::STAGES>()) {
          if (!wait(&sh.full_x[st.idx], st.use & 1)) {
            ok = false;
            break;
          }
          // descriptor of the stage's first x sub-tile; the K16 steps only move
          // its start-address field (16-byte units, no carry inside shared memory)
          const uint64_t bdesc = sw128_desc(smem_u32(tiles + st.idx * C::STAGE));
          const uint32_t idesc = c < nk ? id_main : id_lora;
#pragma unroll
          for (int hc = 0; hc < C::CPS; ++hc, at.next<C::AST>()) {
            QRR_STAMP(2, 2, chunks);
            if (!wait(&sh.a_full[at.idx], at.use & 1)) {
              ok = false;
              break;
            }
            QRR_STAMP(1, 0, chunks);
            tc_fence_after();
            const uint32_t a0 = tmem + C::A_COL + C::ACOLS * at.idx;
            constexpr int NK = C::ACH / 16;  // K16 steps per chunk
            static_assert(NK == 4 || NK == 8, "chunk of 64 or 128 K");
            uint64_t bd[NK];
#pragma unroll
            for (int k = 0; k < NK; ++k) {
              const int kk = hc * NK + k;  // K16 step within the stage
              bd[k] = bdesc + static_cast<uint64_t>(((kk >> 2) * C::X_SUB + 32 * (kk & 3)) >> 4);
            }
            const uint32_t acc = (c > 0 || hc > 0) ? 1u : 0u;
            if constexpr (PAIR) {
              static_assert(!PAIR || NK == 4, "CTA pairs use 64-wide K chunks");
              mma4_ts_pair(dcol, a0, bd, idesc, acc);
            } else if constexpr (NK == 8) {
              mma8_ts(dcol, a0, bd, idesc, acc);
            } else {
              mma4_ts(dcol, a0, bd, idesc, acc);
            }
            if constexpr (C::SLOT_BARS) commit(&sh.a_empty[at.idx]);
            QRR_STAMP(1, 1, chunks);
            if (chunks == 0) QRR_GSTAMP(2);
            ++chunks;
          }
          QRR_STAMP(2, 0, chunks / C::CPS);
          if (ok) commit(&sh.empty[st.idx]);
          QRR_STAMP(2, 1, chunks / C::CPS);
        }
        if (!ok) break;
        commit(&sh.d_full[db]);
        QRR_STAMP(2, 3, units);
      }
#ifdef QRR_TRACE_BUILD
      if (blockIdx.x < 256) qrr_gtrace_buf[blockIdx.x][4] = chunks;
#endif
      if constexpr (PAIR)
        mma_commit_pair(&sh.done, 0x1);
      else
        mma_commit(&sh.done);
      volatile int no_abort = 0;
      mbar_wait(&sh.done, 0, &no_abort, p.status);
    }
  } else if (epi_warp) {
    // ------------------------------ epilogue ------------------------------
    // Layer fields are copied to registers once per unit: read through the
    // parameter reference they would be re-read after every store (the
    // compiler cannot rule out aliasing), each a dependent memory round trip.
    const int q = warp & 3;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    if constexpr (F16) griddep_wait();  // the per-token exponents come from the prologue kernel
    uint32_t units = 0;
    for (int ui = 0; ui < n_my; ++ui, ++units) {
      int j, nt, mt, sp, c0, nk, nl;
      locate(unit_at(ui), j, nt, mt, sp, c0, nk, nl);
      const int M = p.layer[j].M, N = p.layer[j].N, n_tiles = p.layer[j].n_tiles;
      const int splits = unit_pieces(unit_at(ui), j);  // pieces of this tile
      const int* const pexp = p.layer[j].pexp;
      __nv_bfloat16* const y = p.layer[j].y;
      float* const partial = p.layer[j].partial;
      uint32_t* const counters = p.layer[j].counters;
      const float st = *p.layer[j].tensor_scale;
      const int n = nt * 128 + 32 * q + lane;
      const int db = units % C::DBUF;
      if (warp == kEpi && lane == 0) QRR_STAMP(3, 0, units);
      if (!wait(&sh.d_full[db], (units / C::DBUF) & 1)) break;
      if (warp == kEpi && lane == 0) QRR_STAMP(3, 1, units);
      tc_fence_after();
      const float g = st > 0.0f ? st : 1.0f;
      const int m0 = mt * BN;
      // split-K is planned for the decode (f16) path only
      float* const part = (F16 && splits > 1) ? partial + static_cast<int64_t>(sp) * M * N : nullptr;
      constexpr int CW = BN == 16 ? 16 : 32;
      // Every test below is warp-uniform and taken once per slab: with one
      // epilogue warp per sub-partition, a branch per element would cost a
      // branch resolution each (about ten times the slab's arithmetic).
#pragma unroll 1
      for (int cc = 0; cc < BN / CW; ++cc) {
        const int mb = m0 + CW * cc;
        const int cnt = M - mb;  // tokens of this slab, when fewer than CW
        if (cnt <= 0) break;
        uint32_t r[CW];
        if constexpr (CW == 16)
          tmem_ld16(tmem + lane_addr + db * C::D_COLS, r);
        else
          tmem_ld32(tmem + lane_addr + db * C::D_COLS + 32 * cc, r);
        // the per-token factors of this slab first, all loads in flight
        float v[CW];
        if (pexp != nullptr) {
          if (cnt >= CW) {
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] = __fmul_rn(g, pow2_from_exp(__ldg(pexp + mb + i)));
          } else {
#pragma unroll
            for (int i = 0; i < CW; ++i) v[i] = __fmul_rn(g, pow2_from_exp(__ldg(pexp + mb + min(i, cnt - 1))));
          }
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]) * v[i];
        } else {
          tmem_ld_wait();
          // two outputs per instruction on the paired fp32 pipe (each half
          // one correctly rounded fp32 multiply)
#pragma unroll
          for (int i = 0; i < CW; i += 2)
            asm("{\n\t.reg .b64 rr, gg;\n\tmov.b64 rr, {%2, %3};\n\tmov.b64 gg, {%4, %4};\n\t"
                "mul.rn.f32x2 rr, rr, gg;\n\tmov.b64 {%0, %1}, rr;\n\t}"
                : "=f"(v[i]), "=f"(v[i + 1])
                : "f"(__uint_as_float(r[i])), "f"(__uint_as_float(r[i + 1])), "f"(g));
        }
        if (part != nullptr) {
          float* const dst = part + static_cast<int64_t>(mb) * N + n;
          if (cnt >= CW) {
#pragma unroll
            for (int i = 0; i < CW; ++i) dst[static_cast<int64_t>(i) * N] = v[i];
          } else {
#pragma unroll
            for (int i = 0; i < CW; ++i)
              if (i < cnt) dst[static_cast<int64_t>(i) * N] = v[i];
          }
        } else {
          __nv_bfloat16* const dst = y + static_cast<int64_t>(mb) * N + n;
          if (cnt >= CW) {
            // Token pairs: each lane rounds its tokens i, i + 1 into one
            // bf16x2 word and swaps it with lane n ^ 1; a byte permute then
            // forms the word of two adjacent outputs of one token (the even
            // lane token i, the odd lane token i + 1): one conversion, one
            // shuffle, one permute and one store per two outputs.
            const int odd = lane & 1;
            const uint32_t sel = odd ? 0x3276u : 0x5410u;
            uint32_t* const dstw = reinterpret_cast<uint32_t*>(dst - odd);
#pragma unroll
            for (int i = 0; i < CW; i += 2) {
              const uint32_t own = pack_bf16x2(v[i], v[i + 1]);
              const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, own, 1);
              dstw[static_cast<int64_t>(i + odd) * (N / 2)] = __byte_perm(own, other, sel);
            }
          } else {
#pragma unroll
            for (int i = 0; i < CW; ++i)
              if (i < cnt) dst[static_cast<int64_t>(i) * N] = __float2bfloat16_rn(v[i]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(&sh.d_empty[db]);
      if (warp == kEpi && lane == 0) QRR_STAMP(3, 2, units);
      if (F16 && part != nullptr) {
        // all 128 epilogue threads have written their partials; one thread
        // makes them visible GPU-wide (the fence is cumulative over the
        // barrier) and takes a ticket; the last split of the tile sums all
        // partials in split order
        named_bar(1, 128);
        if (warp == kEpi && lane == 0) {
          __threadfence();
          uint32_t* cnt = counters + mt * n_tiles + nt;
          const uint32_t prev = atomicAdd(cnt, 1u);
          sh.last = prev == static_cast<uint32_t>(splits - 1);
          if (sh.last) {
            *cnt = 0u;  // ready for the next call
            __threadfence();
          }
        }
        named_bar(1, 128);
        if (sh.last) {
          constexpr int TB = 8, SB = 4;  // tokens per batch; loads of SB splits in flight
          for (int i0 = 0; i0 < BN && m0 + i0 < M; i0 += TB) {
            float sum[TB];
#pragma unroll
            for (int i = 0; i < TB; ++i) sum[i] = 0.0f;
            const bool whole = m0 + i0 + TB <= M;  // a batch of TB tokens without a ragged end
            for (int s0 = 0; s0 < splits; s0 += SB) {
              float v[SB][TB];
              const float* const src = partial + (static_cast<int64_t>(s0) * M + m0 + i0) * N + n;
              const int64_t sstride = static_cast<int64_t>(M) * N;
              if (whole && s0 + SB <= splits) {
#pragma unroll
                for (int s1 = 0; s1 < SB; ++s1)
#pragma unroll
                  for (int i = 0; i < TB; ++i) v[s1][i] = __ldcg(src + s1 * sstride + static_cast<int64_t>(i) * N);
              } else {
#pragma unroll
                for (int s1 = 0; s1 < SB; ++s1)
#pragma unroll
                  for (int i = 0; i < TB; ++i)
                    v[s1][i] = (s0 + s1 < splits && m0 + i0 + i < M)
                                   ? __ldcg(src + s1 * sstride + static_cast<int64_t>(i) * N)
                                   : 0.0f;
              }
#pragma unroll
              for (int s1 = 0; s1 < SB; ++s1)
#pragma unroll
                for (int i = 0; i < TB; ++i) sum[i] += v[s1][i];
            }
            __nv_bfloat16* const dst = y + static_cast<int64_t>(m0 + i0) * N + n;
            if (whole) {
#pragma unroll
              for (int i = 0; i < TB; ++i) dst[static_cast<int64_t>(i) * N] = __float2bfloat16_rn(sum[i]);
            } else {
#pragma unroll
              for (int i = 0; i < TB; ++i)
                if (m0 + i0 + i < M) dst[static_cast<int64_t>(i) * N] = __float2bfloat16_rn(sum[i]);
            }
          }
        }
        named_bar(1, 128);
      }
      if (warp == kEpi && lane == 0) QRR_STAMP(3, 3, units);
    }
  } else {
    // ------------------------------ dequant ------------------------------
    // The G warps of a sub-partition share its TMEM lane quarter q and take A
    // chunks from a per-quarter counter in order, so a warp that falls behind
    // holds up only its own chunk: the next free warp takes the chunks after it.
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    // TMA swizzle of the code tile: 16-byte piece p of row r sits at
    // p ^ (r & 7) for 128-byte rows and p ^ ((r >> 2) & 1) for 32-byte rows,
    // which keeps every 8-thread phase of a 16-byte shared load on distinct banks
    const int rot = BK == 256 ? (row & 7) : ((row >> 2) & 1);
    // this CTA's A chunks: its units in order, (nk + nl) stages of CPS chunks
    uint32_t total = 0;
    for (int ui = 0; ui < n_my; ++ui) {
      int j, nt, mt, sp, c0, nk, nl;
      locate(unit_at(ui), j, nt, mt, sp, c0, nk, nl);
      total += static_cast<uint32_t>((nk + nl) * C::CPS);
    }
    int ui = -1;
    uint32_t ubeg = 0, uend = 0;  // chunk range of unit u
    int j = 0, nt = 0, mt = 0, sp = 0, c0 = 0, nk = 0, nl = 0;
    // the unit's layer fields, read once per unit (see the epilogue)
    int LM = 0, Lr = 0, n = 0;
    const uint16_t* LB = nullptr;
    const uint8_t* srow = nullptr;
    while (true) {
      uint32_t chunk = 0;
      if (lane == 0) chunk = atomicAdd(&sh.next_chunk[q], 1u);
      chunk = __shfl_sync(0xFFFFFFFFu, chunk, 0);
      if (chunk >= total) break;
      while (chunk >= uend) {  // claims only grow: move forward to the chunk's unit
        ++ui;
        locate(unit_at(ui), j, nt, mt, sp, c0, nk, nl);
        ubeg = uend;
        uend += static_cast<uint32_t>((nk + nl) * C::CPS);
        LM = p.layer[j].M;
        Lr = p.layer[j].r;
        LB = p.layer[j].B;
        n = nt * 128 + row;
        srow = p.layer[j].scales + static_cast<int64_t>(n) * (p.layer[j].K / 16);
      }
      const int c = static_cast<int>((chunk - ubeg) / C::CPS);   // stage within the unit
      const int hc = static_cast<int>((chunk - ubeg) % C::CPS);  // chunk within the stage
      const uint32_t sseq = chunk / C::CPS;                      // stage sequence number of the CTA
      const int sidx = static_cast<int>(sseq % C::STAGES);
      const int slot = static_cast<int>(chunk % C::AST);
      {
        {
          if (q == 2 && lane == 0) QRR_STAMP(4, 0, chunk);
          if (q != 2 && lane == 0) QRR_STAMP(5 + (q == 3 ? 2 : q), 2, chunk);
          uint32_t scw[C::ACH / 64];
          if constexpr (!C::SC_TMA) {
            if (c < nk) scw[0] = __ldg(reinterpret_cast<const uint32_t*>(srow + (c0 + c) * (BK / 16)));
          }
          // the slot was last written for chunk - AST; its MMAs are done once
          // the slot's own release barrier or (shallow ring) the stage that
          // chunk belonged to has been released
          bool free = true;
          if (chunk >= static_cast<uint32_t>(C::AST)) {
            if constexpr (C::SLOT_BARS) {
              free = wait(&sh.a_empty[slot], (chunk / C::AST - 1) & 1);
            } else {
              const uint32_t prev = (chunk - C::AST) / C::CPS;  // stage sequence number
              free = wait(&sh.empty[prev % C::STAGES], (prev / C::STAGES) & 1);
            }
          }
          if (q == 2 && lane == 0) QRR_STAMP(4, 3, chunk);
          if (!free || !mbar_wait(&sh.full[sidx], (sseq / C::STAGES) & 1, abort, p.status)) break;
          if (q == 2 && lane == 0) QRR_STAMP(4, 1, chunk);
          if (q != 2 && lane == 0) QRR_STAMP(5 + (q == 3 ? 2 : q), 1, chunk);
          tc_fence_after();
          const uint8_t* stage = tiles + sidx * C::STAGE;
          const uint32_t a_addr = tmem + lane_addr + C::A_COL + C::ACOLS * slot;
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
            // LoRA chunk: A word i holds (B[n, rb+i], B[n, rb+i]) against the
            // (high, low) halves of t' (on the f16 path the prologue wrote t'
            // already scaled by the token's 2^-p_m, the factor the
            // accumulator carries); zero past rank r.  The decode tile's B
            // rows sit in the stage's code slot, row-major [128][r].
            const int rb = (c - nk) * (BK / 2) + hc * (C::ACH / 2);
            const uint16_t* brow = F16 ? reinterpret_cast<const uint16_t*>(stage + C::X_BYTES) + row * Lr + rb
                                       : LB + static_cast<int64_t>(n) * Lr + rb;
#pragma unroll
            for (int h = 0; h < C::ACH / 64; ++h) {
              uint32_t out[32];
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                const int v8 = 4 * h + v4;
                uint4 bv = make_uint4(0, 0, 0, 0);
                if (rb + 8 * v8 < Lr) {
                  if constexpr (F16)
                    bv = reinterpret_cast<const uint4*>(brow)[v8];
                  else
                    bv = __ldg(reinterpret_cast<const uint4*>(brow) + v8);
                }
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
          if (q != 2 && lane == 0) QRR_STAMP(5 + (q == 3 ? 2 : q), 0, chunk);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            arrive_leader(&sh.a_full[slot]);
            mbar_arrive(&sh.empty[sidx]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) QRR_GSTAMP(3);
  // a pair ends together: no remote arrive or x half may reach a CTA that
  // has exited, and the pair's TMEM is released by both
  if constexpr (PAIR) cluster_sync();
  if (warp == kMma) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else
      tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------

namespace {

// dequant warpgroups of the decode (f16) kernels: three per lane quarter
// (measured: two are about 6% slower at 1 and 8 tokens, and four do not fit
// the TMEM ring beside double-buffered 64-column accumulators)
constexpr int kDecodeGroups = 3;

// grid: CTAs for units one at a time; a paired launch runs min(units,
// co-resident 2-CTA clusters) clusters instead.
template <int BN, int BK, bool F16, int G, bool PAIR = false>
cudaError_t launch_bn(const W4Params& p, int grid, bool after_prologue, cudaStream_t stream) {
  using C = Cfg<BN, BK, G, PAIR>;
  auto kernel = w4a16_tc_kernel<BN, BK, F16, G, PAIR>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute la[2];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = after_prologue ? 1 : 0;
  la[1].id = cudaLaunchAttributeClusterDimension;
  la[1].val.clusterDim.x = PAIR ? 2 : 1;
  la[1].val.clusterDim.y = 1;
  la[1].val.clusterDim.z = 1;
  cfg.attrs = la;
  cfg.numAttrs = PAIR ? 2 : 1;
  if (PAIR) {
    cfg.gridDim = dim3(2);
    int clusters = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorLaunchOutOfResources;
    grid = 2 * (grid < clusters ? grid : clusters);
  }
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

int decode_grid() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return kSMs;
  }
  if (cached[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
      cudaGetLastError();
      sms = kSMs;
    }
    cached[dev] = sms < kMaxTableCtas ? sms : kMaxTableCtas;
  }
  return cached[dev];
}

namespace {

int stream_k_units_build(const int* kc, const int* nl, const int* n_tiles, const int* m_tiles, int count, int grid,
                         W4Params* p, int* max_pieces) {
  long long total = 0;
  for (int j = 0; j < count; ++j) {
    max_pieces[j] = 1;
    total += static_cast<long long>(n_tiles[j]) * m_tiles[j] * (kc[j] + nl[j]);
  }
  if (total == 0 || count > 16) return total == 0 ? 0 : -1;
  if (grid > total) grid = static_cast<int>(total);
  if (grid < 1 || grid > kMaxTableCtas) return -1;
  struct Seg {
    int j, t, s0, s1;
  };
  std::vector<Seg> seg;
  std::vector<int> first(grid + 1);
  int j = 0, t = 0;
  long long ts = 0;  // first stage of tile (j, t)
  for (int b = 0; b < grid; ++b) {
    const long long lo = total * b / grid, hi = total * (b + 1) / grid;
    first[b] = static_cast<int>(seg.size());
    long long pos = lo;
    while (pos < hi) {
      while (n_tiles[j] * m_tiles[j] == 0 || kc[j] + nl[j] == 0) {  // layers without stages
        ++j;
        t = 0;
      }
      const long long len = kc[j] + nl[j];
      const long long end = hi < ts + len ? hi : ts + len;
      seg.push_back({j, t, static_cast<int>(pos - ts), static_cast<int>(end - ts)});
      pos = end;
      if (end == ts + len) {  // next tile
        ts += len;
        if (++t == n_tiles[j] * m_tiles[j]) {
          ++j;
          t = 0;
        }
      }
    }
  }
  first[grid] = static_cast<int>(seg.size());
  const int n = static_cast<int>(seg.size());
  if (n > kMaxTableUnits) return -1;
  // a tile's pieces are consecutive: index within the tile and tile counts
  std::vector<int> sp(n), pieces(n);
  for (int i = 0; i < n; ++i) sp[i] = (i > 0 && seg[i - 1].j == seg[i].j && seg[i - 1].t == seg[i].t) ? sp[i - 1] + 1 : 0;
  for (int i = n - 1; i >= 0; --i)
    pieces[i] = (i + 1 < n && seg[i + 1].j == seg[i].j && seg[i + 1].t == seg[i].t) ? pieces[i + 1] : sp[i] + 1;
  for (int i = 0; i < n; ++i) {
    const Seg& g = seg[i];
    const int mt = g.t / n_tiles[g.j], nt = g.t % n_tiles[g.j];
    const int K = kc[g.j];
    const int c0 = g.s0 < K ? g.s0 : K;
    const int nk = (g.s1 < K ? g.s1 : K) - c0;
    const int l = (nl[g.j] > 0 && g.s1 > K) ? 1 : 0;
    if (mt > 15 || nt > 0xFFFF || pieces[i] > 0xFF || c0 > 0xFFF || nk > 0x7FF || sp[i] > 0xFF) return -1;
    max_pieces[g.j] = pieces[i] > max_pieces[g.j] ? pieces[i] : max_pieces[g.j];
    if (p != nullptr) {
      p->unit[i][0] = static_cast<uint32_t>(g.j) | static_cast<uint32_t>(mt) << 4 | static_cast<uint32_t>(nt) << 8 |
                      static_cast<uint32_t>(pieces[i]) << 24;
      p->unit[i][1] = static_cast<uint32_t>(c0) | static_cast<uint32_t>(nk) << 12 |
                      static_cast<uint32_t>(sp[i]) << 23 | static_cast<uint32_t>(l) << 31;
    }
  }
  if (p != nullptr) {
    for (int b = 0; b <= grid; ++b) p->unit_off[b] = static_cast<uint16_t>(first[b]);
    p->use_table = 1;
    p->table_grid = grid;
    p->total_units = n;
  }
  return n;
}

// Longest processing time first: a unit costs its K stages plus its LoRA
// stage plus its epilogue (about half a stage, or three when it writes a
// split-K partial and may run the reduction); each unit in turn, costliest
// first, goes to the least loaded CTA, which takes its units in index order.
void lpt_units_build(W4Params& p, int bk, int grid) {
  p.use_table = 0;
  struct U {
    double cost;
    int j, mt, nt, sp, c0, nk, nl, pieces;
  };
  std::vector<U> us;
  for (int j = 0; j < p.count; ++j) {
    const W4Layer& L = p.layer[j];
    const int kc = L.K / bk, ksub = bk / 64;
    for (int sp = 0; sp < L.splits; ++sp)
      for (int mt = 0; mt < L.m_tiles; ++mt)
        for (int nt = 0; nt < L.n_tiles; ++nt) {
          const int c0 = sp * L.kcps;
          const int nk = std::min(c0 + L.kcps, kc) - c0;
          const int nl = (L.r > 0 && sp == L.splits - 1) ? (L.lora_chunks + ksub - 1) / ksub : 0;
          us.push_back({nk + nl + (L.splits > 1 ? 3.0 : 0.5), j, mt, nt, sp, c0, nk, nl, L.splits});
        }
  }
  const int n = static_cast<int>(us.size());
  if (n == 0 || n > kMaxTableUnits || p.count > 16) return;
  if (grid > n) grid = n;
  if (grid < 1 || grid > kMaxTableCtas) return;
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return us[a].cost > us[b].cost; });
  std::vector<double> load(grid, 0.0);
  std::vector<std::vector<int>> mine(grid);
  for (int i : order) {
    int best = 0;
    for (int b = 1; b < grid; ++b)
      if (load[b] < load[best]) best = b;
    load[best] += us[i].cost;
    mine[best].push_back(i);
  }
  int k = 0;
  for (int b = 0; b < grid; ++b) {
    std::sort(mine[b].begin(), mine[b].end());
    p.unit_off[b] = static_cast<uint16_t>(k);
    for (int i : mine[b]) {
      const U& u = us[i];
      if (u.mt > 15 || u.nt > 0xFFFF || u.pieces > 0xFF || u.c0 > 0xFFF || u.nk > 0x7FF || u.sp > 0xFF) return;
      p.unit[k][0] = static_cast<uint32_t>(u.j) | static_cast<uint32_t>(u.mt) << 4 |
                     static_cast<uint32_t>(u.nt) << 8 | static_cast<uint32_t>(u.pieces) << 24;
      p.unit[k][1] = static_cast<uint32_t>(u.c0) | static_cast<uint32_t>(u.nk) << 12 |
                     static_cast<uint32_t>(u.sp) << 23 | static_cast<uint32_t>(u.nl) << 31;
      ++k;
    }
  }
  p.unit_off[grid] = static_cast<uint16_t>(k);
  p.total_units = n;
  p.table_grid = grid;
  p.use_table = 1;
}

// The last few unit tables, kept while the caller repeats a launch shape
// (decode calls cycle through a handful of token counts): building one walks
// every stage or sorts every unit, host time that would otherwise be spent
// on every call.
struct TableEntry {
  bool used = false;
  std::vector<int> key;
  int n = -1, grid_used = 0, use_table = 0;
  int pieces[kMaxW4Layers];
  uint16_t off[kMaxTableCtas + 1];
  uint32_t unit[kMaxTableUnits][2];
};
std::mutex g_table_mu;
TableEntry g_tables[4];
int g_table_next = 0;
W4Params g_table_scratch;  // guarded by g_table_mu

TableEntry* table_find(const std::vector<int>& key) {
  for (TableEntry& e : g_tables)
    if (e.used && e.key == key) return &e;
  TableEntry& e = g_tables[g_table_next];
  g_table_next = (g_table_next + 1) % 4;
  e.used = false;
  e.key = key;
  return &e;
}

void table_store(TableEntry& e, const W4Params& p, int n) {
  e.n = n;
  e.use_table = p.use_table;
  e.grid_used = p.table_grid;
  if (p.use_table) {
    memcpy(e.off, p.unit_off, sizeof(uint16_t) * static_cast<size_t>(p.table_grid + 1));
    memcpy(e.unit, p.unit, sizeof(uint32_t) * 2 * static_cast<size_t>(p.total_units));
  }
  e.used = true;
}

void table_load(const TableEntry& e, W4Params& p, int n_units) {
  p.use_table = e.use_table;
  if (!e.use_table) return;
  p.table_grid = e.grid_used;
  p.total_units = n_units;
  memcpy(p.unit_off, e.off, sizeof(uint16_t) * static_cast<size_t>(e.grid_used + 1));
  memcpy(p.unit, e.unit, sizeof(uint32_t) * 2 * static_cast<size_t>(n_units));
}

}  // namespace

int stream_k_units(const int* kc, const int* nl, const int* n_tiles, const int* m_tiles, int count, int grid,
                   W4Params* p, int* max_pieces) {
  std::vector<int> key = {0, count, grid};
  for (int j = 0; j < count; ++j) key.insert(key.end(), {kc[j], nl[j], n_tiles[j], m_tiles[j]});
  std::lock_guard<std::mutex> lock(g_table_mu);
  TableEntry* e = table_find(key);
  if (!e->used) {
    g_table_scratch.use_table = 0;
    const int n = stream_k_units_build(kc, nl, n_tiles, m_tiles, count, grid, &g_table_scratch, e->pieces);
    table_store(*e, g_table_scratch, n);
  }
  for (int j = 0; j < count; ++j) max_pieces[j] = e->pieces[j];
  if (p != nullptr && e->n >= 0) table_load(*e, *p, e->n);
  return e->n;
}

void lpt_units(W4Params& p, int bk, int grid) {
  std::vector<int> key = {1, p.count, bk, grid};
  for (int j = 0; j < p.count; ++j) {
    const W4Layer& L = p.layer[j];
    key.insert(key.end(), {L.n_tiles, L.m_tiles, L.splits, L.kcps, L.K, L.r, L.lora_chunks});
  }
  std::lock_guard<std::mutex> lock(g_table_mu);
  TableEntry* e = table_find(key);
  if (!e->used) {
    g_table_scratch.count = p.count;
    for (int j = 0; j < p.count; ++j) g_table_scratch.layer[j] = p.layer[j];
    lpt_units_build(g_table_scratch, bk, grid);
    table_store(*e, g_table_scratch, g_table_scratch.use_table ? g_table_scratch.total_units : -1);
  }
  p.use_table = 0;
  if (e->n >= 0) table_load(*e, p, e->n);
}

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

// after_prologue: the previous kernel in the stream is the prologue that
// writes x16 / pexp / t'; this launch may then start before it completes.
cudaError_t launch_w4a16_tc(W4Params& p, int bn, bool f16, bool pair, bool after_prologue, cudaStream_t stream) {
  if (p.use_table) {
    // decode with the unit table the caller built for its grid
    if (p.total_units == 0) return cudaSuccess;
    switch (bn) {
      case 16: return launch_bn<16, 256, true, kDecodeGroups>(p, p.table_grid, after_prologue, stream);
      case 32: return launch_bn<32, 256, true, kDecodeGroups>(p, p.table_grid, after_prologue, stream);
      default: return launch_bn<64, 256, true, kDecodeGroups>(p, p.table_grid, after_prologue, stream);
    }
  }
  int units = 0;
  for (int j = 0; j < p.count; ++j) {
    p.layer[j].first_unit = units;
    units += (pair ? p.layer[j].n_tiles / 2 : p.layer[j].n_tiles) * p.layer[j].m_tiles * p.layer[j].splits;
  }
  p.total_units = units;
  if (units == 0) return cudaSuccess;
  int dev = 0, sms = kSMs;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = units < sms ? units : sms;
  if (f16) {
    switch (bn) {
      case 16: return launch_bn<16, 256, true, kDecodeGroups>(p, grid, after_prologue, stream);
      case 32: return launch_bn<32, 256, true, kDecodeGroups>(p, grid, after_prologue, stream);
      default: return launch_bn<64, 256, true, kDecodeGroups>(p, grid, after_prologue, stream);
    }
  }
  if (bn == 128) return launch_bn<128, 64, false, 2>(p, grid, after_prologue, stream);
  if (pair) return launch_bn<256, 64, false, 3, true>(p, units, after_prologue, stream);
  return launch_bn<256, 64, false, 2>(p, grid, after_prologue, stream);
}

}  // namespace qrr

#ifdef QRR_TRACE_BUILD
extern "C" int qrr_trace_read(unsigned long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, qrr::qrr_trace_buf, sizeof(qrr::qrr_trace_buf)));
}
extern "C" int qrr_gtrace_read(unsigned long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, qrr::qrr_gtrace_buf, sizeof(qrr::qrr_gtrace_buf)));
}
extern "C" int qrr_trace_clear(void) {
  static unsigned long long zeros[8 * 4 * 256] = {};
  cudaMemcpyToSymbol(qrr::qrr_gtrace_buf, zeros, sizeof(qrr::qrr_gtrace_buf));
  return static_cast<int>(cudaMemcpyToSymbol(qrr::qrr_trace_buf, zeros, sizeof(zeros)));
}
#endif

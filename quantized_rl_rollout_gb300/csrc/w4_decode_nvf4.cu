// Decode (at most 64 tokens) of the NVFP4 W4A16 + LoRA linear on the native
// block-scaled tensor-core MMA:
//
//   y[m, n] = s_t 2^e_m (sum_k c[n, k] s_b[n, k / 16] x'[m, k] + l'[m, n])
//
// with c the E2M1 codes, s_b the E4M3 block scales, s_t the tensor scale
// ("QeRL: Beyond Efficiency", abstract: NVFP4 weights under LoRA; the NVFP4
// layout: one E4M3 scale per 16 weights and one fp32 tensor scale),
// x' = x 2^-e_m and l' the adapter term in the same units.
//
// The weight's codes and block scales go from HBM by TMA straight into
// tcgen05.mma kind::mxf4nvf4 (scale_vec::4X, UE4M3 scales): an NVFP4 block
// scale is never negative, so its E4M3 byte is its UE4M3 byte, and no CUDA
// core touches a weight.  The activations enter as the E2M1 digit planes the
// decode prologue writes: x' = sum_p d_p 6^-p to within 6^-5 (|x'| <= 6),
// plane p one block of the B operand's rows, all B scales 1.  The
// accumulator keeps every plane's sum in its own columns and the epilogue
// combines them, sum_p 6^-p D_p.  The adapter stage (t' = the prologue's
// scaled x A^T as bf16 high/low pairs) is a kind::f16 MMA chain with A in
// tensor memory (B's rows, each value twice, against t''s pairs), added to
// plane 0's columns.
//
// Work division: the unit table of the launch (stream-K ranges of each
// tile's stages, the adapter stage last); a tile cut between CTAs writes
// fp32 partials, one slot per piece, and the piece that finishes last sums
// them in piece order.
//
//   warp 0      TMA: per stage, codes [128 x 128 B] and block scales
//               [128 x 16 B] (independent of the prologue: the first ring is
//               issued at once), then the x planes [rows x 128 B]; for the
//               adapter stage B's rows [128 x r] and the t' tile
//   warp 1      MMA: 4 x mxf4nvf4 (M 128, N nmma, K 64) per stage and
//               N-half (two halves when the planes exceed 256 rows)
//   warps 2..5  one per TMEM lane quarter: the B scale cells once (1.0), then
//               per stage the tile's block scales from shared into tensor
//               memory, per adapter stage the A operand of the LoRA MMA
//   warps 6..9  epilogue, one per lane quarter
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

// Development builds (-DQRR_TRACE_BUILD) record global-timer stamps per CTA:
// start, planes released (the prologue has completed), first MMA, end.
// Ordinary builds compile them away.
#ifdef QRR_TRACE_BUILD
__device__ unsigned long long qrr_ntrace_buf[256][4];
#define QRR_NSTAMP(ev)                                               \
  do {                                                               \
    unsigned long long t_;                                           \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));           \
    if (blockIdx.x < 256) qrr_ntrace_buf[blockIdx.x][ev] = t_;       \
  } while (0)
#else
#define QRR_NSTAMP(ev) \
  do {                 \
  } while (0)
#endif

namespace {

constexpr int kThreads = 320;
constexpr int kCodeBytes = 128 * 128;  // 128 rows x 256 K of packed E2M1
constexpr int kScaleBytes = 128 * 16;  // 128 rows x 16 block scales
constexpr uint32_t kOnes = 0x38383838u;  // four UE4M3 scales of 1.0
// All of an SM's shared memory, whatever the ring needs: no CTA of another
// grid (the prologue, which allocates tensor memory) can share the SM while
// this CTA holds all 512 columns.
constexpr size_t kSmem = 227 * 1024;
constexpr float kInv6 = 1.0f / 6.0f;

struct Ctl {
  uint64_t full[8], full_x[8], empty[8];  // full: codes + scales (or B's rows); full_x: planes (or t')
  uint64_t sf_full[8], sf_empty[8];      // block-scale cells in tensor memory
  uint64_t lora_full, lora_empty;        // the adapter's A operand in tensor memory
  uint64_t d_full[2], d_empty[2];
  uint64_t done;
  uint32_t tmem;
  int abort;
  int last;
};

// sum_p 6^-p d[p] (Horner), or d[0] alone for a piece that is only the
// adapter stage (the other planes' columns were not written)
__device__ __forceinline__ float combine_planes(const uint32_t (&d)[kXPlanes], bool lora_only) {
  float a = __uint_as_float(d[kXPlanes - 1]);
#pragma unroll
  for (int pl = kXPlanes - 2; pl >= 0; --pl) a = fmaf(a, kInv6, __uint_as_float(d[pl]));
  return lora_only ? __uint_as_float(d[0]) : a;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) w4_decode_nvf4_kernel(const __grid_constant__ W4Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Nvf4Geo g = nvf4_geo(p.layer[0].M);
  const int S = g.stages, SF = g.sf_slots;
  Ctl& sh = *reinterpret_cast<Ctl*>(tiles + S * g.stage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &sh.abort;
  if (threadIdx.x == 0) QRR_NSTAMP(0);
  const int sk0 = p.unit_off[blockIdx.x];
  const int n_my = p.unit_off[blockIdx.x + 1] - sk0;
  auto wait = [&](uint64_t* bar, uint32_t parity) { return mbar_wait(bar, parity, abort, p.status); };
  // unit i of this CTA -> layer, n tile, piece, its K stages, adapter stage,
  // the tile's piece count (the m tile is 0: one tile holds every token)
  auto locate = [&](int i, int& j, int& nt, int& sp, int& c0, int& nk, int& nl, int& pieces) {
    const uint32_t w0 = p.unit[sk0 + i][0], w1 = p.unit[sk0 + i][1];
    j = static_cast<int>(w0 & 0xFu);
    nt = static_cast<int>((w0 >> 8) & 0xFFFFu);
    pieces = static_cast<int>(w0 >> 24);
    c0 = static_cast<int>(w1 & 0xFFFu);
    nk = static_cast<int>((w1 >> 12) & 0x7FFu);
    sp = static_cast<int>((w1 >> 23) & 0xFFu);
    nl = static_cast<int>(w1 >> 31);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.full_x[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int s = 0; s < SF; ++s) {
      mbar_init(&sh.sf_full[s], 4);
      mbar_init(&sh.sf_empty[s], 1);
    }
    mbar_init(&sh.lora_full, 4);
    mbar_init(&sh.lora_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.d_full[b], 1);
      mbar_init(&sh.d_empty[b], 4);
    }
    mbar_init(&sh.done, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  if (warp == 0) {
    // ------------------------------ TMA ------------------------------
    if (elect_one()) {
      struct Cursor {
        int i = -1, c = 0, j = 0, nt = 0, sp = 0, c0 = 0, nk = 0, nl = 0, pieces = 0;
      };
      auto next = [&](Cursor& k) {  // the CTA's next stage; false past the last
        if (k.i >= n_my) return false;
        if (k.i >= 0 && ++k.c < k.nk + k.nl) return true;
        k.c = 0;
        for (++k.i; k.i < n_my; ++k.i) {
          locate(k.i, k.j, k.nt, k.sp, k.c0, k.nk, k.nl, k.pieces);
          if (k.nk + k.nl > 0) return true;
        }
        return false;
      };
      auto issue_w = [&](const Cursor& k, int idx) {
        uint8_t* const st = tiles + idx * g.stage;
        uint64_t* const fb = &sh.full[idx];
        if (k.c < k.nk) {
          mbar_arrive_expect_tx(fb, kCodeBytes + kScaleBytes);
          tma_load_2d(&p.layer[k.j].tcodes, fb, st + g.xb, (k.c0 + k.c) * 128, k.nt * 128);
          tma_load_2d(&p.layer[k.j].tscales, fb, st + g.xb + kCodeBytes, (k.c0 + k.c) * 16, k.nt * 128);
        } else {
          // adapter stage: the tile's rows of B, row-major [128][r]
          mbar_arrive_expect_tx(fb, 128u * static_cast<uint32_t>(p.layer[k.j].r) * 2u);
          tma_load_2d(&p.layer[k.j].tb, fb, st + g.xb, 0, k.nt * 128);
        }
      };
      auto issue_x = [&](const Cursor& k, int idx) {
        uint8_t* const st = tiles + idx * g.stage;
        uint64_t* const fb = &sh.full_x[idx];
        if (k.c < k.nk) {
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(g.rows) * 128u);
          for (int h = 0; h < g.nh; ++h)
            tma_load_2d(&p.layer[k.j].tp, fb, st + h * g.nmma * 128, (k.c0 + k.c) * 128, h * g.nmma);
        } else {
          // t' columns [0, 128): two 64-wide sub-tiles (past t''s width: zeros)
          mbar_arrive_expect_tx(fb, 2u * static_cast<uint32_t>(g.bn) * 128u);
          tma_load_2d(&p.layer[k.j].tt, fb, st, 0, 0);
          tma_load_2d(&p.layer[k.j].tt, fb, st + g.bn * 128, 64, 0);
        }
      };
      Cursor kw, kx;
      uint32_t nw = 0;  // stages whose weights are issued
      while (nw < static_cast<uint32_t>(S) && next(kw)) {
        issue_w(kw, static_cast<int>(nw));
        ++nw;
      }
      griddep_wait();  // the planes and t' are the prologue's
      QRR_NSTAMP(1);
      for (uint32_t nx = 0; nx < nw; ++nx) {
        next(kx);
        issue_x(kx, static_cast<int>(nx));
      }
      while (next(kw)) {
        next(kx);
        const uint32_t idx = nw % S, use = nw / S;
        if (!wait(&sh.empty[idx], (use - 1) & 1)) break;
        issue_w(kw, static_cast<int>(idx));
        issue_x(kx, static_cast<int>(idx));
        ++nw;
      }
      // every issued copy has landed before the CTA exits
      volatile int no_abort = 0;
      for (uint32_t k = 0; k < static_cast<uint32_t>(S) && k < nw; ++k) {
        const uint32_t i = nw - 1 - k;
        mbar_wait(&sh.full[i % S], (i / S) & 1, &no_abort, p.status);
        mbar_wait(&sh.full_x[i % S], (i / S) & 1, &no_abort, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA ------------------------------
    if (elect_one()) {
      const uint32_t id_main = make_idesc_nvf4(128, static_cast<uint32_t>(g.nmma));
      const uint32_t id_lora = make_idesc(kFmtBF16, kFmtBF16, 128, static_cast<uint32_t>(g.bn));
      uint32_t seq = 0, sfseq = 0, lseq = 0;
      bool ok = true;
      for (int ui = 0; ui < n_my && ok; ++ui) {
        int j, nt, sp, c0, nk, nl, pieces;
        locate(ui, j, nt, sp, c0, nk, nl, pieces);
        const int db = ui % g.nd;
        const int duse = ui / g.nd;
        if (duse > 0 && !wait(&sh.d_empty[db], (duse - 1) & 1)) break;
        tc_fence_after();
        const uint32_t dcol = tmem + static_cast<uint32_t>(db * g.rows);
        for (int c = 0; c < nk + nl; ++c, ++seq) {
          const int idx = static_cast<int>(seq % S);
          const uint32_t par = (seq / S) & 1;
          if (!wait(&sh.full[idx], par) || !wait(&sh.full_x[idx], par)) {
            ok = false;
            break;
          }
          const uint32_t xs = smem_u32(tiles + idx * g.stage);
          if (c < nk) {
            const int slot = static_cast<int>(sfseq % SF);
            if (!wait(&sh.sf_full[slot], (sfseq / SF) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (seq == 0) QRR_NSTAMP(2);
            const uint32_t cs = xs + static_cast<uint32_t>(g.xb);
            const uint32_t sfa = tmem + static_cast<uint32_t>(g.sf0 + 16 * slot);
            // plane rows [h nmma, (h + 1) nmma) into accumulator columns alike
            for (int h = 0; h < g.nh; ++h) {
              const uint32_t xh = xs + static_cast<uint32_t>(h * g.nmma * 128);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_nvf4_ss(dcol + static_cast<uint32_t>(h * g.nmma), sw128_desc(cs + 32 * k), sw128_desc(xh + 32 * k),
                            id_main, sfa + 4 * k, tmem + static_cast<uint32_t>(g.sfb0), (c > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(&sh.sf_empty[slot]);
            ++sfseq;
          } else {
            if (!wait(&sh.lora_full, lseq & 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // K16 step k: t' sub-tile k / 4, 32 bytes into its rows per step
            const uint64_t b0 = sw128_desc(xs);
            uint64_t bd[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              bd[k] = b0 + static_cast<uint64_t>(((k >> 2) * g.bn * 128 + 32 * (k & 3)) >> 4);
            mma8_ts(dcol, tmem + static_cast<uint32_t>(g.lora0), bd, id_lora, c > 0 ? 1u : 0u);
            mma_commit(&sh.lora_empty);
            ++lseq;
          }
          mma_commit(&sh.empty[idx]);
        }
        if (!ok) break;
        mma_commit(&sh.d_full[db]);
      }
      // every MMA has completed before the tensor memory is released
      mma_commit(&sh.done);
      volatile int no_abort = 0;
      mbar_wait(&sh.done, 0, &no_abort, p.status);
    }
  } else if (warp < 6) {
    // ------------------------- scale cells / adapter A -------------------------
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    {
      uint32_t ones[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) ones[i] = kOnes;
      tmem_st16(tmem + lane_addr + static_cast<uint32_t>(g.sfb0), ones);
    }
    uint32_t seq = 0, sfseq = 0, lseq = 0;
    bool ok = true;
    for (int ui = 0; ui < n_my && ok; ++ui) {
      int j, nt, sp, c0, nk, nl, pieces;
      locate(ui, j, nt, sp, c0, nk, nl, pieces);
      const int r = p.layer[j].r;
      for (int c = 0; c < nk + nl; ++c, ++seq) {
        const int idx = static_cast<int>(seq % S);
        if (!wait(&sh.full[idx], (seq / S) & 1)) {
          ok = false;
          break;
        }
        const uint8_t* const st = tiles + idx * g.stage;
        uint64_t* arrive_on;
        if (c < nk) {
          const int slot = static_cast<int>(sfseq % SF);
          if (sfseq >= static_cast<uint32_t>(SF) && !wait(&sh.sf_empty[slot], ((sfseq / SF) - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // the row's 16 block scales of this stage, four per MMA; each MMA's
          // cell is written to the four columns of its group, which covers
          // every column the MMA may read for the row
          const uint4 sv = *reinterpret_cast<const uint4*>(st + g.xb + kCodeBytes + row * 16);
          const uint32_t wv[4] = {sv.x, sv.y, sv.z, sv.w};
          uint32_t cells[16];
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) cells[4 * k + i] = wv[k];
          tmem_st16(tmem + lane_addr + static_cast<uint32_t>(g.sf0 + 16 * slot), cells);
          arrive_on = &sh.sf_full[slot];
          ++sfseq;
        } else {
          if (lseq > 0 && !wait(&sh.lora_empty, (lseq - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // A word i holds (B[n, i], B[n, i]) against t''s (high, low) pair
          // of rank i; zero past r
          const uint16_t* const brow = reinterpret_cast<const uint16_t*>(st + g.xb) + row * r;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t out[32];
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              const int v8 = 4 * h + v4;  // ranks 8 v8 .. 8 v8 + 7
              uint4 bv = make_uint4(0u, 0u, 0u, 0u);
              if (8 * v8 < r) bv = reinterpret_cast<const uint4*>(brow)[v8];
              const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                out[8 * v4 + 2 * e] = (bw[e] & 0xFFFFu) * 0x10001u;
                out[8 * v4 + 2 * e + 1] = (bw[e] >> 16) * 0x10001u;
              }
            }
            tmem_st32(tmem + lane_addr + static_cast<uint32_t>(g.lora0 + 32 * h), out);
          }
          arrive_on = &sh.lora_full;
          ++lseq;
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(arrive_on);
      }
    }
  } else {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    griddep_wait();  // the per-token exponents and the tile counters are the prologue's
    for (int ui = 0; ui < n_my; ++ui) {
      int j, nt, sp, c0, nk, nl, pieces;
      locate(ui, j, nt, sp, c0, nk, nl, pieces);
      // the layer's fields, read once: read through the parameter with a
      // runtime index, they would be reloaded after every store
      const int M = p.layer[j].M, N = p.layer[j].N;
      const int* const pexp = p.layer[j].pexp;
      __nv_bfloat16* const y = p.layer[j].y;
      float* const partial = p.layer[j].partial;
      uint32_t* const counters = p.layer[j].counters;
      const float ts = *p.layer[j].tensor_scale;
      const float gs = ts > 0.0f ? ts : 1.0f;
      const int n = nt * 128 + 32 * q + lane;
      const int db = ui % g.nd;
      if (!wait(&sh.d_full[db], (ui / g.nd) & 1)) break;
      tc_fence_after();
      const bool lora_only = nk == 0;
      float* const part = pieces > 1 ? partial + static_cast<int64_t>(sp) * M * N : nullptr;
      const uint32_t dbase = tmem + lane_addr + static_cast<uint32_t>(db * g.rows);
      if (g.ms == 1) {
        // one token: plane p in column p
        uint32_t v[8];
        tmem_ld8(dbase, v);
        const float f = __fmul_rn(gs, pow2_from_exp(__ldg(pexp)));
        tmem_ld_wait();
        const uint32_t d[kXPlanes] = {v[0], v[1], v[2], v[3], v[4], v[5]};
        const float o = combine_planes(d, lora_only) * f;
        if (part != nullptr)
          part[n] = o;
        else
          y[n] = __float2bfloat16_rn(o);
      } else {
        // slabs of 8 tokens: plane p of token m in column p * ms + m
#pragma unroll 1
        for (int m0 = 0; m0 < M; m0 += 8) {
          uint32_t v[kXPlanes][8];
#pragma unroll
          for (int pl = 0; pl < kXPlanes; ++pl) tmem_ld8(dbase + static_cast<uint32_t>(pl * g.ms + m0), v[pl]);
          const int cnt = M - m0;
          float f[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(gs, pow2_from_exp(__ldg(pexp + min(m0 + i, M - 1))));
          tmem_ld_wait();
          float o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t d[kXPlanes] = {v[0][i], v[1][i], v[2][i], v[3][i], v[4][i], v[5][i]};
            o[i] = combine_planes(d, lora_only) * f[i];
          }
          if (part != nullptr) {
            float* const dst = part + static_cast<int64_t>(m0) * N + n;
            if (cnt >= 8) {
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[static_cast<int64_t>(i) * N] = o[i];
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (i < cnt) dst[static_cast<int64_t>(i) * N] = o[i];
            }
          } else {
            __nv_bfloat16* const dst = y + static_cast<int64_t>(m0) * N + n;
            if (cnt >= 8) {
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[static_cast<int64_t>(i) * N] = __float2bfloat16_rn(o[i]);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (i < cnt) dst[static_cast<int64_t>(i) * N] = __float2bfloat16_rn(o[i]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.d_empty[db]);
      if (part != nullptr) {
        // all 128 epilogue threads have written their partials; one makes
        // them visible GPU-wide (the fence is cumulative over the barrier)
        // and takes a ticket; the tile's last piece sums all of them in
        // piece order
        named_bar(1, 128);
        if (warp == 6 && lane == 0) {
          __threadfence();
          uint32_t* const cnt = counters + nt;
          const uint32_t prev = atomicAdd(cnt, 1u);
          sh.last = prev == static_cast<uint32_t>(pieces - 1);
          if (sh.last) {
            *cnt = 0u;  // ready for the next call
            __threadfence();
          }
        }
        named_bar(1, 128);
        if (sh.last) {
          constexpr int TB = 8, SB = 4;  // tokens per batch; pieces with loads in flight
          const int64_t pstride = static_cast<int64_t>(M) * N;
          for (int i0 = 0; i0 < M; i0 += TB) {
            float sum[TB];
#pragma unroll
            for (int i = 0; i < TB; ++i) sum[i] = 0.0f;
            for (int s0 = 0; s0 < pieces; s0 += SB) {
              float v[SB][TB];
              const float* const src = partial + static_cast<int64_t>(s0) * pstride + static_cast<int64_t>(i0) * N + n;
#pragma unroll
              for (int s1 = 0; s1 < SB; ++s1)
#pragma unroll
                for (int i = 0; i < TB; ++i)
                  v[s1][i] = (s0 + s1 < pieces && i0 + i < M)
                                 ? __ldcg(src + s1 * pstride + static_cast<int64_t>(i) * N)
                                 : 0.0f;
#pragma unroll
              for (int s1 = 0; s1 < SB; ++s1)
#pragma unroll
                for (int i = 0; i < TB; ++i) sum[i] += v[s1][i];
            }
            __nv_bfloat16* const dst = y + static_cast<int64_t>(i0) * N + n;
#pragma unroll
            for (int i = 0; i < TB; ++i)
              if (i0 + i < M) dst[static_cast<int64_t>(i) * N] = __float2bfloat16_rn(sum[i]);
          }
        }
        named_bar(1, 128);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) QRR_NSTAMP(3);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_w4_decode_nvf4(const W4Params& p, cudaStream_t stream) {
  if (p.total_units == 0 || p.count == 0) return cudaSuccess;
  if (p.layer[0].M < 1 || p.layer[0].M > kNvf4MaxM || !p.use_table || p.table_grid < 1 ||
      p.table_grid > kMaxTableCtas)
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e =
        cudaFuncSetAttribute(w4_decode_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.table_grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = la;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, w4_decode_nvf4_kernel, p);
}

}  // namespace qrr

#ifdef QRR_TRACE_BUILD
extern "C" int qrr_ntrace_read(unsigned long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, qrr::qrr_ntrace_buf, sizeof(qrr::qrr_ntrace_buf)));
}
#endif

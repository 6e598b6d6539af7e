// Blockwise-scaled FP8 GEMM with power-of-two scales on the native
// block-scaled tensor-core MMA (tcgen05.mma kind::mxf8f6f4, UE8M0 scales).
//
//   y[m,n] = sum_kb sa[m,kb] sw[n/128,kb] sum_{k in kb} e4m3(qa[m,k]) e4m3(qw[n,k])
//
// ("NVIDIA NeMo RL behaalt 48% ...", section "De technische doorbraak": FP8
// linear layers over 1x128 activation and 128x128 weight blocks; last
// paragraph before "Waarom dit belangrijk is": power-of-two scale factors.)
//
// With power-of-two scales every block's factor sa sw = 2^(ea + ew) is exactly
// what the block-scaled MMA applies to its 32-K products (2^(ua - 127) *
// 2^(uw - 127) for scale bytes ua, uw), so the whole K loop accumulates in one
// TMEM accumulator and nothing is promoted on the CUDA cores.
//
// A persistent CTA per SM computes 128 (tokens) x 256 (weight rows) tiles in
// turn; loads and scale bytes run ahead into the next tile while the epilogue
// drains the last one.
//   warp 0      TMA: per 128-wide K block, qa [128 x 128 B] and qw [256 x 128 B]
//               into a 4-stage ring (128-byte swizzle)
//   warp 1      MMA: 4 x kind::mxf8f6f4 (M128 N256 K32) per K block, scale byte
//               id = K block mod 4
//   warps 2..5  scales, one warp per TMEM lane quarter: for each group of four
//               K blocks, the UE8M0 bytes of the tile's 128 activation rows and
//               2 weight tiles, packed four K blocks per 32-bit cell, into an
//               8-group ring of scale columns
//   warps 6..13 epilogue: the fp32 accumulator out of TMEM, rounded to bf16;
//               TMEM is handed back before the stores
//
// UE8M0 covers 2^-127 .. 2^127.  A K block whose activation exponents ea (over
// the tile's rows) or weight exponents ew fall outside it is shifted as a
// whole: ua = ea + 127 + t, uw = ew + 127 - t with one t per (tile, K block),
// which leaves every product 2^(ea + ew) unchanged.  Only when no such t
// exists (exponents spread over more than the byte's range within one K
// block of one tile) are bytes clamped, and QRR_DEV_SCALE_RANGE is raised.  A
// scale that is not a power of two, negative or non-finite raises
// QRR_DEV_SCALE_RANGE too (the POW2 mode's promise is broken).
#include <cuda_bf16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 4;
constexpr int A_BYTES = BM * BK;                // 16 KB
constexpr int B_BYTES = BN * BK;                // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr int THREADS = 14 * 32;
constexpr uint32_t TMEM_COLS = 512;
constexpr int SF_COL0 = 256;   // scale columns after the 256-column accumulator
constexpr int SF_GROUPS = 8;   // ring of scale groups (four K blocks each)
constexpr int SF_STRIDE = 16;  // columns per group: A at +0..3, B at +8..15
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 1024;

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
  uint64_t full[STAGES], empty[STAGES];
  uint64_t sf_full[SF_GROUPS], sf_empty[SF_GROUPS];
  uint64_t d_full, d_empty, done;
  int ext[2][4][4][2];  // [group parity][writer warp][K block of group][min, max] of activation exponents
  uint32_t tmem;
  int abort;
};

// Exponent of a power-of-two scale: true with e set for s = 2^e (normal or
// subnormal fp32), false for zero; `bad` is raised for anything else.
__device__ __forceinline__ bool pow2_exponent(float s, int& e, bool& bad) {
  const uint32_t b = __float_as_uint(s);
  if (b == 0u || b == 0x80000000u) return false;
  if ((b >> 31) || (b >> 23) == 0xFFu) {
    bad = true;
    return false;
  }
  if (b >= 0x00800000u) {
    if (b & 0x7FFFFFu) bad = true;
    e = static_cast<int>(b >> 23) - 127;
  } else {
    if (b & (b - 1u)) bad = true;
    e = -149 + (31 - __clz(static_cast<int>(b)));
  }
  return true;
}

constexpr int kNone = 1 << 20;  // "no nonzero scale" sentinel of the min/max reductions

}  // namespace

__global__ void __launch_bounds__(THREADS, 1) fp8_gemm_mx_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared& sh = *reinterpret_cast<Shared*>(tiles + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kblocks = p.K / BK;
  const int groups = (kblocks + 3) / 4;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int total = n_tiles * ((p.M + BM - 1) / BM);
  volatile int* abort = &sh.abort;
  // persistent: the CTA takes tiles blockIdx.x, blockIdx.x + gridDim.x, ...;
  // weight tiles vary fastest, so the CTAs working at once share activation rows
  auto tile_of = [&](int t, int& m0, int& n0) {
    m0 = (t / n_tiles) * BM;
    n0 = (t % n_tiles) * BN;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int g = 0; g < SF_GROUPS; ++g) {
      mbar_init(&sh.sf_full[g], 4);
      mbar_init(&sh.sf_empty[g], 1);
    }
    mbar_init(&sh.d_full, 1);
    mbar_init(&sh.d_empty, 8);  // the eight epilogue warps have read the accumulator
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
    // ---------------- TMA producer (runs ahead across tiles) ----------------
    if (elect_one()) {
      tma_prefetch_desc(&p.ta);
      tma_prefetch_desc(&p.tb);
      int issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int m0, n0;
        tile_of(t, m0, n0);
        for (int kb = 0; kb < kblocks; ++kb, ++issued) {
          const int s = issued % STAGES, use = issued / STAGES;
          if (issued >= STAGES && !mbar_wait(&sh.empty[s], (use - 1) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh.full[s], STAGE_BYTES);
          uint8_t* a = tiles + s * STAGE_BYTES;
          tma_load_2d(&p.ta, &sh.full[s], a, kb * BK, m0);
          tma_load_2d(&p.tb, &sh.full[s], a + A_BYTES, kb * BK, n0);
        }
      }
      volatile int no_abort = 0;
      for (int i = issued - 1; i >= 0 && i >= issued - STAGES; --i)
        mbar_wait(&sh.full[i % STAGES], (i / STAGES) & 1, &no_abort, p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (elect_one()) {
      int stage = 0, grp = 0, tiles_done = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tiles_done) {
        // the epilogue has taken the previous tile's accumulator out of TMEM
        if (tiles_done > 0 && !mbar_wait(&sh.d_empty, (tiles_done - 1) & 1, abort, p.status)) break;
        tc_fence_after();
        for (int kb = 0; kb < kblocks; ++kb, ++stage) {
          const int s = stage % STAGES, use = stage / STAGES;
          const int j = kb & 3, slot = grp % SF_GROUPS;
          if (j == 0 && !mbar_wait(&sh.sf_full[slot], (grp / SF_GROUPS) & 1, abort, p.status)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&sh.full[s], use & 1, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(tiles + s * STAGE_BYTES), b = a + A_BYTES;
          const uint32_t sfa = tmem + SF_COL0 + SF_STRIDE * slot, sfb = sfa + 8;
          const uint32_t idesc = make_idesc_mx(BM, BN, static_cast<uint32_t>(j), static_cast<uint32_t>(j));
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_mxf8_ss(tmem, sw128_desc(a + 32 * k), sw128_desc(b + 32 * k), idesc, sfa, sfb,
                        (kb > 0 || k > 0) ? 1u : 0u);
          mma_commit(&sh.empty[s]);
          if (j == 3 || kb == kblocks - 1) {
            mma_commit(&sh.sf_empty[slot]);
            ++grp;
          }
        }
        if (!ok) break;
        mma_commit(&sh.d_full);
      }
      // every MMA has completed before the tensor memory is released
      mma_commit(&sh.done);
      volatile int no_abort = 0;
      mbar_wait(&sh.done, 0, &no_abort, p.status);
    }
  } else if (warp < 6) {
    // ---------------- scale bytes (warps 2..5, run ahead across tiles) ----------------
    const int q = warp & 3, wi = warp - 2;
    const int kbs = kblocks;
    const int wtiles = (p.N + 127) >> 7;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    bool bad = false, clamped = false;
    int grp = 0;  // the CTA's group sequence number (ring slot and barrier parity)
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int m0, n0;
      tile_of(t, m0, n0);
      const int row = m0 + 32 * q + lane;
      const int wt0 = n0 >> 7;
      // scales of group g + 1 are loaded while group g is converted
      float nsa[4], nsw[2][4];
      auto load_group = [&](int g) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kb = 4 * g + j;
          nsa[j] = (kb < kbs && row < p.M) ? __ldg(p.sa + static_cast<int64_t>(row) * kbs + kb) : 0.0f;
#pragma unroll
          for (int h = 0; h < 2; ++h)
            nsw[h][j] =
                (kb < kbs && wt0 + h < wtiles) ? __ldg(p.sw + static_cast<int64_t>(wt0 + h) * kbs + kb) : 0.0f;
        }
      };
      load_group(0);
      bool stop = false;
      for (int g = 0; g < groups; ++g, ++grp) {
        const int slot = grp % SF_GROUPS, par = grp & 1;
        // the four K blocks' exponents of this row and of the tile's two weight tiles
        int ea[4], ew[2][4];
        bool za[4], zw[2][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ea[j] = 0;
          za[j] = !pow2_exponent(nsa[j], ea[j], bad);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            ew[h][j] = 0;
            zw[h][j] = !pow2_exponent(nsw[h][j], ew[h][j], bad);
          }
        }
        if (g + 1 < groups) load_group(g + 1);
        int lo[4], hi[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          lo[j] = __reduce_min_sync(0xFFFFFFFFu, za[j] ? kNone : ea[j]);
          hi[j] = __reduce_max_sync(0xFFFFFFFFu, za[j] ? -kNone : ea[j]);
        }
        // the ring slot is free once the MMAs of group grp - SF_GROUPS are
        // done; every writer warp reaches the barrier below whatever its wait
        // gave, and all of them leave together if any wait gave up
        if (grp >= SF_GROUPS) mbar_wait(&sh.sf_empty[slot], ((grp / SF_GROUPS) - 1) & 1, abort, p.status);
        if (lane == 0)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            sh.ext[par][wi][j][0] = lo[j];
            sh.ext[par][wi][j][1] = hi[j];
          }
        named_bar(1, 128);  // the four writer warps' exponent ranges are in
        if (*abort) {
          stop = true;
          break;
        }
        uint32_t wa = 0, wb[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int amin = kNone, amax = -kNone;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            amin = min(amin, sh.ext[par][w][j][0]);
            amax = max(amax, sh.ext[par][w][j][1]);
          }
          int wmin = kNone, wmax = -kNone;
#pragma unroll
          for (int h = 0; h < 2; ++h)
            if (!zw[h][j]) {
              wmin = min(wmin, ew[h][j]);
              wmax = max(wmax, ew[h][j]);
            }
          // shift t: ua = ea + 127 + t and uw = ew + 127 - t both in [0, 254]
          int tlo = -1000000, thi = 1000000;
          if (amin != kNone) {
            tlo = max(tlo, -127 - amin);
            thi = min(thi, 127 - amax);
          }
          if (wmin != kNone) {
            tlo = max(tlo, wmax - 127);
            thi = min(thi, wmin + 127);
          }
          int tshift = min(max(0, tlo), thi);
          if (tlo > thi) {
            tshift = min(max(0, tlo), 254);  // no exact split: bytes are clamped
            clamped = true;
          }
          const uint32_t ua = za[j] ? 0u : static_cast<uint32_t>(min(max(ea[j] + 127 + tshift, 0), 254));
          wa |= ua << (8 * j);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t uw = zw[h][j] ? 0u : static_cast<uint32_t>(min(max(ew[h][j] + 127 - tshift, 0), 254));
            wb[h] |= uw << (8 * j);
          }
        }
        // A: this quarter's column holds its 32 rows (the other quarters'
        // columns at these lanes are never read); B: eight columns of 32
        // weight rows each, the first four from weight tile wt0, the last four
        // from wt0 + 1
        const uint32_t col = tmem + lane_addr + SF_COL0 + SF_STRIDE * slot;
        const uint32_t va[4] = {wa, wa, wa, wa};
        const uint32_t vb[8] = {wb[0], wb[0], wb[0], wb[0], wb[1], wb[1], wb[1], wb[1]};
        tmem_st4(col, va);
        tmem_st8(col + 8, vb);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.sf_full[slot]);
      }
      if (stop) break;
    }
    if (bad || clamped) flag(p.status, QRR_DEV_SCALE_RANGE);
  } else {
    // ---------------- epilogue (warps 6..13) ----------------
    // The accumulator is read out first (its columns packed to bf16 in
    // registers) and handed back to the MMA warp, then stored, so the next
    // tile's MMAs overlap the stores.
    const int q = warp & 3, h = (warp - 6) >> 2;
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    int tiles_done = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++tiles_done) {
      int m0, n0;
      tile_of(t, m0, n0);
      const int row = m0 + 32 * q + lane;
      const int col0 = n0 + 128 * h;
      if (!mbar_wait(&sh.d_full, tiles_done & 1, abort, p.status) || *abort) break;
      tc_fence_after();
      uint32_t packed[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_addr + 128 * h + 32 * c, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          packed[16 * c + i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.d_empty);
      if (row < p.M && col0 < p.N) {
        uint4* dst = reinterpret_cast<uint4*>(p.y + static_cast<int64_t>(row) * p.N + col0);
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

cudaError_t launch_fp8_gemm_mx(const Fp8GemmArgs& a, int32_t* status, cudaStream_t stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(fp8_gemm_mx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  const int64_t tiles = ((a.N + BN - 1) / BN) * ((a.M + BM - 1) / BM);
  int dev = 0, sms = kSMs;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const unsigned grid = static_cast<unsigned>(tiles < sms ? tiles : sms);
  fp8_gemm_mx_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qrr

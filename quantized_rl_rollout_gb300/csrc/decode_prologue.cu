// Decode prologue of the W4A16 + LoRA linear (at most 64 tokens).
//
// The GEMM takes an image of x: above 8 tokens its f16 operand, which needs
// for each token m the power of two p_m with max_k |x[m, k]| 2^-p_m in
// [2^14, 2^15) and x16 = f16(x 2^-p_m); up to 8 tokens the E2M1 digit planes
// of x 2^-p_m with max |x| 2^-p_m in (3, 6] (write_planes8 below).  The
// adapter path needs
//   t'[m, 2j] = bf16(v), t'[m, 2j+1] = bf16(v - bf16(v)),
//   v = (alpha / r) t[m, j] / g,  t = x A^T,  g = s_t (or 1 when s_t = 0)
// ("NVIDIA and MIT Collaborate on QeRL", Key Features: the adapter runs in
// higher precision beside the 4-bit weights).  Both are reductions over K.
// Each layer gets one cluster of ks CTAs (16, or 8 where the device cannot
// hold a cluster of 16 per layer at once), CTA c owning the c-th K slice:
//   all warps   copy its slice of x ([XR x 64] per 64-wide step) and of A
//               ([R x 64]) into shared memory in the 128-byte-swizzled layout,
//               every copy in flight at once (one round unless the slice is
//               long)
//   warp 1      MMA: t_c = x_c A_c^T, tcgen05 kind::f16, M128 x R per step;
//               the 128-row x operand reads past the XR staged rows into
//               whatever follows in shared memory, which only reaches
//               accumulator rows that are never read
//   warps 2..5  per-token max |x| over the staged tiles; then (warps 4 and 5,
//               TMEM lane quarters 0 and 1) t_c from TMEM into shared memory
// and then, across the cluster through distributed shared memory, every CTA
// takes the token maxima over all slices and writes the image of its own
// slice, and the t outputs are divided among the CTAs, each summing the ks
// slice partials in slice order (the result does not depend on timing).  No
// global partials, tickets or fences: one pass over x and A.  The launch
// also clears the split-K tile counters of the GEMM that follows, which reads
// them only after this grid has completed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

// Development builds (-DQRR_TRACE_BUILD) record global-timer stamps of each
// CTA's phases; ordinary builds compile them away.
#ifdef QRR_TRACE_BUILD
__device__ unsigned long long qrr_dtrace_buf[128][16];
#define QRR_DSTAMP(ev)                                                  \
  do {                                                                  \
    unsigned long long t_;                                              \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));              \
    if (blockIdx.x < 128) qrr_dtrace_buf[blockIdx.x][ev] = t_;           \
  } while (0)
#else
#define QRR_DSTAMP(ev) \
  do {                 \
  } while (0)
#endif

namespace {

constexpr int kKsMax = 16;  // CTAs per cluster = K slices per layer (16: a non-portable cluster size)
constexpr int kThreads = 384;  // 12 warps: roles in warps 0..5, all share the copies and conversions
constexpr int kMaxXR = 64;
constexpr int kMaxR = 64;
constexpr int kMaxStages = 32;
constexpr int kMmaSlack = 128 * 128;   // the x operand spans 128 rows of 128 bytes
constexpr int kDynMax = 192 * 1024;    // dynamic shared memory, alignment slack included
// At least this much dynamic shared memory per CTA, so that no CTA of this
// grid shares an SM with a CTA of the GEMM launched after it: that GEMM
// holds all 512 TMEM columns of its SM until it ends and waits for this grid,
// so a CTA of this grid that had to allocate TMEM beside it would never run.
constexpr int kDynMin = 64 * 1024;

struct ProCtl {
  uint64_t round_done;  // a round's MMAs are done (the next round may overwrite its tiles)
  uint64_t d_full;
  uint32_t tmem;
  int abort;
  uint32_t amax_part[kMaxXR];  // max |x| bits of each token row over this slice
  uint32_t amax[kMaxXR];       // ... over all slices
  int pexp[kMaxXR];
  float tpart[kMaxXR * kMaxR];  // this slice's t, [XR][R]
};

// Loads from a peer CTA's shared memory.  They are read only after the
// cluster barrier that follows the last write (itself a compiler memory
// barrier), so they need none of their own and can all be in flight at once.
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// The power of two p with amax 2^-p in [2^14, 2^15) for max |x| bits `mx`
// (0 for an all-zero row).
__device__ __forceinline__ int pexp_of(uint32_t mx) {
  if (mx == 0u) return 0;
  int e;
  frexpf(bf16bits_to_f32(mx), &e);  // amax = f 2^e, 0.5 <= f < 1
  return e - 15;
}

// For the E2M1 digit planes: the power of two e with max |x| 2^-e in
// (3, 6], so that every scaled value lies on or inside the E2M1 range.
__device__ __forceinline__ int pexp_planes(uint32_t mx) {
  if (mx == 0u) return 0;
  int e;
  const float f = frexpf(bf16bits_to_f32(mx), &e);  // amax = f 2^e, 0.5 <= f < 1
  return f > 0.75f ? e - 2 : e - 3;
}

__device__ __forceinline__ int pexp_for(uint32_t mx, bool planes) { return planes ? pexp_planes(mx) : pexp_of(mx); }

// The digit planes of 8 consecutive values of one token (one 16-byte bf16
// vector): word p of plane p at dst[p * stride] (stride in words), eight
// E2M1 codes, element i in nibble i.  r starts as x 2^-e (|r| <= 6); each
// plane takes d = e2m1_rne(r) and leaves r = (r - d) 6, which stays within
// [-6, 6] because |r - d| <= 1 on the E2M1 grid.
__device__ __forceinline__ void write_planes8(uint4 xv, const Pow2Scaler& sc, uint32_t* dst, int64_t stride) {
  float r[8];
  const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    r[2 * u] = sc(bf16_lo(w[u]));
    r[2 * u + 1] = sc(bf16_hi(w[u]));
  }
#pragma unroll
  for (int pl = 0; pl < kXPlanes; ++pl) {
    const uint32_t code = cvt_e2m1x8(r);
    dst[pl * stride] = code;
    if (pl + 1 < kXPlanes) {
      uint32_t h2[4];  // the digits' values as f16 pairs (exact)
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
          "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
          : "=r"(h2[0]), "=r"(h2[1]), "=r"(h2[2]), "=r"(h2[3])
          : "r"(code));
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        // (r - d) 6 for both halves on the paired fp32 pipe (each half one
        // correctly rounded fp32 subtraction, then one multiplication)
        const float2 d = __half22float2(*reinterpret_cast<const __half2*>(&h2[b]));
        asm("{\n\t.reg .b64 rr, dd, six;\n\t"
            "mov.b64 rr, {%0, %1};\n\tmov.b64 dd, {%2, %3};\n\tmov.b64 six, {%4, %4};\n\t"
            "sub.rn.f32x2 rr, rr, dd;\n\tmul.rn.f32x2 rr, rr, six;\n\tmov.b64 {%0, %1}, rr;\n\t}"
            : "+f"(r[2 * b]), "+f"(r[2 * b + 1])
            : "f"(d.x), "f"(d.y), "f"(6.0f));
      }
    }
  }
}

// t'[m, 2j], t'[m, 2j+1] of one rank: v = (scale t / g) 2^-p_m as (high,
// low) bf16.  The factor 2^-p_m is the one the GEMM's accumulator carries
// for token m (its f16 image of x is scaled by it); multiplying by a power
// of two is exact, so this equals scaling the (high, low) pair afterwards.
__device__ __forceinline__ void write_tprime(__nv_bfloat16* trow, int jj, float scale, float t, float g, int pexp) {
  const float v = Pow2Scaler(pexp)(__fdiv_rn(scale * t, g));
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
  trow[2 * jj] = hi;
  trow[2 * jj + 1] = lo;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) decode_prologue_kernel(const __grid_constant__ DecodeProBatch b) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ ProCtl sh;
  uint8_t* const xs = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int ks = b.ks;
  const DecodeProLayer& L = b.l[blockIdx.x / ks];
  const int rank = static_cast<int>(cluster_rank());
  // the GEMM may be scheduled now: it streams its weights while this runs
  // and waits for this grid before it reads x16, p and t'
  griddep_launch_dependents();
  if (tid == 0) QRR_DSTAMP(0);
  const int XR = b.xr, S = b.stages;
  const int M = L.M, K = L.K, r = L.r, R = L.R;
  uint8_t* const as = xs + S * XR * 128;  // A tiles after all x tiles
  const int kc_all = K / 64;
  const int spc = (kc_all + ks - 1) / ks;
  const int k0 = rank * spc;  // first 64-wide step of this slice
  const int steps = max(0, min(spc, kc_all - k0));
  const bool lora = r > 0;
  const bool mma = lora && steps > 0;
  volatile int* abort = &sh.abort;
  const float st = lora ? *L.tensor_scale : 1.0f;  // read early: it is needed only at the end

  if (tid == 0) {
    mbar_init(&sh.round_done, 1);
    mbar_init(&sh.d_full, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  // The slice moves in rounds of up to S steps (one round unless the slice
  // is long): every thread copies its share of the round's 16-byte pieces
  // straight into the 128-byte-swizzled layout the MMA reads (piece c of row
  // w at c ^ (w & 7)), rows past M (x) or r (A) as zeros, all copies in
  // flight at once.
  const int et = tid - 64;                    // max warps: thread (row group, piece)
  const int piece = et & 7, row0 = et >> 3;   // rows row0 + 16 i
  uint32_t mx[4] = {0u, 0u, 0u, 0u};
  const uint16_t* const xg = L.x;
  const uint16_t* const ag = L.A;
  const int rows_step = XR + (lora ? R : 0);
  int round = 0;
  for (int c0 = 0; c0 < steps; c0 += S, ++round) {
    const int n = min(S, steps - c0);
    if (round > 0) {
      // the previous round's MMAs have read their tiles
      if (mma) (void)mbar_wait(&sh.round_done, (round - 1) & 1, abort, b.status);
      __syncthreads();
    }
    {
      // thread: 16-byte piece tid % 8 of rows tid / 8, tid / 8 + 24, ...
      const int pc = tid & 7;
      for (int row = tid >> 3; row < rows_step; row += kThreads / 8) {
        const bool is_x = row < XR;
        const int rr = is_x ? row : row - XR;
        const bool valid = is_x ? rr < M : rr < r;
        const uint16_t* src = (is_x ? xg : ag) + static_cast<int64_t>(valid ? rr : 0) * K + (k0 + c0) * 64 + pc * 8;
        uint8_t* dst = (is_x ? xs : as) + rr * 128 + ((pc ^ (rr & 7)) << 4);
        const int dstep = is_x ? XR * 128 : R * 128;
        for (int st = 0; st < n; ++st)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst + st * dstep)),
                       "l"(src + st * 64), "r"(valid ? 16 : 0)
                       : "memory");
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // the copies were made through the generic proxy; the MMA reads through
    // the async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (round == 0 && tid == 0) QRR_DSTAMP(1);
    if (warp == 1) {
      if (mma && elect_one()) {
        tc_fence_after();
        const uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, 128, static_cast<uint32_t>(R));
        for (int c = 0; c < n; ++c) {
          const uint32_t xa = smem_u32(xs + c * XR * 128), aa = smem_u32(as + c * R * 128);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16_ss(tmem, sw128_desc(xa + 32 * k), sw128_desc(aa + 32 * k), idesc,
                        (c0 + c > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(c0 + n < steps ? &sh.round_done : &sh.d_full);
      }
      __syncwarp();
    } else if (warp >= 2 && warp < 6) {
      // per-token max |x| over the round's tiles; the swizzle only permutes
      // pieces within a row, which a maximum ignores
      for (int c = 0; c < n; ++c) {
        const uint8_t* tile = xs + c * XR * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = row0 + 16 * i;
          if (row < XR) mx[i] = max(mx[i], absmax_bits8(*reinterpret_cast<const uint4*>(tile + row * 128 + piece * 16)));
        }
      }
    }
  }
  if (warp >= 2 && warp < 6) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mx[i] = max(mx[i], __shfl_xor_sync(0xFFFFFFFFu, mx[i], 1));
      mx[i] = max(mx[i], __shfl_xor_sync(0xFFFFFFFFu, mx[i], 2));
      mx[i] = max(mx[i], __shfl_xor_sync(0xFFFFFFFFu, mx[i], 4));
      const int row = row0 + 16 * i;
      if (piece == 0 && row < XR) sh.amax_part[row] = mx[i];
    }
    if (et == 0) QRR_DSTAMP(2);
    // t of this slice: the two warps on TMEM lane quarters 0 and 1 (tokens 0..63)
    if (lora && warp >= 4) {
      const int q = warp & 3;
      const int m = 32 * q + lane;
      bool have = mma && mbar_wait(&sh.d_full, 0, abort, b.status);
      have = __all_sync(0xFFFFFFFFu, have);
      if (warp == 4 && lane == 0) QRR_DSTAMP(3);
      if (have) tc_fence_after();
      for (int cc = 0; cc < R; cc += 16) {
        uint32_t v[16];
        if (have) {
          tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(cc), v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0u;
        }
        if (m < XR)
#pragma unroll
          for (int i = 0; i < 16; ++i) sh.tpart[m * R + cc + i] = __uint_as_float(v[i]);
      }
    }
  }
  if (warp == 1 && mma && elect_one()) {
    // the accumulator is complete (or abandoned) before TMEM is released
    volatile int no_abort = 0;
    mbar_wait(&sh.d_full, 0, &no_abort, b.status);
  }
  __syncwarp();
  cluster_sync();  // every slice's maxima and t partials are in place
  if (tid == 0) QRR_DSTAMP(4);

  // token maxima over all slices, and the pre-scale exponents
  for (int m = tid; m < M; m += kThreads) {
    uint32_t part[kKsMax];
#pragma unroll
    for (int rr = 0; rr < kKsMax; ++rr) part[rr] = rr < ks ? ld_cluster_u32(cluster_addr(&sh.amax_part[m], rr)) : 0u;
    uint32_t mx = 0u;
#pragma unroll
    for (int rr = 0; rr < kKsMax; ++rr) mx = max(mx, part[rr]);
    const int pe = pexp_for(mx, L.planes != nullptr);
    sh.pexp[m] = pe;
    if (rank == 0) {
      if (mx >= 0x7F80u) flag(b.status, QRR_DEV_NONFINITE);
      L.pexp[m] = pe;
    }
  }
  __syncthreads();
  if (tid == 0) QRR_DSTAMP(5);

  // f16 image (or digit planes) of this slice: from the staged tiles while
  // the ring held the whole slice, else from x again (an L2 hit: the tiles
  // were just loaded)
  {
    const int nvec = steps * 8;  // 16-byte vectors per token row of the slice
    const bool resident = steps <= S;  // one round: step c still sits in slot c
    __half* const x16 = L.x16;
    // element i = m nvec + v, stepped by kThreads without a division per step
    const int dm = nvec > 0 ? kThreads / nvec : 0, dv = kThreads - dm * nvec;
    int m = nvec > 0 ? tid / nvec : M, v = tid - m * nvec;
    for (; m < M; m += dm, v += dv) {
      if (v >= nvec) {
        v -= nvec;
        ++m;
        if (m >= M) break;
      }
      const int c = v >> 3, pc = v & 7;
      uint4 xv;
      if (resident)
        xv = *reinterpret_cast<const uint4*>(xs + c * XR * 128 + m * 128 + ((pc ^ (m & 7)) << 4));
      else
        xv = __ldg(reinterpret_cast<const uint4*>(xg + static_cast<int64_t>(m) * K + (k0 + c) * 64) + pc);
      const Pow2Scaler sc(sh.pexp[m]);
      if (L.planes != nullptr) {
        const int64_t stride = static_cast<int64_t>(L.ms) * (K / 8);  // words per plane
        write_planes8(xv, sc,
                      reinterpret_cast<uint32_t*>(L.planes) + static_cast<int64_t>(m) * (K / 8) + (k0 + c) * 8 + pc,
                      stride);
        continue;
      }
      const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t o[4];
      if (sc.f2 == 1.0f) {  // 2^-p a normal fp32 number: one exact multiply
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const __half2 h = __floats2half2_rn(__fmul_rn(bf16_lo(w[u]), sc.f1), __fmul_rn(bf16_hi(w[u]), sc.f1));
          o[u] = *reinterpret_cast<const uint32_t*>(&h);
        }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const __half2 h = __floats2half2_rn(sc(bf16_lo(w[u])), sc(bf16_hi(w[u])));
          o[u] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      *(reinterpret_cast<uint4*>(x16 + static_cast<int64_t>(m) * K + (k0 + c) * 64) + pc) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }

  if (tid == 0) QRR_DSTAMP(6);
  // t': the outputs divided among the cluster, each the slice partials
  // summed in slice order
  if (lora) {
    const float g = st > 0.0f ? st : 1.0f;
    const float lscale = L.lora_scale;
    __nv_bfloat16* const t = L.t;
    const int t_cols = L.t_cols;
    for (int idx = rank * kThreads + tid; idx < M * r; idx += ks * kThreads) {
      const int m = idx / r, jj = idx - m * r;
      float part[kKsMax];
#pragma unroll
      for (int rr = 0; rr < kKsMax; ++rr) part[rr] = rr < ks ? ld_cluster_f32(cluster_addr(&sh.tpart[m * R + jj], rr)) : 0.0f;
      float sum = 0.0f;
#pragma unroll
      for (int rr = 0; rr < kKsMax; ++rr) sum += part[rr];  // slice order; the slices past ks add 0
      write_tprime(t + static_cast<int64_t>(m) * t_cols, jj, lscale, sum, g, sh.pexp[m]);
    }
    const int pad = t_cols - 2 * r;
    for (int idx = rank * kThreads + tid; idx < M * pad; idx += ks * kThreads)
      t[static_cast<int64_t>(idx / pad) * t_cols + 2 * r + idx % pad] = __float2bfloat16_rn(0.0f);
  }

  if (tid == 0) QRR_DSTAMP(7);
  for (int w = static_cast<int>(blockIdx.x) * kThreads + tid; w < b.clear_words;
       w += static_cast<int>(gridDim.x) * kThreads)
    b.clear[w] = 0u;

  tc_fence_before();
  __syncwarp();
  cluster_sync();  // no CTA leaves while a peer may still read its shared memory
  if (tid == 0) QRR_DSTAMP(8);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
  if (tid == 0) QRR_DSTAMP(9);
}

// A single token (at most kSmallM): the same outputs on the CUDA cores, each
// from one pass over its data and a reduction inside one CTA, with every
// load of a thread in flight at once for K up to 16384 (one memory round
// trip; the tensor-core clusters above pay for TMA, TMEM and two cluster
// barriers, which a single token does not repay).
//   x CTAs, one per (layer, token): the row's max |x| (a block reduction),
//     then the row again (now from L1) into x16
//   t CTAs, one per (layer, 2 adapter ranks): thread i takes the 16-byte
//     vectors i, i + 512, ... of the 2 rows of A and of every token's x and
//     accumulates the 2 x M dot products in fp32; the 512 partial sums of
//     each output then meet in a fixed tree (warp shuffles, then the 16
//     warps in order), so the result does not depend on timing
constexpr int kSmallM = 1;
constexpr int kSmallThreads = 512;
constexpr int kRanksPerCta = 2;
// x CTAs per token row: one per 4096 values of the row (each takes the whole
// row's maximum, an L2 read, and writes the image of its own slice)
constexpr int kSliceVecs = 512;  // 16-byte vectors of a slice

__host__ __device__ constexpr int x_slices(int K) { return (K / 8 + kSliceVecs - 1) / kSliceVecs; }

// bf16 bits -> 8 fp32 values
__device__ __forceinline__ void unpack8_bf16(uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_lo(w[i]);
    f[2 * i + 1] = bf16_hi(w[i]);
  }
}

__global__ void __launch_bounds__(kSmallThreads) decode_prologue_small_kernel(const __grid_constant__ DecodeProBatch b) {
  __shared__ uint32_t red_u[kSmallThreads / 32];
  __shared__ float red_f[kSmallThreads / 32][kSmallM * kRanksPerCta];
  __shared__ uint32_t red_m[kSmallThreads / 32][kSmallM];
  griddep_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) QRR_DSTAMP(10);
  int j = 0;
  while (j + 1 < b.count && b.l[j + 1].first_cta <= static_cast<int>(blockIdx.x)) ++j;
  const DecodeProLayer& L = b.l[j];
  const int local = static_cast<int>(blockIdx.x) - L.first_cta;
  const int M = L.M, K = L.K, nv = K / 8;
  for (int w = static_cast<int>(blockIdx.x) * kSmallThreads + tid; w < b.clear_words;
       w += static_cast<int>(gridDim.x) * kSmallThreads)
    b.clear[w] = 0u;
  const int xs = x_slices(K);
  if (local < M * xs) {
    // ---- x image and p of token m, slice sl of its row ----
    const int m = local / xs, sl = local - m * xs;
    const int v0 = sl * kSliceVecs, v1 = min(nv, v0 + kSliceVecs);
    const uint4* xr = reinterpret_cast<const uint4*>(L.x + static_cast<int64_t>(m) * K);
    uint32_t mx = 0u;
#pragma unroll 8
    for (int v = tid; v < nv; v += kSmallThreads) mx = max(mx, absmax_bits8(__ldg(xr + v)));
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) red_u[warp] = mx;
    __syncthreads();
    mx = 0u;
#pragma unroll
    for (int w = 0; w < kSmallThreads / 32; ++w) mx = max(mx, red_u[w]);
    const int pe = pexp_for(mx, L.planes != nullptr);
    if (tid == 0 && sl == 0) {
      if (mx >= 0x7F80u) flag(b.status, QRR_DEV_NONFINITE);
      L.pexp[m] = pe;
    }
    const Pow2Scaler sc(pe);
    if (L.planes != nullptr) {
      uint32_t* const pw = reinterpret_cast<uint32_t*>(L.planes) + static_cast<int64_t>(m) * (K / 8);
      const int64_t stride = static_cast<int64_t>(L.ms) * (K / 8);
      for (int v = v0 + tid; v < v1; v += kSmallThreads) write_planes8(__ldg(xr + v), sc, pw + v, stride);
      if (tid == 0) QRR_DSTAMP(11);
      return;
    }
    uint4* x16 = reinterpret_cast<uint4*>(L.x16 + static_cast<int64_t>(m) * K);
    for (int v = v0 + tid; v < v1; v += kSmallThreads) {
      const uint4 xv = __ldg(xr + v);
      const uint32_t w[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t o[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const __half2 h = __floats2half2_rn(sc(bf16_lo(w[u])), sc(bf16_hi(w[u])));
        o[u] = *reinterpret_cast<const uint32_t*>(&h);
      }
      x16[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    return;
  }
  // ---- t of kRanksPerCta ranks, all tokens ----
  const int r = L.r, j0 = (local - M * xs) * kRanksPerCta;
  float acc[kSmallM][kRanksPerCta];
  uint32_t xmax[kSmallM];  // each token's max |x| (its p scales t')
#pragma unroll
  for (int mm = 0; mm < kSmallM; ++mm) {
    xmax[mm] = 0u;
#pragma unroll
    for (int jj = 0; jj < kRanksPerCta; ++jj) acc[mm][jj] = 0.0f;
  }
  const uint4* arow[kRanksPerCta];
#pragma unroll
  for (int jj = 0; jj < kRanksPerCta; ++jj)
    arow[jj] = reinterpret_cast<const uint4*>(L.A + static_cast<int64_t>(min(j0 + jj, r - 1)) * K);
  const uint4* xbase = reinterpret_cast<const uint4*>(L.x);
  // batches of kBatch vectors per thread, every load of a batch issued
  // before the first product
  constexpr int kBatch = 4;
  for (int v0 = tid; v0 < nv; v0 += kBatch * kSmallThreads) {
    uint4 av[kBatch][kRanksPerCta], xv[kBatch][kSmallM];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int v = v0 + b * kSmallThreads;
      const bool in = v < nv;
#pragma unroll
      for (int jj = 0; jj < kRanksPerCta; ++jj) av[b][jj] = in ? __ldg(arow[jj] + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int mm = 0; mm < kSmallM; ++mm)
        xv[b][mm] = (in && mm < M) ? __ldg(xbase + static_cast<int64_t>(mm) * nv + v) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      float a[kRanksPerCta][8];
#pragma unroll
      for (int jj = 0; jj < kRanksPerCta; ++jj) unpack8_bf16(av[b][jj], a[jj]);
#pragma unroll
      for (int mm = 0; mm < kSmallM; ++mm) {
        xmax[mm] = max(xmax[mm], absmax_bits8(xv[b][mm]));
        float xf[8];
        unpack8_bf16(xv[b][mm], xf);
#pragma unroll
        for (int jj = 0; jj < kRanksPerCta; ++jj)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[mm][jj] = fmaf(a[jj][e], xf[e], acc[mm][jj]);
      }
    }
  }
#pragma unroll
  for (int mm = 0; mm < kSmallM; ++mm)
#pragma unroll
    for (int jj = 0; jj < kRanksPerCta; ++jj) {
      float v = acc[mm][jj];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      if (lane == 0) red_f[warp][mm * kRanksPerCta + jj] = v;
    }
#pragma unroll
  for (int mm = 0; mm < kSmallM; ++mm) {
    const uint32_t v = __reduce_max_sync(0xFFFFFFFFu, xmax[mm]);
    if (lane == 0) red_m[warp][mm] = v;
  }
  __syncthreads();
  if (tid < M * kRanksPerCta) {
    const int mm = tid / kRanksPerCta, jj = tid % kRanksPerCta;
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kSmallThreads / 32; ++w) t += red_f[w][tid];
    uint32_t mx = 0u;
#pragma unroll
    for (int w = 0; w < kSmallThreads / 32; ++w) mx = max(mx, red_m[w][mm]);
    if (j0 + jj < r) {
      const float st = *L.tensor_scale;
      write_tprime(L.t + static_cast<int64_t>(mm) * L.t_cols, j0 + jj, L.lora_scale, t, st > 0.0f ? st : 1.0f,
                   pexp_for(mx, L.planes != nullptr));
    }
  }
  // the padding columns of t' past 2 r: the first t CTA of the layer
  if (j0 == 0) {
    const int pad = L.t_cols - 2 * r;
    for (int idx = tid; idx < M * pad; idx += kSmallThreads)
      L.t[static_cast<int64_t>(idx / pad) * L.t_cols + 2 * r + idx % pad] = __float2bfloat16_rn(0.0f);
  }
  if (tid == 0) QRR_DSTAMP(11);
}

namespace {

cudaLaunchConfig_t pro_config(int count, int ks, int dyn, cudaLaunchAttribute* la, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(count * ks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(dyn);
  cfg.stream = stream;
  la[0].id = cudaLaunchAttributeClusterDimension;
  la[0].val.clusterDim.x = static_cast<unsigned>(ks);
  la[0].val.clusterDim.y = 1;
  la[0].val.clusterDim.z = 1;
  cfg.attrs = la;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

// Clusters of 16 when the device can hold one cluster per layer of that size
// at once (then each CTA streams half as much of x and A), else of 8.
cudaError_t launch_decode_prologue(DecodeProBatch& b, cudaStream_t stream) {
  if (b.count == 0) return cudaSuccess;
  int M = 0, Rmax = 0;
  for (int j = 0; j < b.count; ++j) {
    const DecodeProLayer& L = b.l[j];
    M = L.M;
    if (L.M > kMaxXR || L.R > kMaxR || L.R % 16 != 0 || L.K % 64 != 0) return cudaErrorInvalidValue;
    Rmax = L.R > Rmax ? L.R : Rmax;
  }
  if (M <= kSmallM) {
    int ctas = 0;
    for (int j = 0; j < b.count; ++j) {
      DecodeProLayer& L = b.l[j];
      L.first_cta = ctas;
      ctas += L.M * x_slices(L.K) + (L.r + kRanksPerCta - 1) / kRanksPerCta;
    }
    decode_prologue_small_kernel<<<ctas, kSmallThreads, 0, stream>>>(b);
    return cudaGetLastError();
  }
  b.xr = (M + 7) / 8 * 8;
  static bool attr = false;
  static int big_clusters = 0;  // 16-CTA clusters co-resident at the largest shared-memory size
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynMax);
    if (e != cudaSuccess) return e;
    if (cudaFuncSetAttribute(decode_prologue_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchAttribute la[1];
      cudaLaunchConfig_t cfg = pro_config(1, kKsMax, kDynMax, la, stream);
      if (cudaOccupancyMaxActiveClusters(&big_clusters, decode_prologue_kernel, &cfg) != cudaSuccess) big_clusters = 0;
    }
    cudaGetLastError();  // a refused probe leaves no error behind
    attr = true;
  }
  b.ks = big_clusters >= b.count ? kKsMax : 8;
  int steps_max = 1;
  for (int j = 0; j < b.count; ++j) {
    const int spc = (b.l[j].K / 64 + b.ks - 1) / b.ks;
    steps_max = spc > steps_max ? spc : steps_max;
  }
  const int stage = (b.xr + Rmax) * 128;
  int stages = (kDynMax - 1024 - kMmaSlack) / stage;
  stages = stages < steps_max ? stages : steps_max;
  stages = stages < kMaxStages ? stages : kMaxStages;
  b.stages = stages;
  int dyn = 1024 + stages * stage + kMmaSlack;
  dyn = dyn > kDynMin ? dyn : kDynMin;
  cudaLaunchAttribute la[1];
  cudaLaunchConfig_t cfg = pro_config(b.count, b.ks, dyn, la, stream);
  return cudaLaunchKernelEx(&cfg, decode_prologue_kernel, b);
}

}  // namespace qrr

#ifdef QRR_TRACE_BUILD
extern "C" int qrr_dtrace_read(unsigned long long* host) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, qrr::qrr_dtrace_buf, sizeof(qrr::qrr_dtrace_buf)));
}
extern "C" int qrr_dtrace_clear(void) {
  static unsigned long long zeros[128 * 16] = {};
  return static_cast<int>(cudaMemcpyToSymbol(qrr::qrr_dtrace_buf, zeros, sizeof(zeros)));
}
#endif

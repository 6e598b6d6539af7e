// Quantizers: NVFP4 (tensor absmax sweep + encode sweep), blockwise FP8 for
// 1x128 activation blocks and 128x128 weight tiles, and the rounding probe.
//
// All of them are HBM-streaming kernels.  Each thread moves 16-byte vectors,
// consecutive threads touch consecutive vectors (coalesced), and grids are a
// multiple of the SM count with grid-stride loops.  NVFP4 and FP8-weight
// kernels take a batch of tensors ("jobs") so re-quantizing a whole layer set
// is two (NVFP4) or one (FP8) launch.
//
// NVFP4 layout and rule ("QeRL: Beyond Efficiency", abstract; standard NVFP4
// layout): s_t = amax/2688, s_b = e4m3(amax_b / (6 s_t)), d_b = e4m3(s_b) s_t,
// code = e2m1(x / d_b); every step one correctly-rounded fp32 operation.
// FP8 ("NVIDIA NeMo RL behaalt 48% ...", "De technische doorbraak"): E4M3
// codes with one scale per 1x128 activation block / 128x128 weight tile,
// s = amax/448 or the next power of two.
#include "quant.cuh"
#include "tc.cuh"

namespace qrr {

// ---------------------------------------------------------------------------
// NVFP4, both passes streamed through shared memory by bulk copies (TMA):
// one thread keeps kStreamStages chunks of kStreamChunk bytes in flight per
// CTA, two CTAs per SM, whatever the registers the arithmetic needs (loads
// into registers cap the bytes in flight by occupancy).  A chunk lies inside
// one tensor; chunk c of the launch is taken by CTA c mod grid.  The job table
// (chunk boundaries, pointers) sits in shared memory.

namespace {

constexpr int kStreamChunk = 16384;  // bytes: 8192 bf16, 512 NVFP4 blocks
constexpr int kStreamStages = 6;     // absmax: 2 CTAs per SM
// absmax with AQN noise: its arithmetic, not HBM, bounds it, so a shallower
// ring and more CTAs per SM (more warps to issue from: 607 -> 582 us for the
// 8B-class set against 6 stages at 2 CTAs per SM)
constexpr int kAqnAmaxStages = 2;
constexpr int kAqnAmaxPerSm = 6;
constexpr int kEncodeStages = 3;     // encode: 4 CTAs per SM (more warps for its arithmetic)
constexpr int kEncodeThreads = 256;  // encode: threads per CTA, each kStreamChunk / 32 / kEncodeThreads blocks a chunk
constexpr int kEncodeBlocksPerThread = kStreamChunk / 32 / kEncodeThreads;

struct StreamRing {
  uint64_t full[kStreamStages], empty[kStreamStages];
  int abort;
};

// Producer side, run by thread 0 before consuming step i: issue the load of
// the CTA's step i + kStreamStages - 1 once that ring slot has been consumed.
template <int S, typename ChunkSrc>
__device__ __forceinline__ bool stream_issue(StreamRing& r, uint8_t* ring, int64_t step, int64_t steps,
                                             const ChunkSrc& src_of, int32_t* status) {
  if (step >= steps) return true;
  const int s = static_cast<int>(step % S);
  const int64_t use = step / S;
  if (use > 0 && !mbar_wait(&r.empty[s], (use - 1) & 1, &r.abort, status)) return false;
  const void* src;
  uint32_t bytes;
  src_of(step, src, bytes);
  mbar_arrive_expect_tx(&r.full[s], bytes);
  bulk_load(ring + static_cast<size_t>(s) * kStreamChunk, src, bytes, &r.full[s]);
  return true;
}

}  // namespace

// NVFP4 pass 1: tensor absmax.  A block's absmax is the max of |bf16| bit
// patterns; `amax_bits[j]` must be zero before the launch.  Each warp keeps a
// running max over its chunks and publishes it with one atomic per tensor it
// leaves (same-address atomics serialize in L2).
//
// With AQN noise only the largest |W'| of a tensor matters, W' = bf16(W + t)
// with |t| <= T = fp32(sigma) * zmax.  Over a warp's share of a chunk, with M
// its largest |W|: the element holding M has |W'| >= L = bf16(fp32(M - T))
// (or 0), and an element has |W'| <= bf16(fp32(|W| + T)), both because
// rounding is monotone.  So only 8-value vectors whose largest |W| passes
// bf16(fp32(max + T)) >= L can hold the share's largest |W'|; the warp
// queues those and draws noise for them alone, exactly.  Non-finite input
// (M at or past the infinity pattern) takes every vector.
template <bool NOISE>
__global__ void __launch_bounds__(256, NOISE ? kAqnAmaxPerSm : 2) nvfp4_amax_kernel(const __grid_constant__ Nvfp4Batch batch) {
  constexpr int S = NOISE ? kAqnAmaxStages : kStreamStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  StreamRing& r = *reinterpret_cast<StreamRing*>(smem_raw + S * kStreamChunk);
  __shared__ int64_t s_first[kMaxJobs + 1];
  __shared__ int64_t s_bytes[kMaxJobs];
  __shared__ const uint8_t* s_src[kMaxJobs];
  __shared__ uint32_t s_tensor[kMaxJobs];
  constexpr int kVecPerThread = kStreamChunk / 16 / 256;
  __shared__ uint16_t s_queue[NOISE ? 8 : 1][NOISE ? 32 * kVecPerThread : 1];  // per warp: vectors to draw noise for
  const int count = batch.count;
  const int64_t chunks = batch.total_amax_chunks;
  const AqnParams& aqn = batch.aqn;  // read from the launch parameters
  const float tbound = __fmul_rn(aqn.sigma, aqn_zmax());  // bounds |fp32(sigma z)|
  for (int j = threadIdx.x; j < count; j += blockDim.x) {
    s_first[j] = batch.job[j].first_amax_chunk;
    s_bytes[j] = batch.job[j].N * batch.job[j].K * 2;
    s_src[j] = reinterpret_cast<const uint8_t*>(batch.job[j].W);
    s_tensor[j] = batch.job[j].tensor;
  }
  if (threadIdx.x == 0) {
    s_first[count] = chunks;
    for (int s = 0; s < S; ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], 8);  // one arrival per warp
    }
    r.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  uint32_t* const amax_bits = batch.amax_bits;
  int32_t* const status = batch.status;
  const int64_t steps = chunks > blockIdx.x ? (chunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  int jp = 0;  // producer's job cursor
  auto src_of = [&](int64_t step, const void*& src, uint32_t& bytes) {
    const int64_t c = blockIdx.x + step * gridDim.x;
    while (s_first[jp + 1] <= c) ++jp;
    const int64_t off = (c - s_first[jp]) * kStreamChunk;
    src = s_src[jp] + off;
    const int64_t left = s_bytes[jp] - off;
    bytes = static_cast<uint32_t>(left < kStreamChunk ? left : kStreamChunk);
  };
  if (threadIdx.x == 0)
    for (int64_t i = 0; i < S - 1; ++i) stream_issue<S>(r, ring, i, steps, src_of, status);
  int cur = -1, j = 0;
  uint32_t run = 0;
  auto publish = [&]() {
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, run);
    if ((threadIdx.x & 31) == 0 && m) {
      atomicMax(amax_bits + cur, m);
      if (m >= 0x7F80u) flag(status, QRR_DEV_NONFINITE);
    }
    run = 0;
  };
  for (int64_t i = 0; i < steps; ++i) {
    if (threadIdx.x == 0 && !stream_issue<S>(r, ring, i + S - 1, steps, src_of, status)) break;
    const int s = static_cast<int>(i % S);
    if (!mbar_wait(&r.full[s], (i / S) & 1, &r.abort, status)) break;
    const int64_t c = blockIdx.x + i * gridDim.x;
    while (s_first[j + 1] <= c) ++j;
    if (j != cur) {
      if (cur >= 0) publish();
      cur = j;
    }
    const int64_t left = s_bytes[j] - (c - s_first[j]) * kStreamChunk;
    const int nvec = static_cast<int>((left < kStreamChunk ? left : kStreamChunk) / 16);
    const uint4* v = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(s) * kStreamChunk);
    const int64_t e0 = (c - s_first[j]) * (kStreamChunk / 2);  // first element of the chunk
    if constexpr (!NOISE) {
#pragma unroll
      for (int u = 0; u < kVecPerThread; ++u) {
        const int e = u * 256 + threadIdx.x;
        if (e < nvec) run = max(run, absmax_bits8(v[e]));
      }
    } else {
      uint32_t vm[kVecPerThread], m = 0u;
#pragma unroll
      for (int u = 0; u < kVecPerThread; ++u) {
        const int e = u * 256 + threadIdx.x;
        vm[u] = e < nvec ? absmax_bits8(v[e]) : 0u;
        m = max(m, vm[u]);
      }
      const uint32_t M = __reduce_max_sync(0xFFFFFFFFu, m);
      const int lane = threadIdx.x & 31;
      uint16_t* const q = s_queue[threadIdx.x >> 5];
      int cnt = 0;
      const float lo = __fsub_rn(bf16bits_to_f32(M), tbound);
      const uint32_t L = lo > 0.0f ? static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) : 0u;
#pragma unroll
      for (int u = 0; u < kVecPerThread; ++u) {
        const int e = u * 256 + threadIdx.x;
        const uint32_t ub = static_cast<uint32_t>(
            __bfloat16_as_ushort(__float2bfloat16_rn(__fadd_rn(bf16bits_to_f32(vm[u]), tbound))));
        const bool cand = e < nvec && (M >= 0x7F80u || ub >= L);
        const uint32_t mask = __ballot_sync(0xFFFFFFFFu, cand);
        if (cand) q[cnt + __popc(mask & ((1u << lane) - 1u))] = static_cast<uint16_t>(e);
        cnt += __popc(mask);
      }
      __syncwarp();
      for (int i = lane; i < cnt; i += 32) {
        const int e = q[i];
        run = max(run, absmax_bits8(aqn_noisy8(v[e], e0 + 8 * e, s_tensor[j], aqn)));
      }
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[s]);
  }
  if (cur >= 0) publish();
  // every issued copy has landed before the CTA exits
  if (threadIdx.x == 0) {
    volatile int no_abort = 0;
    for (int64_t k = steps - 1; k >= 0 && k >= steps - S; --k)
      mbar_wait(&r.full[k % S], (k / S) & 1, &no_abort, status);
  }
}

// NVFP4 pass 2: encode.  Block b of a tensor (16 elements, K % 16 == 0) is
// elements [16b, 16b+16) of the flat row-major matrix; its codes are bytes
// [8b, 8b+8) and its scale is byte b.  256 threads, two blocks of a chunk
// each, four CTAs per SM with 3-stage rings: the encode is issue-bound, and
// two independent blocks per thread halve the per-chunk bookkeeping per
// block (measured: 221 -> 193 us for the 8B-class layer set against one
// block per thread in 512-thread CTAs).  The chunks run in the reverse of
// the absmax pass's order, so the first ones read what that pass read last,
// while it is still in L2.
template <bool NOISE>
__global__ void __launch_bounds__(kEncodeThreads, 4) nvfp4_encode_kernel(const __grid_constant__ Nvfp4Batch batch) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  StreamRing& r = *reinterpret_cast<StreamRing*>(smem_raw + kEncodeStages * kStreamChunk);
  __shared__ int64_t s_first[kMaxJobs + 1];
  __shared__ int64_t s_bytes[kMaxJobs];
  __shared__ const uint8_t* s_src[kMaxJobs];
  __shared__ uint8_t* s_codes[kMaxJobs];
  __shared__ uint8_t* s_scales[kMaxJobs];
  __shared__ float* s_ts[kMaxJobs];
  __shared__ float s_st[kMaxJobs];
  __shared__ SharedDivisor s_six[kMaxJobs];  // the per-tensor divisor 6 s_t of every block's absmax
  __shared__ uint32_t s_tensor[kMaxJobs];
  const int count = batch.count;
  const int64_t chunks = batch.total_encode_chunks;
  const AqnParams& aqn = batch.aqn;  // read from the launch parameters
  for (int j = threadIdx.x; j < count; j += blockDim.x) {
    s_tensor[j] = batch.job[j].tensor;
    s_first[j] = batch.job[j].first_encode_chunk;
    s_bytes[j] = batch.job[j].N * batch.job[j].K * 2;
    s_src[j] = reinterpret_cast<const uint8_t*>(batch.job[j].W);
    s_codes[j] = batch.job[j].codes;
    s_scales[j] = batch.job[j].scales;
    s_ts[j] = batch.job[j].tensor_scale;
    s_st[j] = __fdiv_rn(bf16bits_to_f32(batch.amax_bits[j]), 2688.0f);
    s_six[j] = SharedDivisor(__fmul_rn(6.0f, s_st[j]));
  }
  if (threadIdx.x == 0) {
    s_first[count] = chunks;
    for (int s = 0; s < kEncodeStages; ++s) {
      mbar_init(&r.full[s], 1);
      mbar_init(&r.empty[s], kEncodeThreads / 32);  // one arrival per warp
    }
    r.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  int32_t* const status = batch.status;
  const int64_t steps = chunks > blockIdx.x ? (chunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  int jp = count - 1;  // producer's job cursor (chunks shrink)
  auto chunk_of = [&](int64_t step) { return chunks - 1 - (blockIdx.x + step * gridDim.x); };
  auto src_of = [&](int64_t step, const void*& src, uint32_t& bytes) {
    const int64_t c = chunk_of(step);
    while (s_first[jp] > c) --jp;
    const int64_t off = (c - s_first[jp]) * kStreamChunk;
    src = s_src[jp] + off;
    const int64_t left = s_bytes[jp] - off;
    bytes = static_cast<uint32_t>(left < kStreamChunk ? left : kStreamChunk);
  };
  if (threadIdx.x == 0)
    for (int64_t i = 0; i < kEncodeStages - 1; ++i) stream_issue<kEncodeStages>(r, ring, i, steps, src_of, status);
  int j = count - 1;
  for (int64_t i = 0; i < steps; ++i) {
    if (threadIdx.x == 0 && !stream_issue<kEncodeStages>(r, ring, i + kEncodeStages - 1, steps, src_of, status)) break;
    const int s = static_cast<int>(i % kEncodeStages);
    const int64_t c = chunk_of(i);
    while (s_first[j] > c) --j;
    const float s_t = s_st[j];
    const int64_t nb = s_bytes[j] / 32;                    // blocks of the tensor
    const int64_t b0 = (c - s_first[j]) * (kStreamChunk / 32);  // first block of the chunk
    if (b0 == 0 && threadIdx.x == 0) *s_ts[j] = s_t;
    if (!mbar_wait(&r.full[s], (i / kEncodeStages) & 1, &r.abort, status)) break;
    const uint4* v = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(s) * kStreamChunk);
    uint4 xs0[kEncodeBlocksPerThread], xs1[kEncodeBlocksPerThread];
#pragma unroll
    for (int u = 0; u < kEncodeBlocksPerThread; ++u) {
      const int lb = u * kEncodeThreads + static_cast<int>(threadIdx.x);  // block within the chunk
      xs0[u] = v[2 * lb];
      xs1[u] = v[2 * lb + 1];
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&r.empty[s]);
#pragma unroll
    for (int u = 0; u < kEncodeBlocksPerThread; ++u) {
    const int64_t b = b0 + u * kEncodeThreads + threadIdx.x;
    if (b >= nb) continue;
    uint4 x0 = xs0[u], x1 = xs1[u];
    if constexpr (NOISE) {
      x0 = aqn_noisy8(x0, 16 * b, s_tensor[j], aqn);
      x1 = aqn_noisy8(x1, 16 * b + 8, s_tensor[j], aqn);
    }
    uint32_t sb = 0;
    uint2 packed = make_uint2(0u, 0u);
    if (s_t > 0.0f) {
      const float amax_b = bf16bits_to_f32(max(absmax_bits8(x0), absmax_bits8(x1)));
      sb = cvt_e4m3x2(s_six[j](amax_b), 0.0f) & 0xFFu;
      const float d = __fmul_rn(e4m3_to_f32_cvt(sb), s_t);
      if (d > 0.0f) {
        const SharedDivisor2 div(d);  // 16 quotients x / d, each correctly rounded
        const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float q[2][8];
        if (div.ok) {  // one test per block for the divisor's range
#pragma unroll
          for (int k = 0; k < 8; ++k)
            div.fast(bf16_lo(w[k]), bf16_hi(w[k]), q[k >> 2][2 * (k & 3)], q[k >> 2][2 * (k & 3) + 1]);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) div(bf16_lo(w[k]), bf16_hi(w[k]), q[k >> 2][2 * (k & 3)], q[k >> 2][2 * (k & 3) + 1]);
        }
        packed = make_uint2(cvt_e2m1x8(q[0]), cvt_e2m1x8(q[1]));
      }
    }
    reinterpret_cast<uint2*>(s_codes[j])[b] = packed;
    s_scales[j][b] = static_cast<uint8_t>(sb);
    }
  }
  if (threadIdx.x == 0) {
    volatile int no_abort = 0;
    for (int64_t k = steps - 1; k >= 0 && k >= steps - kEncodeStages; --k)
      mbar_wait(&r.full[k % kEncodeStages], (k / kEncodeStages) & 1, &no_abort, status);
  }
}

// ---------------------------------------------------------------------------
// FP8 activations, 1x128 blocks.  Thread i handles elements [8i, 8i+8) of the
// flat [M, K] matrix; 16 consecutive threads (a half warp) form one 128-block,
// whose flat index is also the index of its scale in [M, K/128].

__global__ void __launch_bounds__(256) fp8_a1x128_kernel(const uint16_t* __restrict__ x, int64_t nvec,
                                                        uint8_t* __restrict__ q, float* __restrict__ scales,
                                                        int mode, int32_t* status) {
  // U vectors per thread per step, all loads issued first: one 16-byte load
  // in flight per thread is too few bytes in flight per SM to cover HBM latency
  constexpr int U = 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * U;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * U; base < nvec; base += stride) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + u * 256 + threadIdx.x;
      v[u] = i < nvec ? __ldg(reinterpret_cast<const uint4*>(x) + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + u * 256 + threadIdx.x;
      // all 32 lanes shuffle; nvec is a multiple of 16, so a half warp (one
      // 128-block) is wholly live or wholly past the end
      uint32_t m = absmax_bits8(v[u]);
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      if (i >= nvec) continue;
      if (m >= 0x7F80u && (threadIdx.x & 15) == 0) flag(status, QRR_DEV_NONFINITE);
      const float amax = bf16bits_to_f32(m);
      const float v448 = __fdiv_rn(amax, 448.0f);
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t out[2] = {0u, 0u};
      float s = 0.0f;
      if (v448 > 0.0f) {
        if (mode == QRR_SCALE_FP32) {
          s = v448;
          const SharedDivisor2 div(s);
          if (div.ok) {  // one test per vector for the divisor's range
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float a, b;
              div.fast(bf16_lo(w[k]), bf16_hi(w[k]), a, b);
              out[k >> 1] |= cvt_e4m3x2(a, b) << (16 * (k & 1));
            }
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float a, b;
              div(bf16_lo(w[k]), bf16_hi(w[k]), a, b);
              out[k >> 1] |= cvt_e4m3x2(a, b) << (16 * (k & 1));
            }
          }
        } else {
          const int e = pow2_ceil_exp(v448);
          s = pow2_from_exp(e);
          const Pow2Scaler sc(e);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            out[k >> 1] |= cvt_e4m3x2(sc(bf16_lo(w[k])), sc(bf16_hi(w[k]))) << (16 * (k & 1));
        }
      }
      reinterpret_cast<uint2*>(q)[i] = make_uint2(out[0], out[1]);
      if ((threadIdx.x & 15) == 0) scales[i >> 4] = s;
    }
  }
}

// ---------------------------------------------------------------------------
// FP8 weights, 128x128 tiles.  One CTA (256 threads) per tile: thread t holds
// row (u * 16 + t / 16), 16-byte column chunk t % 16, for u = 0..7 (a warp
// reads two full 256-byte tile rows), so the tile's absmax is reduced in
// registers, then encoded without re-reading HBM.

template <bool NOISE>
__global__ void __launch_bounds__(256) fp8_w128_kernel(const __grid_constant__ Fp8WBatch batch) {
  __shared__ uint32_t warp_max[8];
  __shared__ int64_t s_first[kMaxJobs + 1];  // job table in shared memory (see the NVFP4 kernels)
  const int count = batch.count;
  const int64_t total = batch.total_tiles;
  for (int j = threadIdx.x; j < count; j += blockDim.x) s_first[j] = batch.job[j].first_tile;
  if (threadIdx.x == 0) s_first[count] = total;
  __syncthreads();
  const int mode = batch.mode;
  int j = 0;
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    while (s_first[j + 1] <= t) ++j;  // tiles only grow
    const int64_t N = batch.job[j].N, K = batch.job[j].K;
    const uint16_t* const W = batch.job[j].W;
    uint8_t* const qout = batch.job[j].q;
    float* const scales = batch.job[j].scales;
    const int64_t local = t - s_first[j];
    const int64_t kt = K / 128;
    const int64_t tr = local / kt, tc = local % kt;
    const int64_t row0 = tr * 128;
    const int cchunk = threadIdx.x & 15;
    uint4 v[8];
    uint32_t m = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t row = row0 + u * 16 + (threadIdx.x >> 4);
      if (row < N) {
        v[u] = __ldg(reinterpret_cast<const uint4*>(W + row * K + tc * 128) + cchunk);
        if constexpr (NOISE) v[u] = aqn_noisy8(v[u], row * K + tc * 128 + 8 * cchunk, batch.job[j].tensor, batch.aqn);
        m = max(m, absmax_bits8(v[u]));
      } else {
        v[u] = make_uint4(0, 0, 0, 0);
      }
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
    __syncthreads();
    m = warp_max[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = max(m, warp_max[w]);
    __syncthreads();  // warp_max is reused by the next tile
    if (m >= 0x7F80u && threadIdx.x == 0) flag(batch.status, QRR_DEV_NONFINITE);
    const float v448 = __fdiv_rn(bf16bits_to_f32(m), 448.0f);
    float s = 0.0f;
    int e = 0;
    if (v448 > 0.0f) {
      if (mode == QRR_SCALE_FP32) {
        s = v448;
      } else {
        e = pow2_ceil_exp(v448);
        s = pow2_from_exp(e);
      }
    }
    if (threadIdx.x == 0) scales[tr * kt + tc] = s;
    const Pow2Scaler sc(e);
    const SharedDivisor2 div(s > 0.0f ? s : 1.0f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t row = row0 + u * 16 + (threadIdx.x >> 4);
      if (row >= N) continue;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t out[2] = {0u, 0u};
      if (s > 0.0f) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float a, b;
          if (mode == QRR_SCALE_FP32) {
            div(bf16_lo(w[k]), bf16_hi(w[k]), a, b);
          } else {
            a = sc(bf16_lo(w[k]));
            b = sc(bf16_hi(w[k]));
          }
          out[k >> 1] |= cvt_e4m3x2(a, b) << (16 * (k & 1));
        }
      }
      reinterpret_cast<uint2*>(qout + row * K + tc * 128)[cchunk] = make_uint2(out[0], out[1]);
    }
  }
}

// ---------------------------------------------------------------------------
// Rounding probe: the same cvt primitives the quantizers use.
__global__ void round_probe_kernel(const float* __restrict__ in, int64_t n, int fmt, uint8_t* __restrict__ out) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float v = in[i];
    out[i] = static_cast<uint8_t>(fmt == 0 ? (cvt_e2m1x2(v, 0.0f) & 0xFu) : (cvt_e4m3x2(v, 0.0f) & 0xFFu));
  }
}

// ---------------------------------------------------------------------------
// Host launchers.

int grid_for(int64_t work_units, int per_sm) {
  int dev = 0, sms = kSMs;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  return static_cast<int>(work_units < cap ? (work_units > 0 ? work_units : 1) : cap);
}

constexpr int kNvfp4Chunk = kStreamChunk;
constexpr int kNvfp4Smem = kStreamStages * kStreamChunk + static_cast<int>(sizeof(StreamRing));
constexpr int kAqnAmaxSmem = kAqnAmaxStages * kStreamChunk + static_cast<int>(sizeof(StreamRing));
constexpr int kEncodeSmem = kEncodeStages * kStreamChunk + static_cast<int>(sizeof(StreamRing));

cudaError_t launch_nvfp4(Nvfp4Batch& batch, cudaStream_t stream) {
  int64_t amax_chunks = 0, enc_chunks = 0;
  for (int j = 0; j < batch.count; ++j) {
    Nvfp4Job& job = batch.job[j];
    job.first_amax_chunk = amax_chunks;
    job.first_encode_chunk = enc_chunks;
    const int64_t bytes = job.N * job.K * 2;
    amax_chunks += (bytes + kNvfp4Chunk - 1) / kNvfp4Chunk;
    // every tensor gets at least one encode chunk: its first thread writes s_t
    enc_chunks += std::max<int64_t>(1, (bytes + kNvfp4Chunk - 1) / kNvfp4Chunk);
  }
  batch.total_amax_chunks = amax_chunks;
  batch.total_encode_chunks = enc_chunks;
  cudaError_t err = cudaMemsetAsync(batch.amax_bits, 0, sizeof(uint32_t) * batch.count, stream);
  if (err != cudaSuccess) return err;
  static bool attr = false;
  if (!attr) {
    err = cudaFuncSetAttribute(nvfp4_amax_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kNvfp4Smem);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(nvfp4_amax_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAqnAmaxSmem);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(nvfp4_encode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kEncodeSmem);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(nvfp4_encode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kEncodeSmem);
    if (err != cudaSuccess) return err;
    attr = true;
  }
  // sigma 0 adds exactly nothing (W + 0 z = W), so it takes the plain kernels
  if (batch.aqn.sigma != 0.0f) {
    if (amax_chunks > 0)
      nvfp4_amax_kernel<true><<<grid_for(amax_chunks, kAqnAmaxPerSm), 256, kAqnAmaxSmem, stream>>>(batch);
    nvfp4_encode_kernel<true><<<grid_for(enc_chunks, 4), kEncodeThreads, kEncodeSmem, stream>>>(batch);
  } else {
    if (amax_chunks > 0) nvfp4_amax_kernel<false><<<grid_for(amax_chunks, 2), 256, kNvfp4Smem, stream>>>(batch);
    nvfp4_encode_kernel<false><<<grid_for(enc_chunks, 4), kEncodeThreads, kEncodeSmem, stream>>>(batch);
  }
  return cudaGetLastError();
}

cudaError_t launch_fp8_a1x128(const void* x, int64_t M, int64_t K, uint8_t* q, float* scales, int mode,
                              int32_t* status, cudaStream_t stream) {
  const int64_t nvec = M * K / 8;
  if (nvec == 0) return cudaSuccess;
  // 8 CTAs per SM of which 5 are resident at once (48 registers): the extra
  // ones start as the first finish, which measured faster on these short
  // launches than one wave of 5 (129 against 138 us for the 8B-class set)
  fp8_a1x128_kernel<<<grid_for((nvec + 1023) / 1024, 8), 256, 0, stream>>>(static_cast<const uint16_t*>(x), nvec, q,
                                                                            scales, mode, status);
  return cudaGetLastError();
}

cudaError_t launch_fp8_w128(Fp8WBatch& batch, cudaStream_t stream) {
  int64_t tiles = 0;
  for (int j = 0; j < batch.count; ++j) {
    batch.job[j].first_tile = tiles;
    tiles += ((batch.job[j].N + 127) / 128) * (batch.job[j].K / 128);
  }
  batch.total_tiles = tiles;
  if (tiles == 0) return cudaSuccess;
  // one wave of persistent CTAs: as many per SM as the kernel's registers
  // allow (a grid past that leaves a second, partial wave to run every CTA's
  // whole share of tiles after the first)
  static int per_sm[2] = {0, 0};
  const int nz = batch.aqn.sigma != 0.0f ? 1 : 0;
  if (per_sm[nz] == 0) {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm[nz], nz ? fp8_w128_kernel<true> : fp8_w128_kernel<false>, 256, 0);
    if (e != cudaSuccess) return e;
    if (per_sm[nz] < 1) per_sm[nz] = 1;
  }
  if (nz)
    fp8_w128_kernel<true><<<grid_for(tiles, per_sm[nz]), 256, 0, stream>>>(batch);
  else
    fp8_w128_kernel<false><<<grid_for(tiles, per_sm[nz]), 256, 0, stream>>>(batch);
  return cudaGetLastError();
}

__global__ void aqn_noise_probe_kernel(float* __restrict__ out, int64_t n, int64_t start, uint32_t tensor,
                                       const __grid_constant__ AqnParams a) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = start + i;
    uint32_t r[4];
    aqn_words(static_cast<uint64_t>(e) >> 2, tensor, a, r);
    out[i] = aqn_z(r[e & 3]);
  }
}

cudaError_t launch_aqn_noise_probe(float* out, int64_t n, int64_t start, uint32_t tensor, const AqnParams& a,
                                   cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  aqn_noise_probe_kernel<<<grid_for((n + 255) / 256, 8), 256, 0, stream>>>(out, n, start, tensor, a);
  return cudaGetLastError();
}

cudaError_t launch_round_probe(const float* in, int64_t n, int fmt, uint8_t* out, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  round_probe_kernel<<<grid_for((n + 255) / 256, 8), 256, 0, stream>>>(in, n, fmt, out);
  return cudaGetLastError();
}

}  // namespace qrr

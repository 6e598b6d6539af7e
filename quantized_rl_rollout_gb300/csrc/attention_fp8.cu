// Decode attention over an FP8 (E4M3) key/value cache, and the append of a
// decode step's keys and values to that cache.
//
// ("NVIDIA NeMo RL behaalt 48% ...", section "Praktische prestatiewinsten":
// FP8 extended to the KV cache and the attention operations; section "De
// technische doorbraak": activations in 1x128 E4M3 blocks.)  Each cached key
// or value row (one token, one KV head, 128 values) is E4M3 codes with one
// fp32 scale, the 1x128 activation rule; query head h reads KV head
// h / (Hq / Hkv); o = softmax(q . K^T / sqrt(128)) . V.
//
// Layout: caches [B][Hkv][Lmax][128] bytes, scales [B][Hkv][Lmax] fp32 (a
// sequence's rows of one KV head are contiguous), q and o [B][Hq][128] bf16.
//
// Decode attention reads every cached byte once and does G = Hq / Hkv
// multiply-adds per byte, so it is HBM-bound; it runs on the CUDA cores in
// fp32 (the E4M3 codes convert exactly).  The scores take each key value as
// f16 into mixed-precision FMAs (f16 x f16 products are exact in fp32)
// against the query scaled by a power of two into f16, which leaves out one
// conversion per key value, the most frequent instruction of the kernel.  Split over the sequence: a CTA
// takes 512 tokens of one (sequence, KV head), streams their key and value
// rows and scales through shared memory in 64-token chunks by bulk copies
// (two in flight), and writes a partial (max, sum, unnormalized output) per
// query head of the group; a second kernel merges the partials in split
// order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "linear.cuh"
#include "quant.cuh"
#include "tc.cuh"

namespace qrr {

namespace {

constexpr int D = 128;
constexpr int kThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// four E4M3 bytes -> four fp32 (exact)
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float (&f)[4]) {
  uint32_t lo, hi;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

// a += k.lo q.lo + k.hi q.hi for two f16 pairs: mixed-precision FMAs, whose
// f16 x f16 products are exact in fp32
__device__ __forceinline__ void fma_f16pair(float& a, uint32_t k2, uint32_t q2) {
  asm("{\n\t.reg .b16 kl, kh, ql, qh;\n\tmov.b32 {kl, kh}, %1;\n\tmov.b32 {ql, qh}, %2;\n\t"
      "fma.rn.f32.f16 %0, kl, ql, %0;\n\tfma.rn.f32.f16 %0, kh, qh, %0;\n\t}"
      : "+f"(a)
      : "r"(k2), "r"(q2));
}

// four E4M3 bytes -> two f16 pairs (bytes 0,1 and 2,3; exact)
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

constexpr int CH = 64;      // tokens per pipeline chunk
// chunks in flight: two leave room for six CTAs per SM (the per-warp output
// buffer shares the ring's space), and the warps of six CTAs cover the copy
// latency better than a third chunk of three or four CTAs did (136 against
// 147 and 163 us for 64 sequences)
constexpr int NST = 2;
constexpr int TSPLIT = 512; // tokens per CTA

template <int G>
struct AttnShared {
  union {
    struct {
      uint8_t k[NST][CH * D];  // 8 KB per chunk
      uint8_t v[NST][CH * D];
    } ring;
    // per-warp outputs, merged at the end: written only after the last
    // chunk's barrier, when no warp reads the ring and no copy is in flight
    float o[4][G][D];
  } u;
  float ks[NST][CH], vs[NST][CH];
  float p[CH][G];   // this chunk's softmax numerators times the value row scale
  float red[4][G];  // per-warp partial max / sum
  uint64_t full[NST], empty[NST];
  int abort;
};
}  // namespace

// ---------------------------------------------------------------------------
// Append one decode step's key and value rows: row (b, g) of k_new / v_new
// (bf16 [B][Hkv][128]) is quantized by the 1x128 rule and written at slot
// pos[b] of the caches.  One warp per row, lane = 4 values.
__global__ void kv_append_fp8_kernel(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new, int B,
                                     int Hkv, const int32_t* __restrict__ pos, int Lmax, uint8_t* __restrict__ kc,
                                     float* __restrict__ ksc, uint8_t* __restrict__ vc, float* __restrict__ vsc,
                                     int mode, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);  // over 2 * B * Hkv
  if (row >= 2 * B * Hkv) return;
  const int kind = row / (B * Hkv), bg = row % (B * Hkv), b = bg / Hkv;
  const int p = __ldg(pos + b);
  if (p < 0 || p >= Lmax) {
    if (lane == 0) flag(status, QRR_DEV_BAD_INDEX);
    return;
  }
  const uint16_t* src = (kind ? v_new : k_new) + static_cast<int64_t>(bg) * D;
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(src) + lane);
  uint32_t m = max(max(w.x & 0x7FFFu, w.x >> 16 & 0x7FFFu), max(w.y & 0x7FFFu, w.y >> 16 & 0x7FFFu));
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if (m >= 0x7F80u && lane == 0) flag(status, QRR_DEV_NONFINITE);
  const float v448 = __fdiv_rn(bf16bits_to_f32(m), 448.0f);
  uint32_t out = 0u;
  float s = 0.0f;
  if (v448 > 0.0f) {
    float a0, a1, a2, a3;
    if (mode == QRR_SCALE_FP32) {
      s = v448;
      const SharedDivisor2 div(s);
      div(bf16_lo(w.x), bf16_hi(w.x), a0, a1);
      div(bf16_lo(w.y), bf16_hi(w.y), a2, a3);
    } else {
      const int e = pow2_ceil_exp(v448);
      s = pow2_from_exp(e);
      const Pow2Scaler sc(e);
      a0 = sc(bf16_lo(w.x));
      a1 = sc(bf16_hi(w.x));
      a2 = sc(bf16_lo(w.y));
      a3 = sc(bf16_hi(w.y));
    }
    out = cvt_e4m3x2(a0, a1) | (cvt_e4m3x2(a2, a3) << 16);
  }
  const int64_t slot = static_cast<int64_t>(bg) * Lmax + p;
  reinterpret_cast<uint32_t*>((kind ? vc : kc) + slot * D)[lane] = out;
  if (lane == 0) (kind ? vsc : ksc)[slot] = s;
}

// ---------------------------------------------------------------------------
// Partial attention of one (sequence b, KV head g, split s) for the G query
// heads of the group: part_m / part_l [.., G] (base-2 max, sum) and part_o
// [.., G, 128] (unnormalized).  The split's tokens stream through a ring of
// 64-token chunks (key rows, value rows and their scales by bulk copies);
// each chunk updates a running max, sum and output (online softmax), so the
// loads of later chunks overlap the arithmetic of earlier ones.
template <int G>
__global__ void __launch_bounds__(kThreads) attn_decode_fp8_kernel(
    const uint16_t* __restrict__ q, const uint8_t* __restrict__ kc, const float* __restrict__ ksc,
    const uint8_t* __restrict__ vc, const float* __restrict__ vsc, const int32_t* __restrict__ lens, int Hkv, int Lmax,
    int splits, float* __restrict__ part_m, float* __restrict__ part_l, float* __restrict__ part_o,
    int32_t* status) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  AttnShared<G>& sh = *reinterpret_cast<AttnShared<G>*>(smem_raw);
  // q 2^-e_h in f16 (e_h: head h's power of two that brings max |q| into
  // [2^14, 2^15), exact for bf16 values) as [16-value piece][value pair]
  // [head] f16 pairs, each piece's row padded by 4 words: the 8 pieces that
  // the threads of a shared-memory phase read at once (see the rotated key
  // reads below) sit on distinct banks.  The score is then
  // (sum_d k q 2^-e_h) 2^e_h / sqrt(128) log2(e) times the key row's scale.
  constexpr int QROW = 8 * G + 4;
  __shared__ __align__(16) uint32_t qs[8][QROW];
  __shared__ uint32_t qmax[kThreads / 32][G];
  __shared__ float qf[G];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x % splits, bg = blockIdx.x / splits;
  const int b = bg / Hkv, g = bg % Hkv;
  const int len = min(__ldg(lens + b), Lmax);
  const int t0 = s * TSPLIT;
  const int n = min(TSPLIT, len - t0);  // tokens of this split (<= 0: nothing)
  const int64_t pidx = static_cast<int64_t>(blockIdx.x) * G;
  if (n <= 0) {
    if (tid < G) {
      part_m[pidx + tid] = -INFINITY;
      part_l[pidx + tid] = 0.0f;
    }
    return;
  }
  const int chunks = (n + CH - 1) / CH;
  const int64_t row0 = static_cast<int64_t>(bg) * Lmax + t0;
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], kThreads / 32);
    }
    sh.abort = 0;
    fence_barrier_init();
  }
  const float qscale = 0.08838834764831845f * kLog2e;  // 1 / sqrt(128) * log2(e)
  const uint16_t* const qg = q + (static_cast<int64_t>(b) * Hkv * G + g * G) * D;
  {
    // each head's max |q| (thread: value pair tid of every head)
    uint32_t mx[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint32_t w = tid < D / 2 ? __ldg(reinterpret_cast<const uint32_t*>(qg + h * D) + tid) : 0u;
      mx[h] = __reduce_max_sync(0xFFFFFFFFu, max(w & 0x7FFFu, (w >> 16) & 0x7FFFu));
      if (lane == 0) qmax[warp][h] = mx[h];
    }
  }
  __syncthreads();
  if (tid < G) {
    uint32_t m = 0u;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) m = max(m, qmax[w][tid]);
    int e = 0;
    if (m != 0u) frexpf(bf16bits_to_f32(m), &e);  // max = f 2^e, 0.5 <= f < 1
    const int eh = m != 0u ? e - 15 : 0;
    qmax[0][tid] = static_cast<uint32_t>(eh);
    qf[tid] = __fmul_rn(qscale, pow2_from_exp(eh));
  }
  __syncthreads();
  for (int i = tid; i < G * (D / 2); i += kThreads) {
    const int h = i / (D / 2), jp = i % (D / 2);  // value pair jp of head h
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(qg + h * D) + jp);
    const Pow2Scaler sc(static_cast<int>(qmax[0][h]));
    const __half2 h2 = __floats2half2_rn(sc(bf16_lo(w)), sc(bf16_hi(w)));
    qs[jp >> 3][(jp & 7) * G + h] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  __syncthreads();
  // chunk c: n_c tokens; scales move in multiples of 4 (16 bytes), which stay
  // inside the cache because Lmax % 4 == 0
  auto issue = [&](int c) {
    const int st = c % NST;
    const int nc = min(CH, n - c * CH), nr = (nc + 3) & ~3;
    const int64_t r = row0 + c * CH;
    mbar_arrive_expect_tx(&sh.full[st], 2 * nc * D + 2 * nr * 4);
    bulk_load(sh.u.ring.k[st], kc + r * D, nc * D, &sh.full[st]);
    bulk_load(sh.u.ring.v[st], vc + r * D, nc * D, &sh.full[st]);
    bulk_load(sh.ks[st], ksc + r, nr * 4, &sh.full[st]);
    bulk_load(sh.vs[st], vsc + r, nr * 4, &sh.full[st]);
  };
  if (tid == 0)
    for (int c = 0; c < NST && c < chunks; ++c) issue(c);
  // running state (every thread keeps the head maxima; l and o per thread)
  float m_run[G], l_run[G], o[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) o[h][c] = 0.0f;
  }
  bool ok = true;
  for (int c = 0; c < chunks; ++c) {
    const int st = c % NST;
    const int nc = min(CH, n - c * CH);
    ok = mbar_wait(&sh.full[st], (c / NST) & 1, &sh.abort, status) && ok;
    // ---- scores: two threads per token, each half of the head dimension
    // (key pieces read in a rotated order, distinct banks per phase)
    const int t = tid >> 1, half = tid & 1;
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.0f;
    if (ok && t < nc) {
      const uint4* row = reinterpret_cast<const uint4*>(sh.u.ring.k[st] + t * D);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int piece = 4 * half + ((i + t) & 3);
        const uint4 w = row[piece];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t k01, k23;
          e4m3x4_to_f16x4(ws[e], k01, k23);
          const uint32_t* qp = &qs[piece][(2 * e) * G];  // value pairs 2e, 2e + 1 of the piece
#pragma unroll
          for (int h = 0; h < G; ++h) {
            fma_f16pair(acc[h], k01, qp[h]);
            fma_f16pair(acc[h], k23, qp[G + h]);
          }
        }
      }
    }
    float cmax[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      acc[h] += __shfl_xor_sync(0xFFFFFFFFu, acc[h], 1);  // the two halves of the token
      const float sc = (ok && t < nc) ? acc[h] * (sh.ks[st][t] * qf[h]) : -INFINITY;
      acc[h] = sc;
      float v = sc;
      for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
      cmax[h] = v;
    }
    if (lane == 0)
#pragma unroll
      for (int h = 0; h < G; ++h) sh.red[warp][h] = cmax[h];
    __syncthreads();
    float alpha[G], mnew[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float cm = fmaxf(fmaxf(sh.red[0][h], sh.red[1][h]), fmaxf(sh.red[2][h], sh.red[3][h]));
      mnew[h] = fmaxf(m_run[h], cm);
      alpha[h] = m_run[h] == -INFINITY ? 0.0f : ex2f(m_run[h] - mnew[h]);
      m_run[h] = mnew[h];
      l_run[h] *= alpha[h];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) o[h][cc] *= alpha[h];
    }
    if (half == 0 && t < nc) {
      const float vscale = sh.vs[st][t];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pe = ok ? ex2f(acc[h] - mnew[h]) : 0.0f;
        l_run[h] += pe;
        sh.p[t][h] = pe * vscale;
      }
    }
    __syncthreads();
    // ---- p . V: warp w takes tokens w, w + 4, ...; lane = 4 values of d
    if (ok)
      for (int tt = warp; tt < nc; tt += 4) {
        float f[4];
        e4m3x4_to_f32(reinterpret_cast<const uint32_t*>(sh.u.ring.v[st] + tt * D)[lane], f);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pw = sh.p[tt][h];
          // two values per instruction on the paired fp32 pipe (each half an
          // ordinary fp32 FMA)
          asm("{\n\t.reg .b64 aa, bb, ff, gg, pp;\n\t"
              "mov.b64 aa, {%0, %1};\n\tmov.b64 bb, {%2, %3};\n\t"
              "mov.b64 ff, {%4, %5};\n\tmov.b64 gg, {%6, %7};\n\tmov.b64 pp, {%8, %8};\n\t"
              "fma.rn.f32x2 aa, pp, ff, aa;\n\tfma.rn.f32x2 bb, pp, gg, bb;\n\t"
              "mov.b64 {%0, %1}, aa;\n\tmov.b64 {%2, %3}, bb;\n\t}"
              : "+f"(o[h][0]), "+f"(o[h][1]), "+f"(o[h][2]), "+f"(o[h][3])
              : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(pw));
        }
      }
    __syncthreads();  // sh.p and sh.red are rewritten by the next chunk
    if (lane == 0) mbar_arrive(&sh.empty[st]);
    if (tid == 0 && c + NST < chunks) {
      // the ring slot is free once every warp has read it
      if (!mbar_wait(&sh.empty[st], (c / NST) & 1, &sh.abort, status)) ok = false;
      else issue(c + NST);
    }
  }
  // ---- merge the warps' outputs and the threads' sums
#pragma unroll
  for (int h = 0; h < G; ++h) {
    *reinterpret_cast<float4*>(&sh.u.o[warp][h][4 * lane]) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
    float v = l_run[h];
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    if (lane == 0) sh.red[warp][h] = v;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += kThreads) {
    const int h = i / D, d = i % D;
    part_o[pidx * D + i] = sh.u.o[0][h][d] + sh.u.o[1][h][d] + sh.u.o[2][h][d] + sh.u.o[3][h][d];
  }
  if (tid < G) {
    part_m[pidx + tid] = ok ? m_run[tid] : -INFINITY;
    part_l[pidx + tid] = ok ? (sh.red[0][tid] + sh.red[1][tid] + sh.red[2][tid] + sh.red[3][tid]) : 0.0f;
  }
  // every issued copy has landed before the CTA exits
  if (tid == 0) {
    volatile int no_abort = 0;
    for (int c = max(0, chunks - NST); c < chunks; ++c)
      mbar_wait(&sh.full[c % NST], (c / NST) & 1, &no_abort, status);
  }
}

// Merge the splits of every (sequence, query head) in split order: one warp
// per output row, lane = 4 values.
__global__ void attn_combine_kernel(const float* __restrict__ part_m, const float* __restrict__ part_l,
                                    const float* __restrict__ part_o, int B, int Hkv, int G, int splits,
                                    __nv_bfloat16* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);  // (b, h) over B * Hq
  if (row >= B * Hkv * G) return;
  const int bg = row / G, h = row % G;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part_m[(static_cast<int64_t>(bg) * splits + s) * G + h]);
  float L = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (M > -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const int64_t pi = (static_cast<int64_t>(bg) * splits + s) * G + h;
      const float ms = part_m[pi];
      if (ms == -INFINITY) continue;
      const float w = ex2f(ms - M);
      L += w * part_l[pi];
      const float4 v = *reinterpret_cast<const float4*>(part_o + pi * D + 4 * lane);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    }
  }
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  const __nv_bfloat162 a = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  const __nv_bfloat162 c = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&c);
  reinterpret_cast<uint2*>(out + static_cast<int64_t>(row) * D)[lane] = w;
}

int attn_splits(int Lmax) { return (Lmax + TSPLIT - 1) / TSPLIT; }

cudaError_t launch_kv_append_fp8(const void* k_new, const void* v_new, int B, int Hkv, const int32_t* pos, int Lmax,
                                 uint8_t* kc, float* ksc, uint8_t* vc, float* vsc, int mode, int32_t* status,
                                 cudaStream_t stream) {
  const int rows = 2 * B * Hkv;
  if (rows == 0) return cudaSuccess;
  kv_append_fp8_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(static_cast<const uint16_t*>(k_new),
                                                           static_cast<const uint16_t*>(v_new), B, Hkv, pos, Lmax, kc,
                                                           ksc, vc, vsc, mode, status);
  return cudaGetLastError();
}

template <int G>
static cudaError_t launch_attn_g(const void* q, const uint8_t* kc, const float* ksc, const uint8_t* vc,
                                 const float* vsc, const int32_t* lens, int B, int Hkv, int Lmax, float* pm, float* pl,
                                 float* po, int32_t* status, cudaStream_t stream) {
  static bool attr = false;
  const int smem = static_cast<int>(sizeof(AttnShared<G>));
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_fp8_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int splits = attn_splits(Lmax);
  const unsigned grid = static_cast<unsigned>(B * Hkv * splits);
  attn_decode_fp8_kernel<G><<<grid, kThreads, smem, stream>>>(static_cast<const uint16_t*>(q), kc, ksc, vc, vsc, lens,
                                                             Hkv, Lmax, splits, pm, pl, po, status);
  return cudaGetLastError();
}

cudaError_t launch_attention_decode_fp8(const void* q, const uint8_t* kc, const float* ksc, const uint8_t* vc,
                                        const float* vsc, const int32_t* lens, int B, int Hq, int Hkv, int Lmax,
                                        void* out, float* pm, float* pl, float* po, int32_t* status,
                                        cudaStream_t stream) {
  if (B == 0 || Hq == 0) return cudaSuccess;
  const int G = Hq / Hkv;
  cudaError_t e;
  switch (G) {
    case 1: e = launch_attn_g<1>(q, kc, ksc, vc, vsc, lens, B, Hkv, Lmax, pm, pl, po, status, stream); break;
    case 2: e = launch_attn_g<2>(q, kc, ksc, vc, vsc, lens, B, Hkv, Lmax, pm, pl, po, status, stream); break;
    case 4: e = launch_attn_g<4>(q, kc, ksc, vc, vsc, lens, B, Hkv, Lmax, pm, pl, po, status, stream); break;
    default: e = launch_attn_g<8>(q, kc, ksc, vc, vsc, lens, B, Hkv, Lmax, pm, pl, po, status, stream); break;
  }
  if (e != cudaSuccess) return e;
  const int rows = B * Hq;
  attn_combine_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(pm, pl, po, B, Hkv, G, attn_splits(Lmax),
                                                          static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace qrr

// Adaptive quantization noise on the device: the counter-based generator and
// the noisy bf16 master it produces.
//
// QeRL ("QeRL: Beyond Efficiency -- Quantization-enhanced Reinforcement
// Learning for LLMs", Abstract) adds noise to the quantized policy whose
// strength changes during training.  Here element e of tensor j at training
// step s gets
//   z = sqrt(3) (k1 + k2 + k3 + k4 - 510) / 256
// from the four bytes k_i of output word r[e % 4] of Philox4x32-10
// (J. K. Salmon et al., "Parallel random numbers: as easy as 1, 2, 3",
// SC'11) at counter (e / 4 low, e / 4 high, j, s), key (seed low, seed
// high), and the master becomes
//   W' = bf16_rn(fp32(W) + fp32(sigma z)).
// Every step is an integer operation or one correctly rounded fp32 operation
// (no contraction into an FMA), so the noise and W' are reproducible bit for
// bit on any IEEE machine; one generator call serves four elements.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace qrr {

struct AqnParams {
  float sigma;    // 0: no noise
  uint32_t step;  // training step (third counter word)
  uint64_t seed;  // key
  // the generator's round keys for this seed (round i: the seed's words
  // plus i times the Weyl constants), set by aqn_params(); kernels read them
  // straight from their launch parameters
  uint32_t rk0[10], rk1[10];
};

__host__ __device__ inline AqnParams aqn_params(float sigma, uint32_t step, uint64_t seed) {
  AqnParams a{sigma, step, seed, {}, {}};
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    a.rk0[i] = k0;
    a.rk1[i] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return a;
}

__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, const AqnParams& a,
                                              uint32_t (&r)[4]) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c0, p1 = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
    const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
    const uint32_t n0 = hi1 ^ c1 ^ a.rk0[i], n2 = hi0 ^ c3 ^ a.rk1[i];
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  r[0] = c0;
  r[1] = c1;
  r[2] = c2;
  r[3] = c3;
}

// The standardized sum of the four bytes of a word: one dot-product
// instruction sums the bytes, the bit pattern 2^23 + sum less 2^23 + 510
// (both integers below 2^24, so the difference is exact) is sum - 510, and
// one correctly rounded multiply scales it by fp32(sqrt 3) 2^-8 -- bit for
// bit fp32(sqrt 3) times the exact (sum - 510) 2^-8, as scaling by a power
// of two commutes with rounding.
__device__ __forceinline__ float aqn_z(uint32_t w) {
  const uint32_t sum = __dp4a(w, 0x01010101u, 0u);  // 0 .. 1020
  const float f = __fsub_rn(__uint_as_float(0x4B000000u | sum), 8389118.0f);  // = sum - 510, exactly
  return __fmul_rn(f, 1.7320508075688772f * 0x1p-8f);
}

// The largest |z| aqn_z can return, with the same rounding: fp32 of 510
// times the same constant.  fp32(sigma) times it bounds |fp32(sigma z)|,
// because rounding is monotone.
__device__ __forceinline__ float aqn_zmax() { return __fmul_rn(510.0f, 1.7320508075688772f * 0x1p-8f); }

// The four generator words of elements 4 c .. 4 c + 3 of tensor `tensor`.
__device__ __forceinline__ void aqn_words(uint64_t c, uint32_t tensor, const AqnParams& a, uint32_t (&r)[4]) {
  philox4x32_10(static_cast<uint32_t>(c), static_cast<uint32_t>(c >> 32), tensor, a.step, a, r);
}

// bf16x2 bits of bf16_rn(fp32(w) + fp32(sigma z)) for both halves of the
// bf16x2 w (za for the low half, zb for the high one): one paired
// round-to-nearest-even conversion.
__device__ __forceinline__ uint32_t aqn_noisy2(uint32_t w, float sigma, float za, float zb) {
  const float lo = __fadd_rn(__uint_as_float(w << 16), __fmul_rn(sigma, za));
  const float hi = __fadd_rn(__uint_as_float(w & 0xFFFF0000u), __fmul_rn(sigma, zb));
  uint32_t o;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o) : "f"(hi), "f"(lo));
  return o;
}

// Eight consecutive bf16 values starting at element e0 (a multiple of 8):
// two generator calls.
__device__ __forceinline__ uint4 aqn_noisy8(uint4 v, uint64_t e0, uint32_t tensor, const AqnParams& a) {
  uint32_t r0[4], r1[4];
  aqn_words(e0 >> 2, tensor, a, r0);
  aqn_words((e0 >> 2) + 1, tensor, a, r1);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t za = i < 2 ? r0[2 * i] : r1[2 * i - 4], zb = i < 2 ? r0[2 * i + 1] : r1[2 * i - 3];
    o[i] = aqn_noisy2(w[i], a.sigma, aqn_z(za), aqn_z(zb));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace qrr

// Adaptive quantization noise on the device: the counter-based generator and
// the noisy bf16 master it produces.
//
// QeRL ("QeRL: Beyond Efficiency -- Quantization-enhanced Reinforcement
// Learning for LLMs", Abstract) adds noise to the quantized policy whose
// strength changes during training.  Here element e of tensor j at training
// step s gets
//   z = sqrt(3) (k1 + k2 + k3 + k4 - 131070) / 65536
// from the four 16-bit halves k_i of two output words of Philox4x32-10
// (J. K. Salmon et al., "Parallel random numbers: as easy as 1, 2, 3",
// SC'11) at counter (e / 2 low, e / 2 high, j, s), key (seed low, seed high)
// -- words r0, r1 for even e, r2, r3 for odd e -- and the master becomes
//   W' = bf16_rn(fp32(W) + fp32(sigma z)).
// Every step is an integer operation or one correctly rounded fp32 operation
// (no contraction into an FMA), so the noise and W' are reproducible bit for
// bit on any IEEE machine.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace qrr {

struct AqnParams {
  float sigma;    // 0: no noise
  uint32_t step;  // training step (third counter word)
  uint64_t seed;  // key
};

__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                              uint32_t k1, uint32_t (&r)[4]) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  r[0] = c0;
  r[1] = c1;
  r[2] = c2;
  r[3] = c3;
}

// The standardized sum of the four 16-bit halves of two words.
__device__ __forceinline__ float aqn_z(uint32_t a, uint32_t b) {
  const int centred = static_cast<int>((a & 0xFFFFu) + (a >> 16) + (b & 0xFFFFu) + (b >> 16)) - 131070;
  const float zc = __fmul_rn(__int2float_rn(centred), 0x1p-16f);  // exact
  return __fmul_rn(zc, 1.7320508075688772f);
}

// z of elements 2 p and 2 p + 1 of tensor `tensor`.
__device__ __forceinline__ void aqn_z2(uint64_t p, uint32_t tensor, const AqnParams& a, float& z0, float& z1) {
  uint32_t r[4];
  philox4x32_10(static_cast<uint32_t>(p), static_cast<uint32_t>(p >> 32), tensor, a.step,
                static_cast<uint32_t>(a.seed), static_cast<uint32_t>(a.seed >> 32), r);
  z0 = aqn_z(r[0], r[1]);
  z1 = aqn_z(r[2], r[3]);
}

// bf16 bits of bf16_rn(fp32(w) + fp32(sigma z)).
__device__ __forceinline__ uint32_t aqn_noisy(uint32_t wbits, float sigma, float z) {
  const float s = __fadd_rn(__uint_as_float(wbits << 16), __fmul_rn(sigma, z));
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(s)));
}

// The packed pair of bf16 values in `w` (elements 2 p, 2 p + 1), made noisy.
__device__ __forceinline__ uint32_t aqn_noisy2(uint32_t w, uint64_t p, uint32_t tensor, const AqnParams& a) {
  float z0, z1;
  aqn_z2(p, tensor, a, z0, z1);
  return aqn_noisy(w & 0xFFFFu, a.sigma, z0) | (aqn_noisy(w >> 16, a.sigma, z1) << 16);
}

// Eight consecutive bf16 values starting at element e0 (even).
__device__ __forceinline__ uint4 aqn_noisy8(uint4 v, uint64_t e0, uint32_t tensor, const AqnParams& a) {
  const uint64_t p = e0 >> 1;
  return make_uint4(aqn_noisy2(v.x, p, tensor, a), aqn_noisy2(v.y, p + 1, tensor, a), aqn_noisy2(v.z, p + 2, tensor, a),
                    aqn_noisy2(v.w, p + 3, tensor, a));
}

}  // namespace qrr

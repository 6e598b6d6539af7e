// Device helpers shared by the sm_103a kernels: rounding onto the E2M1 / E4M3
// grids, exact E4M3 decode, bf16 absmax, and the power-of-two scale rule.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qrr.h"

namespace qrr {

constexpr int kSMs = 152;  // GB300: 2 dies x 76 SMs (grids are sized from the live device count)

// ---- rounding primitives (hardware cvt: round-to-nearest-even, satfinite,
//      sign kept) ------------------------------------------------------------

// Two fp32 -> one byte of two E2M1 codes; `lo` lands in bits 3..0.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Eight fp32 -> one word of eight E2M1 codes, value k in nibble k: four
// conversions whose bytes are packed by one register move.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\tcvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\tcvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// Two fp32 -> two E4M3 bytes; `lo` lands in bits 7..0.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Exact value of an E4M3 (FN) byte, from its bit fields.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20))  // (1 + m/8) 2^(e-7)
                : static_cast<float>(m) * 0.001953125f;            // m 2^-9
  return __uint_as_float(__float_as_uint(mag) | ((b & 0x80u) << 24));
}

// The same value through the hardware conversion (every E4M3 value is an
// f16, and every f16 an fp32).
__device__ __forceinline__ float e4m3_to_f32_cvt(uint32_t b) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(b));
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// bf16 bits -> fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Largest |bf16| bit pattern (sign cleared) of the 8 values in a uint4, as a
// 15-bit integer: non-negative bf16 order like their bit patterns, so an
// integer max is the absmax, and >= 0x7F80 means inf/NaN.
__device__ __forceinline__ uint32_t absmax_bits8(uint4 v) {
  uint32_t m = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
  m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
  return max(m & 0xFFFFu, m >> 16);
}

__device__ __forceinline__ float bf16bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// ---- FP8 scale rules --------------------------------------------------------

// Power-of-two scale: the smallest 2^e with 2^e >= v (v > 0, finite).
// Returns e; the scale itself is pow2_from_exp(e).
__device__ __forceinline__ int pow2_ceil_exp(float v) {
  const uint32_t bits = __float_as_uint(v);
  if (bits >= 0x00800000u) {  // normal
    const int ex = static_cast<int>(bits >> 23) - 127;
    return ex + ((bits & 0x7FFFFFu) != 0u);
  }
  // subnormal: v = m 2^-149, ceil(log2 m) = 32 - clz(m - 1)
  return -149 + (32 - __clz(static_cast<int>(bits - 1u)));
}

__device__ __forceinline__ float pow2_from_exp(int e) {  // e in [-149, 127]
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                   : __uint_as_float(1u << (e + 149));
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

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// An f16x2 of E2M1 values (only the top mantissa bit can be set) re-read as
// the bf16x2 of the same values times 2^-112: each half's exponent and
// mantissa fields move down three bits (an f16 exponent under the bf16 bias,
// 127 - 15 = 112; the bits shifted out are zero), the sign stays.  One bf16x2
// multiply by s 2^112 then gives v s exactly whenever v s has at most eight
// significant bits and both factors are normal bf16 numbers.
__device__ __forceinline__ uint32_t e2m1_f16x2_rebias_bf16x2(uint32_t h) {
  return ((h & 0x7FFF7FFFu) >> 3) | (h & 0x80008000u);
}

// x * 2^-e, exact for the magnitudes that reach the E4M3 grid.
struct Pow2Scaler {
  float f1, f2;
  __device__ __forceinline__ explicit Pow2Scaler(int e) {
    const int ne = -e;  // in [-127, 149]
    if (ne <= 127) {
      f1 = __uint_as_float(static_cast<uint32_t>(ne + 127) << 23);
      f2 = 1.0f;
    } else {
      f1 = __uint_as_float(254u << 23);  // 2^127
      f2 = __uint_as_float(static_cast<uint32_t>(ne - 127 + 127) << 23);
    }
  }
  __device__ __forceinline__ float operator()(float x) const { return __fmul_rn(__fmul_rn(x, f1), f2); }
};

// ---- correctly rounded division by a value shared across many numerators ----
//
// x / d rounded to nearest-even in fp32 with FMA corrections (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990): with y = RN(1/d) and q an
// approximation of x/d within one ulp, the residual r = x - d q is exact
// under an FMA and RN(q + r y) = RN(x / d).  Here q0 = RN(x y) can miss by a
// little more than an ulp, so one correction first makes it faithful
// (q1 = RN(q0 + r0 y)) and a second gives the correctly rounded quotient.
// The residuals stay exact while d (and so y) lies in [1e-20, 1e20]: every
// quotient that can reach a nonzero E2M1 / E4M3 code (|x/d| >= 2^-10) then
// has |x| >= 1e-23 and its residuals are far from the subnormal range.
// Outside that range the divisor falls back to __fdiv_rn.  The divisor is
// positive; the quotient takes the numerator's sign, which keeps -0 / d = -0
// (the FMA corrections alone would turn it into +0).
struct SharedDivisor {
  float d, y;
  bool ok;
  SharedDivisor() = default;
  __device__ __forceinline__ explicit SharedDivisor(float d_) : d(d_) {
    y = __frcp_rn(d_);
    const float ad = fabsf(d_);
    ok = ad >= 1.0e-20f && ad <= 1.0e20f;
  }
  __device__ __forceinline__ float operator()(float x) const {
    if (!ok) return __fdiv_rn(x, d);
    const float q0 = __fmul_rn(x, y);
    const float q1 = __fmaf_rn(__fmaf_rn(-q0, d, x), y, q0);
    return copysignf(__fmaf_rn(__fmaf_rn(-q1, d, x), y, q1), x);
  }
};

// The same division for two numerators at once on the paired fp32 pipe
// (fma.rn.f32x2: each half an ordinary correctly-rounded fp32 FMA, so the
// quotients are bit-identical to SharedDivisor's).  The residual x - q d is
// formed as fma(q, -d, x), the same exact value as fma(-q, d, x).
struct SharedDivisor2 {
  float d;
  uint64_t y2, nd2;
  bool ok;
  __device__ __forceinline__ explicit SharedDivisor2(float d_) : d(d_) {
    const float y = __frcp_rn(d_);
    const float ad = fabsf(d_);
    ok = ad >= 1.0e-20f && ad <= 1.0e20f;
    asm("mov.b64 %0, {%1, %1};" : "=l"(y2) : "f"(y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(nd2) : "f"(-d_));
  }
  __device__ __forceinline__ void operator()(float x0, float x1, float& q0, float& q1) const {
    if (!ok) {
      q0 = __fdiv_rn(x0, d);
      q1 = __fdiv_rn(x1, d);
      return;
    }
    fast(x0, x1, q0, q1);
  }
  // the same for a divisor known to lie in [1e-20, 1e20] (ok set)
  __device__ __forceinline__ void fast(float x0, float x1, float& q0, float& q1) const {
    uint64_t x, q, r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q) : "l"(x), "l"(y2));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q), "l"(nd2), "l"(x));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(r), "l"(y2), "l"(q));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(q), "l"(nd2), "l"(x));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(r), "l"(y2), "l"(q));
    float a, b;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(q));
    q0 = copysignf(a, x0);
    q1 = copysignf(b, x1);
  }
};

__device__ __forceinline__ void flag(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

}  // namespace qrr

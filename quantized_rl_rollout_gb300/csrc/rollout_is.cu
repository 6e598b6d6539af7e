// Token log-probabilities and token-level importance-sampling weights.
//
//   logp[t] = logits[t, tok[t]] - log(sum_v exp(logits[t, v]))
//   w[t]    = min(exp(logp[t] - logp_rollout[t]), cap)     (cap <= 0: no cap)
//
// ("NVIDIA NeMo RL behaalt 48% ...", the paragraph on importance sampling in
// "Waarom dit belangrijk is voor AI-economie": the shift between the
// generation engine's and the trainer's distributions is corrected token by
// token.)
//
// HBM-bound: every logit is read once.  One CTA (256 threads) per token row;
// each thread streams its share of the row with 16-byte loads, four in
// flight, and keeps a running (max, sum of exp(x - max)) in fp32: the max of
// each 32 values by packed bf16 max, then one FMA, one exp2 and one add per
// value; the CTA then merges the 256 pairs.  Exponent and logarithm use the
// base-2 hardware approximations (relative error about 2^-22).  A NaN or +inf
// logit is detected from the final log-sum-exp, not per value.
#include <cuda_bf16.h>

#include "linear.cuh"
#include "tc.cuh"

namespace qrr {

namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Running log-sum-exp state in log2(e)-scaled units: m = max of x log2(e)
// (-inf while empty), s = sum of 2^(x log2(e) - m).
struct Lse {
  float m = -INFINITY, s = 0.0f;
  __device__ __forceinline__ void add_block(const float* v, int n, float bmax) {
    if (bmax == -INFINITY) return;  // all -inf: contributes nothing
    if (bmax > m) {
      s = m == -INFINITY ? 0.0f : s * ex2(m - bmax);
      m = bmax;
    }
    float acc = 0.0f;
    for (int i = 0; i < n; ++i) acc += ex2(v[i] - m);
    s += acc;
  }
  __device__ __forceinline__ void merge(float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) {
      m = m2;
      s = s2;
      return;
    }
    const float mx = fmaxf(m, m2);
    s = s * ex2(m - mx) + s2 * ex2(m2 - mx);
    m = mx;
  }
};

}  // namespace

// Largest of the 16 bf16 pairs in q[4] as an fp32 value (packed bf16 max).
__device__ __forceinline__ float bf16_max32(const uint4 (&q)[4]) {
  uint32_t w[16] = {q[0].x, q[0].y, q[0].z, q[0].w, q[1].x, q[1].y, q[1].z, q[1].w,
                    q[2].x, q[2].y, q[2].z, q[2].w, q[3].x, q[3].y, q[3].z, q[3].w};
#pragma unroll
  for (int n = 8; n >= 1; n >>= 1)
#pragma unroll
    for (int i = 0; i < n; ++i) asm("max.bf16x2 %0, %1, %2;" : "=r"(w[i]) : "r"(w[i]), "r"(w[i + n]));
  return fmaxf(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u));
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 6) token_logprob_is_kernel(const uint16_t* __restrict__ logits, int64_t T,
                                                                       int64_t V, const int32_t* __restrict__ tokens,
                                                                       const float* __restrict__ rollout_logp,
                                                                       float cap, float* __restrict__ logp,
                                                                       float* __restrict__ w, int32_t* status) {
  __shared__ float red_m[kThreads / 32], red_s[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const int tok = __ldg(tokens + t);
    const bool live = tok >= 0 && tok < V;
    // running state: xm = max of the raw logits seen, s = sum of e^(x - xm)
    float xm = -INFINITY, s = 0.0f;
    if (live) {
      const uint16_t* row = logits + t * V;
      if constexpr (VEC) {
        const uint4* rv = reinterpret_cast<const uint4*>(row);
        const int64_t nvec = V / 8;
        const uint4 pad = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);  // bf16 -inf
        for (int64_t base = threadIdx.x; base < nvec; base += 4 * kThreads) {
          uint4 q[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int64_t i = base + u * kThreads;
            q[u] = i < nvec ? __ldcs(rv + i) : pad;  // streamed once: evict first
          }
          const float bmax = bf16_max32(q);
          if (!(bmax > -INFINITY)) {
            // all -inf, or NaN beside -inf (the packed max skips NaN, and a
            // sum whose max is -inf is dropped by the merge): report it here
            bool nan_seen = false;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t wd[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                nan_seen |= (wd[e] & 0x7FFFu) > 0x7F80u || (wd[e] & 0x7FFF0000u) > 0x7F800000u;
            }
            if (nan_seen) flag(status, QRR_DEV_NONFINITE);
            continue;
          }
          if (bmax > xm) {
            s = xm == -INFINITY ? 0.0f : s * ex2((xm - bmax) * kLog2e);
            xm = bmax;
          }
          const float nm = -xm * kLog2e;
          float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t wd[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc0 += ex2(fmaf(__uint_as_float(wd[e] << 16), kLog2e, nm));
              acc1 += ex2(fmaf(__uint_as_float(wd[e] & 0xFFFF0000u), kLog2e, nm));
            }
          }
          s += acc0 + acc1;
        }
      } else {
        for (int64_t i = threadIdx.x; i < V; i += kThreads) {
          const float x = __uint_as_float(static_cast<uint32_t>(__ldcs(row + i)) << 16);
          if (!(x > -INFINITY)) {
            if (x != x) flag(status, QRR_DEV_NONFINITE);
            continue;
          }
          if (x > xm) {
            s = xm == -INFINITY ? 0.0f : s * ex2((xm - x) * kLog2e);
            xm = x;
          }
          s += ex2((x - xm) * kLog2e);
        }
      }
    }
    // CTA merge of the (max, sum) pairs, in log2(e)-scaled units
    Lse st;
    st.m = xm * kLog2e;
    st.s = s;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, st.m, o);
      const float s2 = __shfl_xor_sync(0xFFFFFFFFu, st.s, o);
      st.merge(m2, s2);
    }
    if (lane == 0) {
      red_m[warp] = st.m;
      red_s[warp] = st.s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      Lse all;
      for (int i = 0; i < kThreads / 32; ++i) all.merge(red_m[i], red_s[i]);
      float lp = 0.0f, wt = 0.0f;
      if (live) {
        const float lse2 = all.m + lg2(all.s);  // log2 of sum_v 2^(x_v log2 e)
        // a NaN or +inf logit leaves the log-sum-exp NaN or +inf
        if (lse2 != lse2 || lse2 == INFINITY) flag(status, QRR_DEV_NONFINITE);
        const float x = __uint_as_float(static_cast<uint32_t>(__ldg(logits + t * V + tok)) << 16);
        lp = x - lse2 * kLn2;
        if (rollout_logp) {
          wt = ex2((lp - __ldg(rollout_logp + t)) * kLog2e);
          if (cap > 0.0f) wt = fminf(wt, cap);
        }
      }
      if (tok >= V) flag(status, QRR_DEV_BAD_INDEX);
      logp[t] = lp;
      if (rollout_logp) w[t] = wt;
    }
    __syncthreads();  // red_m / red_s are reused by the next row
  }
}

cudaError_t launch_token_logprob_is(const void* logits, int64_t T, int64_t V, const int32_t* tokens,
                                    const float* rollout_logp, float cap, float* logp, float* w, int32_t* status,
                                    cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  int dev = 0, sms = kSMs;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap_ctas = static_cast<int64_t>(sms) * 6;  // 6 resident CTAs per SM
  const unsigned grid = static_cast<unsigned>(T < cap_ctas ? T : cap_ctas);
  const bool vec = V % 8 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0;
  if (vec)
    token_logprob_is_kernel<true><<<grid, kThreads, 0, stream>>>(static_cast<const uint16_t*>(logits), T, V, tokens,
                                                                  rollout_logp, cap, logp, w, status);
  else
    token_logprob_is_kernel<false><<<grid, kThreads, 0, stream>>>(static_cast<const uint16_t*>(logits), T, V,
                                                                   tokens, rollout_logp, cap, logp, w, status);
  return cudaGetLastError();
}

}  // namespace qrr

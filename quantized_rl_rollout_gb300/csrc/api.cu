// C ABI of the library (include/qrr.h): host-side validation, workspace
// carving and dispatch to the kernels.  Nothing here allocates device memory
// or synchronizes with the host.
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "linear.cuh"
#include "quant.cuh"
#include "tc.cuh"

using namespace qrr;

namespace {

constexpr size_t kAlign = 256;

inline size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Host-side fault injection for tests of the error path: with
// QRR_INJECT_FAULT=cuda every call reports QRR_ERR_CUDA after validation and
// launches nothing.
inline bool injected_cuda_fault() {
  const char* v = getenv("QRR_INJECT_FAULT");
  return v && strcmp(v, "cuda") == 0;
}

inline qrr_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QRR_OK : QRR_ERR_CUDA; }

inline bool is_fp8_mode(int32_t m) { return m == QRR_SCALE_FP32 || m == QRR_SCALE_POW2; }

// How one linear call runs: operand type, token tile, split-K, workspace.
struct LinPlan {
  bool f16;
  int bn, m_tiles, n_tiles, splits, kcps, lora_chunks;
  size_t t_off, x16_off, p_off, part_off, cnt_off, total;
};

// Decode (<= 64 tokens) takes the f16 operand path and splits K until there
// are about two work units per SM, as long as the fp32 partials stay under a
// few percent of the weight bytes; prefill runs one unit per output tile.
LinPlan plan_linear(int64_t M, int64_t N, int64_t K, int32_t r) {
  LinPlan p{};
  const bool decode = M <= 64;
  p.f16 = decode;
  p.bn = w4_bn_for(M);
  p.n_tiles = static_cast<int>(N / 128);
  p.m_tiles = static_cast<int>((M + p.bn - 1) / p.bn);
  p.lora_chunks = r > 0 ? static_cast<int>((2 * r + 63) / 64) : 0;
  const int kc = static_cast<int>(K / 64);
  int splits = 1;
  if (decode && kc >= 8) {
    const int base = std::max(1, p.n_tiles * p.m_tiles);
    const int target = (2 * kSMs + base - 1) / base;
    const int cap = std::max<int>(1, static_cast<int>(0.035 * static_cast<double>(K) / static_cast<double>(std::max<int64_t>(M, 1))));
    splits = std::max(1, std::min(std::min(target, cap), kc / 4));
  }
  p.kcps = ((kc + splits - 1) / splits + 3) / 4 * 4;
  p.splits = std::max(1, (kc + p.kcps - 1) / std::max(1, p.kcps));
  size_t off = 0;
  p.t_off = off;
  off += round_up(static_cast<size_t>(M) * 64 * p.lora_chunks * 2);
  p.x16_off = off;
  if (p.f16) off += round_up(static_cast<size_t>(M) * static_cast<size_t>(K) * 2);
  p.p_off = off;
  if (p.f16) off += round_up(static_cast<size_t>(M) * 4);
  p.part_off = off;
  if (p.splits > 1) off += round_up(static_cast<size_t>(p.splits) * M * N * 4);
  p.cnt_off = off;
  off += round_up(static_cast<size_t>(p.m_tiles) * p.n_tiles * 4);
  p.total = off + kAlign;
  return p;
}

size_t linear_ws_bytes(int64_t M, int64_t N, int64_t K, int32_t r) {
  if (M < 0 || N < 0 || K < 0 || r < 0) return 0;
  return plan_linear(M, N, K, r).total;
}

}  // namespace

extern "C" {

const char* qrr_status_string(int status) {
  switch (status) {
    case QRR_OK: return "QRR_OK";
    case QRR_ERR_INVALID_ARG: return "QRR_ERR_INVALID_ARG";
    case QRR_ERR_UNSUPPORTED_SHAPE: return "QRR_ERR_UNSUPPORTED_SHAPE";
    case QRR_ERR_MISALIGNED: return "QRR_ERR_MISALIGNED";
    case QRR_ERR_WORKSPACE: return "QRR_ERR_WORKSPACE";
    case QRR_ERR_CUDA: return "QRR_ERR_CUDA";
    default: return "QRR_UNKNOWN_STATUS";
  }
}

int qrr_abi_version(void) { return 1; }

size_t qrr_quantize_nvfp4_workspace_bytes(void) { return kAlign; }

size_t qrr_requantize_workspace_bytes(int32_t count) {
  return count <= 0 ? kAlign : round_up(static_cast<size_t>(count) * sizeof(uint32_t));
}

size_t qrr_linear_nvfp4_lora_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r) {
  return linear_ws_bytes(M, N, K, r);
}

static qrr_status check_nvfp4_tensor(const void* W, int64_t N, int64_t K, const uint8_t* codes,
                                     const uint8_t* scales, const float* tensor_scale) {
  if (N < 0 || K < 0) return QRR_ERR_INVALID_ARG;
  if (!tensor_scale) return QRR_ERR_INVALID_ARG;
  if (N * K > 0 && (!W || !codes || !scales)) return QRR_ERR_INVALID_ARG;
  if (K % 32 != 0) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(W) || !aligned16(codes) || !aligned16(scales) || (reinterpret_cast<uintptr_t>(tensor_scale) & 3u))
    return QRR_ERR_MISALIGNED;
  return QRR_OK;
}

qrr_status qrr_quantize_nvfp4(const void* W, int64_t N, int64_t K, uint8_t* codes, uint8_t* scales,
                              float* tensor_scale, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream) {
  qrr_status st = check_nvfp4_tensor(W, N, K, codes, scales, tensor_scale);
  if (st != QRR_OK) return st;
  if (!workspace || workspace_bytes < qrr_quantize_nvfp4_workspace_bytes()) return QRR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  Nvfp4Batch batch{};
  batch.count = 1;
  batch.job[0] = Nvfp4Job{static_cast<const uint16_t*>(W), codes, scales, tensor_scale, N, K, 0, 0};
  batch.amax_bits = static_cast<uint32_t*>(workspace);
  batch.status = dev_status;
  return from_cuda(launch_nvfp4(batch, as_stream(stream)));
}

qrr_status qrr_linear_nvfp4_lora(const void* x, int64_t M, int64_t K, const uint8_t* codes, const uint8_t* scales,
                                 const float* tensor_scale, int64_t N, const void* lora_A, const void* lora_B,
                                 int32_t r, float alpha, void* y, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, void* stream) {
  (void)dev_status;
  if (M < 0 || N < 0 || K < 0 || r < 0) return QRR_ERR_INVALID_ARG;
  const bool lora = r > 0 && lora_A && lora_B;
  if (!tensor_scale) return QRR_ERR_INVALID_ARG;
  if (M * N > 0 && !y) return QRR_ERR_INVALID_ARG;
  if (M * K > 0 && !x) return QRR_ERR_INVALID_ARG;
  if (N * K > 0 && (!codes || !scales)) return QRR_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 128 != 0) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (lora && (r > 256 || r % 8 != 0)) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) || !aligned16(y) ||
      (lora && (!aligned16(lora_A) || !aligned16(lora_B))))
    return QRR_ERR_MISALIGNED;
  const int32_t rr = lora ? r : 0;
  if (!workspace || workspace_bytes < linear_ws_bytes(M, N, K, rr)) return QRR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  if (M == 0 || N == 0) return QRR_OK;
  cudaStream_t s = as_stream(stream);
  if (K == 0) return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(M * N) * 2, s));
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return QRR_ERR_UNSUPPORTED_SHAPE;
  const LinPlan pl = plan_linear(M, N, K, rr);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* tbuf = reinterpret_cast<__nv_bfloat16*>(ws + pl.t_off);
  __half* x16 = reinterpret_cast<__half*>(ws + pl.x16_off);
  int* pexp = reinterpret_cast<int*>(ws + pl.p_off);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ws + pl.cnt_off);
  cudaError_t e = cudaSuccess;
  if (pl.splits > 1) e = cudaMemsetAsync(counters, 0, static_cast<size_t>(pl.m_tiles) * pl.n_tiles * 4, s);
  if (e != cudaSuccess) return QRR_ERR_CUDA;
  if (pl.f16 || rr > 0) {
    PrepArgs pa{};
    pa.x = static_cast<const uint16_t*>(x);
    pa.A = static_cast<const uint16_t*>(lora_A);
    pa.tensor_scale = tensor_scale;
    pa.x16 = x16;
    pa.pexp = pexp;
    pa.t = tbuf;
    pa.M = M;
    pa.K = K;
    pa.r = rr;
    pa.t_cols = 64 * pl.lora_chunks;
    pa.lora_scale = rr > 0 ? alpha / static_cast<float>(rr) : 0.0f;
    pa.status = dev_status;
    if (launch_lora_prep(pa, pl.f16, s) != cudaSuccess) return QRR_ERR_CUDA;
  }
  W4Params p{};
  p.count = 1;
  p.status = dev_status;
  W4Layer& L = p.layer[0];
  const void* xsrc = pl.f16 ? static_cast<const void*>(x16) : x;
  const CUtensorMapDataType xt = pl.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_tmap_2d(&L.tx, xsrc, xt, M, K, K * 2, pl.bn, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&L.tcodes, codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, N, K / 2, K / 2, 128, 32,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
    return QRR_ERR_CUDA;
  if (rr > 0) {
    if (!make_tmap_2d(&L.tt, tbuf, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, M, 64 * pl.lora_chunks,
                      64 * pl.lora_chunks * 2, pl.bn, 64, CU_TENSOR_MAP_SWIZZLE_128B))
      return QRR_ERR_CUDA;
  } else {
    L.tt = L.tx;  // never read without an adapter
  }
  L.scales = scales;
  L.tensor_scale = tensor_scale;
  L.B = static_cast<const uint16_t*>(lora_B);
  L.pexp = pl.f16 ? pexp : nullptr;
  L.y = static_cast<__nv_bfloat16*>(y);
  L.partial = reinterpret_cast<float*>(ws + pl.part_off);
  L.counters = counters;
  L.M = static_cast<int>(M);
  L.N = static_cast<int>(N);
  L.K = static_cast<int>(K);
  L.r = rr;
  L.lora_chunks = pl.lora_chunks;
  L.n_tiles = pl.n_tiles;
  L.m_tiles = pl.m_tiles;
  L.splits = pl.splits;
  L.kcps = pl.kcps;
  return from_cuda(launch_w4a16_tc(p, pl.bn, pl.f16, s));
}

qrr_status qrr_quantize_fp8_w128x128(const void* W, int64_t N, int64_t K, uint8_t* q, float* scales,
                                     int32_t scale_mode, int32_t* dev_status, void* stream) {
  if (N < 0 || K < 0 || !is_fp8_mode(scale_mode)) return QRR_ERR_INVALID_ARG;
  if (N * K > 0 && (!W || !q || !scales)) return QRR_ERR_INVALID_ARG;
  if (K % 128 != 0) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(W) || !aligned16(q) || !aligned16(scales)) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  Fp8WBatch batch{};
  batch.count = 1;
  batch.mode = scale_mode;
  batch.status = dev_status;
  batch.job[0] = Fp8WJob{static_cast<const uint16_t*>(W), q, scales, N, K, 0};
  return from_cuda(launch_fp8_w128(batch, as_stream(stream)));
}

qrr_status qrr_quantize_fp8_a1x128(const void* x, int64_t M, int64_t K, uint8_t* q, float* scales,
                                   int32_t scale_mode, int32_t* dev_status, void* stream) {
  if (M < 0 || K < 0 || !is_fp8_mode(scale_mode)) return QRR_ERR_INVALID_ARG;
  if (M * K > 0 && (!x || !q || !scales)) return QRR_ERR_INVALID_ARG;
  if (K % 128 != 0) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(q) || !aligned16(scales)) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  return from_cuda(launch_fp8_a1x128(x, M, K, q, scales, scale_mode, dev_status, as_stream(stream)));
}

qrr_status qrr_gemm_fp8_blockwise(const uint8_t* qa, const float* sa, const uint8_t* qw, const float* sw, int64_t M,
                                  int64_t N, int64_t K, void* y, int32_t scale_mode, int32_t* dev_status,
                                  void* stream) {
  if (M < 0 || N < 0 || K < 0 || !is_fp8_mode(scale_mode)) return QRR_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (M * N > 0 && !y) return QRR_ERR_INVALID_ARG;
  if (M * K > 0 && (!qa || !sa)) return QRR_ERR_INVALID_ARG;
  if (N * K > 0 && (!qw || !sw)) return QRR_ERR_INVALID_ARG;
  if (K % 128 != 0 || N % 128 != 0) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(qw) || !aligned16(sw) || !aligned16(y))
    return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  if (M == 0 || N == 0) return QRR_OK;
  cudaStream_t s = as_stream(stream);
  if (K == 0) return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(M * N) * 2, s));
  Fp8GemmArgs a{qa, sa, qw, sw, y, M, N, K};
  return from_cuda(launch_fp8_gemm_tc(a, dev_status, s));
}

qrr_status qrr_requantize_weights(const qrr_weight_desc* descs, int32_t count, int32_t format, int32_t scale_mode,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (count < 0 || (count > 0 && !descs)) return QRR_ERR_INVALID_ARG;
  if (format != QRR_FORMAT_NVFP4 && format != QRR_FORMAT_FP8_W128) return QRR_ERR_INVALID_ARG;
  if (format == QRR_FORMAT_FP8_W128 && !is_fp8_mode(scale_mode)) return QRR_ERR_INVALID_ARG;
  for (int32_t i = 0; i < count; ++i) {
    const qrr_weight_desc& d = descs[i];
    if (format == QRR_FORMAT_NVFP4) {
      qrr_status st = check_nvfp4_tensor(d.W, d.N, d.K, d.codes, static_cast<const uint8_t*>(d.scales),
                                         d.tensor_scale);
      if (st != QRR_OK) return st;
    } else {
      if (d.N < 0 || d.K < 0) return QRR_ERR_INVALID_ARG;
      if (d.N * d.K > 0 && (!d.W || !d.codes || !d.scales)) return QRR_ERR_INVALID_ARG;
      if (d.K % 128 != 0) return QRR_ERR_UNSUPPORTED_SHAPE;
      if (!aligned16(d.W) || !aligned16(d.codes) || !aligned16(d.scales)) return QRR_ERR_MISALIGNED;
    }
  }
  if (format == QRR_FORMAT_NVFP4) {
    if (count > 0 && (!workspace || workspace_bytes < qrr_requantize_workspace_bytes(kMaxJobs < count ? kMaxJobs : count)))
      return QRR_ERR_WORKSPACE;
    if (!aligned16(workspace)) return QRR_ERR_MISALIGNED;
  }
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  cudaStream_t s = as_stream(stream);
  // groups of up to kMaxJobs tensors per grouped launch; NVFP4 groups reuse
  // the same absmax words, which stream order makes safe
  for (int32_t g = 0; g < count; g += kMaxJobs) {
    const int n = count - g < kMaxJobs ? count - g : kMaxJobs;
    cudaError_t e;
    if (format == QRR_FORMAT_NVFP4) {
      Nvfp4Batch batch{};
      batch.count = n;
      batch.amax_bits = static_cast<uint32_t*>(workspace);
      batch.status = dev_status;
      for (int i = 0; i < n; ++i) {
        const qrr_weight_desc& d = descs[g + i];
        batch.job[i] = Nvfp4Job{static_cast<const uint16_t*>(d.W), d.codes, static_cast<uint8_t*>(d.scales),
                                d.tensor_scale, d.N, d.K, 0, 0};
      }
      e = launch_nvfp4(batch, s);
    } else {
      Fp8WBatch batch{};
      batch.count = n;
      batch.mode = scale_mode;
      batch.status = dev_status;
      for (int i = 0; i < n; ++i) {
        const qrr_weight_desc& d = descs[g + i];
        batch.job[i] = Fp8WJob{static_cast<const uint16_t*>(d.W), d.codes, static_cast<float*>(d.scales), d.N, d.K, 0};
      }
      e = launch_fp8_w128(batch, s);
    }
    if (e != cudaSuccess) return QRR_ERR_CUDA;
  }
  return QRR_OK;
}

qrr_status qrr_round_probe(const float* in, int64_t n, int32_t fmt, uint8_t* out, void* stream) {
  if (n < 0 || (fmt != 0 && fmt != 1)) return QRR_ERR_INVALID_ARG;
  if (n > 0 && (!in || !out)) return QRR_ERR_INVALID_ARG;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  return from_cuda(launch_round_probe(in, n, fmt, out, as_stream(stream)));
}

}  // extern "C"

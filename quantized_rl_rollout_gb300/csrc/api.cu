// C ABI of the library (include/qrr.h): host-side validation, workspace
// carving and dispatch to the kernels.  Nothing here allocates device memory
// or synchronizes with the host.
#include <stdlib.h>
#include <string.h>

#include "linear.cuh"
#include "quant.cuh"

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

// Linear workspace: t fp32 [M, r] (LoRA down projection).
size_t linear_ws_bytes(int64_t M, int64_t /*N*/, int64_t /*K*/, int32_t r) {
  if (M < 0 || r < 0) return 0;
  return round_up(static_cast<size_t>(M) * static_cast<size_t>(r) * sizeof(float)) + kAlign;
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
  float* t = static_cast<float*>(workspace);
  if (K == 0) return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(M * N) * 2, s));
  if (rr > 0) {
    cudaError_t e = launch_lora_down_simt(x, lora_A, M, K, rr, t, s);
    if (e != cudaSuccess) return QRR_ERR_CUDA;
  }
  LinearArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.codes = codes;
  a.scales = scales;
  a.tensor_scale = tensor_scale;
  a.A = static_cast<const uint16_t*>(lora_A);
  a.B = static_cast<const uint16_t*>(lora_B);
  a.t = t;
  a.y = y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.r = rr;
  a.lora_scale = rr > 0 ? alpha / static_cast<float>(rr) : 0.0f;
  return from_cuda(launch_linear_simt(a, s));
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

/*
 * qrr.h -- C ABI of the GB300 (sm_103a) low-precision linear-layer library
 * for RL rollout: NVFP4 W4A16 + BF16 LoRA linear, blockwise FP8 quantize +
 * GEMM, and re-quantization of all weights after a training step.
 *
 * Sources (page title, section):
 *  - "QeRL: Beyond Efficiency -- Quantization-enhanced Reinforcement Learning
 *    for LLMs", abstract: NVFP4 weights combined with LoRA speed up rollout.
 *  - "NVIDIA and MIT Collaborate on QeRL", Key Features and the paragraph
 *    after them: the policy's weight path moves to NVFP4 while logits and
 *    gradients stay in higher precision; prefill and decode both speed up.
 *  - "NVIDIA NeMo RL behaalt 48% snelheidswinst met end-to-end
 *    FP8-precisietraining", section "De technische doorbraak": blockwise E4M3
 *    with 128x128 weight tiles and 1x128 activation blocks, FP8 linear
 *    layers; section "Praktische prestatiewinsten": scales recalibrated after
 *    every training step; last paragraph before "Waarom dit belangrijk is":
 *    optional power-of-two scale factors.
 *
 * Formats.  The pages name NVFP4 but do not spell it out; this library uses
 * the standard layout: element code E2M1 (magnitudes 0, .5, 1, 1.5, 2, 3, 4,
 * 6; bit 3 = sign), two codes per byte with the even K index in the low
 * nibble; one E4M3 (FN) block scale per 16 consecutive elements of a row; one
 * FP32 tensor scale.  Element (n, k) decodes to
 * e2m1(code) * e4m3(scale[n][k/16]) * tensor_scale.  Quantization:
 *   s_t = amax(W) / 2688            (fp32, correctly rounded)
 *   s_b = e4m3_rne(amax_b / (6 * s_t))
 *   d_b = e4m3(s_b) * s_t
 *   code = e2m1_rne(x / d_b)        (x / d_b a correctly rounded fp32 quotient)
 * with round-to-nearest-even, saturation to the largest finite value, the
 * input's sign kept, all-zero codes where d_b == 0 and s_t == 0 for an
 * all-zero tensor.
 *
 * Conventions shared by every call.
 *  - All pointers except `descs` of qrr_requantize_weights are DEVICE
 *    pointers on the current CUDA device, owned by the caller.  The library
 *    allocates no memory; calls that need scratch take a caller-owned
 *    `workspace` whose size the matching *_workspace_bytes() query returns.
 *  - Matrices are row-major and contiguous.  Weights use nn.Linear
 *    orientation W[N = out][K = in], y = x . W^T; LoRA uses A[r][K], B[N][r].
 *  - bf16 / fp32 / byte pointers must be 16-byte aligned.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and never synchronizes with the host, except
 *    qrr_get_last_device_status, the one explicit sync point.  The tensor
 *    scale stays on the device, so quantize -> linear never round-trips.
 *  - Return value: QRR_OK, or an error detected on the host before anything
 *    is launched (invalid argument, unsupported shape, misalignment, small
 *    workspace), or QRR_ERR_CUDA when a launch fails.
 *  - `dev_status` (nullable, device int32): conditions found on the device are
 *    OR-ed into it (QRR_DEV_NONFINITE: a non-finite input was seen; the
 *    outputs are then unspecified; QRR_DEV_TIMEOUT: a tensor-core pipeline
 *    wait gave up after its bounded time and the kernel ended early).  The
 *    library never clears it; the caller zeroes it and reads it when it
 *    chooses (qrr_get_last_device_status).
 */
#ifndef QRR_H_
#define QRR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qrr_status {
  QRR_OK = 0,
  QRR_ERR_INVALID_ARG = 1,       /* null pointer, negative size, unknown enum value */
  QRR_ERR_UNSUPPORTED_SHAPE = 2, /* a size constraint of the call is not met */
  QRR_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned */
  QRR_ERR_WORKSPACE = 4,         /* workspace missing or smaller than the query says */
  QRR_ERR_CUDA = 5               /* a CUDA runtime call or a kernel launch failed */
} qrr_status;

/* Bits OR-ed into the optional device status word. */
#define QRR_DEV_NONFINITE 0x1 /* a non-finite input value was seen */
#define QRR_DEV_TIMEOUT 0x2   /* a pipeline wait gave up after its time limit; outputs unspecified */
#define QRR_DEV_SCALE_RANGE 0x4 /* QRR_SCALE_POW2 GEMM: a scale was not a power of two (or zero), or the
                                   exponents of one 128-K block spread wider than the native MMA's scale
                                   bytes can carry exactly; outputs are then inexact */
#define QRR_DEV_BAD_INDEX 0x8   /* an index read on the device (a token id) was out of range */

typedef enum qrr_scale_mode {
  QRR_SCALE_FP32 = 0, /* s = fp32(amax / 448); codes e4m3_rne(x / s) */
  QRR_SCALE_POW2 = 1  /* s = smallest power of two >= fp32(amax / 448); codes e4m3_rne(x * 2^-e) */
} qrr_scale_mode;

typedef enum qrr_format {
  QRR_FORMAT_NVFP4 = 0,   /* codes [N][K/2], E4M3 scales [N][K/16], fp32 tensor scale */
  QRR_FORMAT_FP8_W128 = 1 /* E4M3 codes [N][K], fp32 scales [ceil(N/128)][K/128] */
} qrr_format;

/* Human-readable name of a qrr_status value (static storage). */
const char* qrr_status_string(int status);

/* ABI version of this header (bumped on any signature change). */
int qrr_abi_version(void);

/* ------------------------------------------------------------------------ */
/* NVFP4 quantization of one bf16 weight ("QeRL: Beyond Efficiency",
 * abstract; layout and formula above).
 *   W            bf16 [N][K], K a multiple of 32, N >= 0
 *   codes        uint8 [N][K/2]  (out)
 *   scales       uint8 [N][K/16] (out, E4M3 bytes)
 *   tensor_scale fp32 [1]        (out, device)
 *   workspace    qrr_quantize_nvfp4_workspace_bytes() bytes of scratch
 * Two kernels on `stream`: a tensor-wide absmax sweep, then the encode sweep
 * (which reads the absmax from the workspace, no host round trip). */
size_t qrr_quantize_nvfp4_workspace_bytes(void);
qrr_status qrr_quantize_nvfp4(const void* W, int64_t N, int64_t K, uint8_t* codes, uint8_t* scales,
                              float* tensor_scale, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* W4A16 + LoRA linear ("NVIDIA and MIT Collaborate on QeRL", paragraph after
 * Key Features: NVFP4 weight path, activations/logits in higher precision;
 * "QeRL: Beyond Efficiency", abstract: NVFP4 with LoRA):
 *   y = x . W_hat^T + (alpha / r) . (x . A^T) . B^T,  y in bf16
 *   x            bf16 [M][K], M >= 0, K a multiple of 256 (the block-scale
 *                rows, K/16 bytes, are fetched by TMA, whose row pitch must be
 *                a multiple of 16 bytes)
 *   codes/scales/tensor_scale: an NVFP4 weight [N][K] as qrr_quantize_nvfp4 writes it
 *   lora_A       bf16 [r][K] or NULL;  lora_B bf16 [N][r] or NULL
 *   r            LoRA rank, 0..64 and a multiple of 8 when the adapter is on;
 *                the adapter is off when r == 0 or A or B is NULL
 *   y            bf16 [M][N] (out); N a multiple of 128
 *   workspace    qrr_linear_nvfp4_lora_workspace_bytes(M, N, K, r) bytes
 * Products are formed exactly and summed in fp32; the dequantized weight
 * e2m1 * e4m3 is exact in bf16.  A decode variant (split-K GEMV) is chosen
 * for M <= 64 and a tensor-core GEMM for larger M; both give the same
 * contract.  For M <= 8 the decode runs on the NVFP4 tensor-core MMA with
 * each token's x (scaled by a power of two so its largest value lies in
 * (3, 6]) carried as six E2M1 digit planes, sum_p d_p 6^-p: every value is
 * represented to within 6^-5 of the token's largest one (below bf16's own
 * half-ulp there), so outputs meet the same tolerance; powers of two are
 * exact. */
size_t qrr_linear_nvfp4_lora_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r);
qrr_status qrr_linear_nvfp4_lora(const void* x, int64_t M, int64_t K, const uint8_t* codes,
                                 const uint8_t* scales, const float* tensor_scale, int64_t N,
                                 const void* lora_A, const void* lora_B, int32_t r, float alpha,
                                 void* y, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* W4A16 + LoRA linear that allocates nothing.  The pages have no counterpart
 * to this call; it exists for callers that cannot get device memory of their
 * own: code that holds only the input and output buffers it was handed, such
 * as a plugin or FFI binding inside a host framework that owns every device
 * allocation and hands out no scratch, or a serving process that reserved its
 * whole HBM budget up front and has none left to give.
 *
 * Same arguments, contract and result as qrr_linear_nvfp4_lora, minus the
 * workspace.  Its scratch is a fixed block of QRR_NOALLOC_SCRATCH_BYTES of
 * device memory built into the library, which every GPU that loads the
 * library holds until the process exits.
 *  - Calls whose scratch need (qrr_linear_nvfp4_lora_workspace_bytes(M, N, K,
 *    r)) exceeds QRR_NOALLOC_SCRATCH_BYTES return QRR_ERR_WORKSPACE and launch
 *    nothing.
 *  - The first call on each device looks up the block's device address (with
 *    that device current) and keeps it for the life of the process; make that
 *    first call before any stream capture.  The address is kept per device
 *    number, so a device reset (cudaDeviceReset, or tearing down the primary
 *    context) while the library stays loaded is not supported.
 *  - Every call shares the block and it keeps the last call's contents (what
 *    must start at zero is cleared on the stream).  Calls that overlap on the
 *    GPU, on different streams or different host threads, race on it: order
 *    them on one stream or serialize them. */
#define QRR_NOALLOC_SCRATCH_BYTES (16u << 20)
size_t qrr_noalloc_scratch_bytes(void);
qrr_status qrr_linear_nvfp4_lora_noalloc(const void* x, int64_t M, int64_t K, const uint8_t* codes,
                                         const uint8_t* scales, const float* tensor_scale, int64_t N,
                                         const void* lora_A, const void* lora_B, int32_t r, float alpha,
                                         void* y, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Grouped W4A16 + LoRA linear: up to 8 independent layers that share the
 * token count M (a decoder layer's q/k/v/o/gate/up/down at one decode step),
 * run as one prologue launch and one persistent tensor-core launch whose work
 * units cover every layer, so small layers do not pay their own launch and
 * pipeline fill.  Each descriptor follows qrr_linear_nvfp4_lora's contract
 * (x [M][K], y [M][N], same alignment and shape rules); the result is the
 * same as calling it once per layer.
 *   descs      HOST array of `count` (1..8) descriptors, read during the call
 *   workspace  qrr_linear_nvfp4_lora_grouped_workspace_bytes(descs, count, M)
 * Returns QRR_ERR_UNSUPPORTED_SHAPE when count > 8. */
typedef struct qrr_linear_desc {
  const void* x;              /* bf16 [M][K] */
  int64_t N, K;
  const uint8_t* codes;       /* [N][K/2] */
  const uint8_t* scales;      /* [N][K/16] */
  const float* tensor_scale;  /* device scalar */
  const void* lora_A;         /* bf16 [r][K] or NULL */
  const void* lora_B;         /* bf16 [N][r] or NULL */
  int32_t r;
  float alpha;
  void* y;                    /* bf16 [M][N] */
} qrr_linear_desc;

size_t qrr_linear_nvfp4_lora_grouped_workspace_bytes(const qrr_linear_desc* descs, int32_t count, int64_t M);
qrr_status qrr_linear_nvfp4_lora_grouped(const qrr_linear_desc* descs, int32_t count, int64_t M,
                                         void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                         void* stream);

/* ------------------------------------------------------------------------ */
/* Blockwise FP8 quantization ("NVIDIA NeMo RL behaalt 48% ...", section "De
 * technische doorbraak": E4M3, 128x128 tiles for weights, 1x128 for
 * activations; power-of-two scales optional).
 * Weights:     W bf16 [N][K] -> q uint8 [N][K], scales fp32 [ceil(N/128)][K/128];
 *              K a multiple of 128, any N >= 0 (the last tile row may be short).
 * Activations: x bf16 [M][K] -> q uint8 [M][K], scales fp32 [M][K/128]; K % 128 == 0.
 * A block whose absmax is 0 gets scale 0 and all-zero codes. */
qrr_status qrr_quantize_fp8_w128x128(const void* W, int64_t N, int64_t K, uint8_t* q, float* scales,
                                     int32_t scale_mode, int32_t* dev_status, void* stream);
qrr_status qrr_quantize_fp8_a1x128(const void* x, int64_t M, int64_t K, uint8_t* q, float* scales,
                                   int32_t scale_mode, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Blockwise-scaled FP8 GEMM (same section: FP8 linear layers):
 *   y[m][n] = sum_kb sa[m][kb] * sw[n/128][kb] * sum_{k in kb} qa[m][k] * qw[n][k]
 *   qa uint8 [M][K], sa fp32 [M][K/128], qw uint8 [N][K], sw fp32 [ceil(N/128)][K/128]
 *   y  bf16 [M][N] (out); K a multiple of 128, N a multiple of 128.
 *   scale_mode  QRR_SCALE_FP32: any non-negative scales.  Each 128-wide block
 *               sum is formed by the tensor core in fp32, then multiplied by
 *               sa * sw and added in fp32 on the CUDA cores (promotion).
 *               QRR_SCALE_POW2: every scale is a power of two or zero (as
 *               QRR_SCALE_POW2 quantization writes them).  The product sa * sw
 *               is then applied by the tensor core itself: tcgen05.mma
 *               kind::mxf8f6f4 with one UE8M0 scale byte per 32 K of each row,
 *               and the whole K loop accumulates in one fp32 accumulator.  A
 *               scale that breaks the promise, or exponents within one 128-K
 *               block of a 128 x 256 output tile spread over more than 254
 *               binades, raise QRR_DEV_SCALE_RANGE (outputs then inexact).
 * The E4M3 products are exact; sums are fp32. */
qrr_status qrr_gemm_fp8_blockwise(const uint8_t* qa, const float* sa, const uint8_t* qw,
                                  const float* sw, int64_t M, int64_t N, int64_t K, void* y,
                                  int32_t scale_mode, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Re-quantize every weight after a training step ("NVIDIA NeMo RL behaalt
 * 48% ...", section "Praktische prestatiewinsten": scales recalibrated after
 * every step).  Each descriptor is quantized from scratch (current absmax, no
 * scale history), exactly as the single-tensor calls above would.
 *   descs   HOST array of `count` descriptors (read during the call only)
 *   format  QRR_FORMAT_NVFP4: codes/scales/tensor_scale as qrr_quantize_nvfp4
 *           QRR_FORMAT_FP8_W128: codes = q, scales = fp32 tile scales,
 *           tensor_scale unused (may be NULL); scale_mode as for FP8
 *   workspace qrr_requantize_workspace_bytes(count) bytes (NVFP4 only; FP8 needs none)
 * All descriptors are processed by grouped launches (one absmax sweep and one
 * encode sweep for NVFP4, one sweep for FP8), not one launch per tensor. */
typedef struct qrr_weight_desc {
  const void* W;       /* bf16 [N][K] */
  int64_t N;
  int64_t K;
  uint8_t* codes;      /* NVFP4 codes [N][K/2] or FP8 codes [N][K] */
  void* scales;        /* NVFP4 uint8 [N][K/16] or FP8 fp32 [ceil(N/128)][K/128] */
  float* tensor_scale; /* NVFP4 only */
} qrr_weight_desc;

size_t qrr_requantize_workspace_bytes(int32_t count);
qrr_status qrr_requantize_weights(const qrr_weight_desc* descs, int32_t count, int32_t format,
                                  int32_t scale_mode, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Backward pass of the W4A16 + LoRA linear through the frozen NVFP4 weight
 * ("NVIDIA and MIT Collaborate on QeRL", Key Features, "Stable
 * Backpropagation": only the adapter is trained, its gradients stay precise;
 * "Jet-RL: Enabling On-Policy FP8 RL ...", Quick Overview: the backward pass
 * stays in BF16).  For the forward y = x . W_hat^T + (alpha/r) (x . A^T) . B^T
 * and the upstream gradient dY:
 *   dX = dY . W_hat + (alpha/r) (dY . B) . A      bf16 [M][K]
 *   dA = (alpha/r) (dY . B)^T . x                 fp32 [r][K]
 *   dB = (alpha/r) dY^T . (x . A^T)               fp32 [N][r]
 *   dy    bf16 [M][N];  x bf16 [M][K] (the forward's input; only read with an adapter)
 *   codes/scales/tensor_scale: the frozen NVFP4 weight [N][K]
 *   lora_A bf16 [r][K], lora_B bf16 [N][r] (both NULL or r == 0: no adapter,
 *          dA / dB untouched and may be NULL)
 *   workspace  qrr_lora_backward_workspace_bytes(M, N, K, r) bytes (it holds
 *          the weight's bf16 transpose, K x N x 2 bytes, among others)
 * Shapes as the forward: K % 256 == 0, N % 128 == 0, r <= 64 and r % 8 == 0.
 * The weight's e2m1 x e4m3 part is exact in bf16 and its tensor scale is
 * applied in fp32; products are exact and sums fp32 (the rank-r projections
 * carried as bf16 (high, low) pairs, about 2^-17 relative).  dA and dB are
 * summed over token slices in a fixed order: results do not depend on
 * timing. */
size_t qrr_lora_backward_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r);
qrr_status qrr_lora_backward_nvfp4(const void* dy, int64_t M, int64_t N, const void* x, int64_t K,
                                   const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                                   const void* lora_A, const void* lora_B, int32_t r, float alpha, void* dx, float* dA,
                                   float* dB, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                   void* stream);

/* ------------------------------------------------------------------------ */
/* FP8 key/value cache and decode attention ("NVIDIA NeMo RL behaalt 48% ...",
 * section "Praktische prestatiewinsten": FP8 extended to the KV cache and the
 * attention operations; section "De technische doorbraak": 1x128 E4M3 blocks
 * for activations).  Each cached row (one token, one KV head, head_dim 128)
 * is E4M3 codes with one fp32 scale, quantized by the 1x128 rule of
 * qrr_quantize_fp8_a1x128 (scale_mode as there).
 * Layout: caches uint8 [B][Hkv][Lmax][128], scales fp32 [B][Hkv][Lmax];
 * queries and outputs bf16 [B][Hq][128]; query head h reads KV head
 * h / (Hq / Hkv).
 *
 * qrr_kv_append_fp8: quantizes one decode step's rows k_new, v_new (bf16
 * [B][Hkv][128]) into slot pos[b] of sequence b (int32 [B]); a slot outside
 * [0, Lmax) raises QRR_DEV_BAD_INDEX and writes nothing; a non-finite value
 * raises QRR_DEV_NONFINITE.  k_new / v_new 8-byte aligned, caches 16-byte.
 *
 * qrr_attention_decode_fp8: o[b][h] = softmax(q[b][h] . K^T / sqrt(128)) . V
 * over the first lens[b] cached tokens of sequence b (lens int32 [B], at most
 * Lmax; 0 gives a zero row).  Hq / Hkv in {1, 2, 4, 8}; Lmax % 4 == 0.  The
 * codes convert exactly; scores and sums are fp32, exponentials the base-2
 * hardware approximation; the sequence is split in 256-token pieces whose
 * partial results are merged in a fixed order.  Workspace:
 * qrr_attention_decode_fp8_workspace_bytes(B, Hq, Lmax). */
qrr_status qrr_kv_append_fp8(const void* k_new, const void* v_new, int32_t B, int32_t Hkv, const int32_t* pos,
                             uint8_t* k_cache, float* k_scales, uint8_t* v_cache, float* v_scales, int32_t Lmax,
                             int32_t scale_mode, int32_t* dev_status, void* stream);
size_t qrr_attention_decode_fp8_workspace_bytes(int32_t B, int32_t Hq, int32_t Lmax);
qrr_status qrr_attention_decode_fp8(const void* q, int32_t B, int32_t Hq, int32_t Hkv, const uint8_t* k_cache,
                                    const float* k_scales, const uint8_t* v_cache, const float* v_scales,
                                    const int32_t* lens, int32_t Lmax, void* out, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Token log-probabilities and token-level importance-sampling weights
 * ("NVIDIA NeMo RL behaalt 48% ...", the paragraph on importance sampling in
 * "Waarom dit belangrijk is voor AI-economie": the shift between the
 * generation engine's and the trainer's token distributions is corrected
 * token by token):
 *   logp[t] = logits[t][tok[t]] - log(sum_v exp(logits[t][v]))
 *   w[t]    = min(exp(logp[t] - rollout_logp[t]), cap)   (cap <= 0: no cap)
 *   logits        bf16 [T][V] row-major (V >= 1); read once
 *   tokens        int32 [T]; a negative id marks padding (logp = w = 0); an id
 *                 >= V also gives 0 and raises QRR_DEV_BAD_INDEX
 *   rollout_logp  fp32 [T] (the rollout engine's log-probabilities) or NULL
 *   logp          fp32 [T] (out)
 *   w             fp32 [T] (out; only written when rollout_logp is given)
 * The sums are fp32; exp and log are the hardware base-2 approximations
 * (relative error about 2^-22).  A NaN or +inf logit raises
 * QRR_DEV_NONFINITE.  Pointers 16-byte aligned (logits; 4-byte for the
 * others); V % 8 == 0 takes 16-byte loads, any other V element loads. */
qrr_status qrr_token_logprobs_is(const void* logits, int64_t T, int64_t V, const int32_t* tokens,
                                 const float* rollout_logp, float cap, float* logp, float* w, int32_t* dev_status,
                                 void* stream);

/* ------------------------------------------------------------------------ */
/* The explicit sync point for device-detected conditions: copies the status
 * word `dev_status` (device int32, as passed to the calls above) into
 * `*host_out` once every call queued on `stream` before it has finished, then
 * returns.  It blocks the calling host thread on `stream` (the only call of
 * the library that does) and does not clear the word.  QRR_ERR_INVALID_ARG for
 * a NULL pointer, QRR_ERR_CUDA when the copy or the stream fails (an error of
 * an earlier kernel on the stream surfaces here). */
qrr_status qrr_get_last_device_status(int32_t* host_out, const int32_t* dev_status, void* stream);

/* One query for every call's scratch need, by operation:
 *   QRR_OP_QUANTIZE_NVFP4      (sizes unused)
 *   QRR_OP_LINEAR_NVFP4_LORA   M tokens, N outputs, K inputs, LoRA rank r
 *   QRR_OP_REQUANTIZE_WEIGHTS  M = number of descriptors
 *   QRR_OP_QUANTIZE_FP8, QRR_OP_GEMM_FP8: no scratch (0)
 *   QRR_OP_LORA_BACKWARD       M tokens, N outputs, K inputs, LoRA rank r
 * It returns the same value as the per-call query; 0 for an unknown op or
 * invalid sizes. */
typedef enum qrr_op {
  QRR_OP_QUANTIZE_NVFP4 = 0,
  QRR_OP_LINEAR_NVFP4_LORA = 1,
  QRR_OP_REQUANTIZE_WEIGHTS = 2,
  QRR_OP_QUANTIZE_FP8 = 3,
  QRR_OP_GEMM_FP8 = 4,
  QRR_OP_LORA_BACKWARD = 5
} qrr_op;
size_t qrr_workspace_bytes(int32_t op, int64_t M, int64_t N, int64_t K, int32_t r);

/* Host-only query of how a decode call (qrr_linear_nvfp4_lora_grouped at
 * 1 <= M <= 64 tokens) divides its work among `grid` CTAs; it launches
 * nothing and needs no GPU.  Every tile (128 weight rows of one layer, all M
 * tokens) is a sequence of K / 256 weight stages followed, when the layer
 * has an adapter (r > 0), by one LoRA stage.  Up to 32 tokens the stages of
 * all tiles, layer after layer, are cut into equal contiguous ranges, one
 * per CTA (stream-K); above, each layer's K is split into equal pieces and
 * the pieces go to the CTAs longest first.
 *   count        layers, 1..8; N[j] % 128 == 0, K[j] % 256 == 0, K[j] > 0,
 *                N[j] > 0, r[j] in {0} or a multiple of 8 up to 64
 *   grid         CTAs offered, 1..160 (fewer are used when there are fewer
 *                stages); *grid_used receives the number used
 *   units        host [max_units][2] uint32: word 0 = layer (bits 0-3), m tile
 *                (4-7), n tile (8-23), the tile's piece count (24-31);
 *                word 1 = first K stage (0-11), K stages (12-22), piece index
 *                within the tile (23-30), LoRA stage (31)
 *   offsets      host [grid + 1]: CTA b takes units offsets[b] .. offsets[b+1]
 * Returns the number of units, or a negative qrr_status (invalid argument,
 * unsupported shape, or a table larger than max_units). */
int64_t qrr_plan_decode_units(int64_t M, int32_t count, const int64_t* N, const int64_t* K, const int32_t* r,
                              int32_t grid, uint32_t* units, int32_t max_units, uint16_t* offsets,
                              int32_t* grid_used);

/* Probe of the bounded-wait path.  Every tensor-core pipeline wait of the
 * library gives up after a bounded time (about 2 s), raises QRR_DEV_TIMEOUT,
 * lets its CTA drain its copies, free its tensor memory and exit, so a broken
 * pipeline ends the kernel instead of hanging the GPU.  This launches one CTA
 * that allocates tensor memory and waits, through that same bounded wait, on
 * a barrier with a give-up time of `limit_cycles` SM clock cycles
 * (1 .. about 4e9).  arrive = 0: nothing arrives, so the wait runs out and
 * QRR_DEV_TIMEOUT is OR-ed into *dev_status; arrive = 1: the barrier is
 * completed first and nothing is flagged.  `cycles` (nullable, device int64)
 * receives the wait's duration in SM cycles.  The context stays usable
 * either way. */
qrr_status qrr_wait_probe(int64_t limit_cycles, int32_t arrive, int32_t* dev_status, int64_t* cycles, void* stream);

/* Memory-system probe: the floor of one pass over a byte matrix, to set
 * beside the decode kernels, which read a weight's packed codes the same way.
 * `data` u8 [rows][row_bytes] (device, 16-byte aligned, rows and row_bytes
 * multiples of 128) goes through an 8-stage shared-memory ring of
 * [128 x 128 B] TMA boxes, one CTA per SM, each a contiguous range of boxes
 * (row tiles outer, 128-byte column tiles inner), with no arithmetic on the
 * bytes.  Nothing is written.  A bounded wait that runs out sets
 * QRR_DEV_TIMEOUT in *dev_status (nullable). */
qrr_status qrr_stream_probe(const void* data, int64_t rows, int64_t row_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Re-quantization with adaptive quantization noise ("QeRL: Beyond Efficiency
 * -- Quantization-enhanced Reinforcement Learning for LLMs", Abstract: noise
 * in the quantized policy raises its entropy and helps exploration; the
 * Adaptive Quantization Noise mechanism adjusts it during training).  The
 * page gives no formula; this library's reading: each master is made noisy
 * before it is quantized,
 *   W'[e] = bf16_rn(fp32(W[e]) + fp32(sigma * z[e]))
 * and W' is quantized exactly as qrr_requantize_weights would (same formats,
 * scale modes, workspace, grouping).  z[e] is a standardized sum of four
 * uniforms (mean 0, variance about 1, within +-2 sqrt 3) drawn from
 * Philox4x32-10 (Salmon et al., SC'11) at counter (e / 4 low word, e / 4 high
 * word, descriptor index j, step), key (seed low word, seed high word): the
 * four bytes k_i of output word r[e % 4] give
 * z = fp32((k1 + k2 + k3 + k4 - 510) / 256) * fp32(sqrt 3).  e is the
 * element's row-major index in its tensor.  Every step is integer or one
 * correctly rounded fp32 operation, so the result is reproducible bit for bit.
 * The noise is regenerated from its counter in every pass: nothing noisy is
 * stored.  sigma >= 0 and finite (0: plain re-quantization), step >= 0. */
qrr_status qrr_requantize_weights_aqn(const qrr_weight_desc* descs, int32_t count, int32_t format,
                                      int32_t scale_mode, float sigma, uint64_t seed, int32_t step, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream);

/* The noise strength of a training step under a geometric schedule from
 * sigma_start (step 0) to sigma_end (step steps - 1 and later):
 *   sigma_start * (sigma_end / sigma_start) ^ (step / (steps - 1)),
 * computed in double precision and rounded to fp32.  Host only. */
float qrr_aqn_sigma(int32_t step, int32_t steps, double sigma_start, double sigma_end);

/* Conformance probe of the noise: z of elements start .. start + n - 1 of
 * descriptor index `tensor` at `step` with `seed`, written to out fp32 [n]. */
qrr_status qrr_aqn_noise_probe(float* out, int64_t n, int64_t start, uint64_t seed, int32_t tensor, int32_t step,
                               void* stream);

/* ------------------------------------------------------------------------ */
/* Conformance probe: the library's own float32 -> E2M1 / E4M3 rounding
 * primitive applied to n values (fmt 0 = E2M1 code in the low 4 bits,
 * fmt 1 = E4M3 byte).  in fp32 [n], out uint8 [n]; n >= 0.  The quantizers
 * take every rounding decision through this primitive, so a test can compare
 * it with the format definition value by value. */
qrr_status qrr_round_probe(const float* in, int64_t n, int32_t fmt, uint8_t* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QRR_H_ */

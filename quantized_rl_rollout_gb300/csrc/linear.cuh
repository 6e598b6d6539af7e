// Argument block and launchers of the linear-path kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda.h>

#include "common.cuh"

namespace qrr {

// ---- tensor-core W4A16 linear (linear_tc.cu) ----

constexpr int kMaxW4Layers = 8;

struct W4Layer {
  CUtensorMap tx;      // x (bf16) or its f16 image [M, K], box [BN (BN/2 for a CTA pair), 64], 128 B swizzle
  CUtensorMap tcodes;  // packed codes u8 [N, K/2], box [128, 32]
  CUtensorMap tt;      // LoRA t' bf16 [M, 64 * lora_chunks], box as tx, 128 B swizzle
  CUtensorMap tscales;  // block scales u8 [N, K/16], box [128, 16] (256-wide K stages)
  CUtensorMap tb;       // decode: LoRA B bf16 [N, r], box [128, r], into the LoRA stage's code slot
  CUtensorMap tp;       // decode on E2M1 planes: x planes u8 [kXPlanes * ms, K/2], box [nmma, 128], 128 B swizzle
  const uint8_t* scales;
  const float* tensor_scale;
  const uint16_t* B;  // LoRA B [N, r], r <= 64
  const int* pexp;    // per-token power-of-two pre-scale (decode) or null
  __nv_bfloat16* y;
  float* partial;      // [splits, M, N] when splits > 1
  uint32_t* counters;  // [m_tiles * n_tiles], zero before the launch
  int M, N, K, r, lora_chunks;
  int n_tiles, m_tiles, splits, kcps;  // kcps: pipeline stages (BK-wide K slices) per split
  int first_unit;
};

// Unit table of a decode launch: CTA b takes units
// unit[unit_off[b] .. unit_off[b + 1]) in that order, each a contiguous piece
// of one tile's stage sequence (a stream-K range, or one split of a per-layer
// split-K).  Word 0: layer (4 bits), m tile (4), n tile (16), the tile's
// piece count (8); word 1: first K stage (12), K stages (11), the piece's
// index within its tile (8), LoRA stage (1).  Without a table (use_table 0)
// the units go round-robin.
constexpr int kMaxTableUnits = 1024;
constexpr int kMaxTableCtas = 160;

struct W4Params {
  W4Layer layer[kMaxW4Layers];
  int count;
  int total_units;
  int32_t* status;
  int use_table, table_grid;
  uint16_t unit_off[kMaxTableCtas + 1];
  uint32_t unit[kMaxTableUnits][2];
};

// The stream-K cut of a decode launch over `grid` CTAs: the stages of every
// tile (its K stages, then its LoRA stage), tile after tile and layer after
// layer, in `grid` ranges of equal length.  kc / nl / tiles per layer;
// writes the units and offsets when `p` is given, and each layer's largest
// piece count.  Returns the number of units, or -1 when a field does not fit
// its bits or the table is too small.
int stream_k_units(const int* kc, const int* nl, const int* n_tiles, const int* m_tiles, int count, int grid,
                   W4Params* p, int* max_pieces);
// The units of a launch with per-layer splits (L.splits, L.kcps), given to
// `grid` CTAs longest first, as a unit table; leaves p.use_table 0 when the
// table cannot hold them.
void lpt_units(W4Params& p, int bk, int grid);
// CTAs of a decode launch (the SM count of the current device).
int decode_grid();

// Prologue of one layer (lora_tc.cu): the LoRA down projection on the tensor
// cores into t' (ks > 1: split over K slices of slice_steps x 64 with fp32
// partials and a ticket per 128-token tile), and, when x16 is set, the f16
// image of x with its per-token pre-scales.
struct LoraDownLayer {
  CUtensorMap tx;  // x bf16 [M, K], box [128, 64], 128 B swizzle
  CUtensorMap ta;  // LoRA A bf16 [r, K], box [R, 64], 128 B swizzle
  __nv_bfloat16* t;  // [M, t_cols]
  const float* tensor_scale;
  float* tpart;        // [M, r, ks rounded up to 4] fp32 partials (ks > 1)
  uint32_t* tickets;   // [ceil(M / 128)], zero before the launch (ks > 1)
  const uint16_t* x;   // bf16 [M, K] (x rows)
  __half* x16;         // f16 [M, K], or null for no x-row CTAs
  int* pexp;           // [M]
  int M, K, r, R, t_cols;  // R: r rounded up to a multiple of 16
  int ks, slice_steps;     // K slices and 64-wide steps per slice
  int x_rows_per_cta;      // set by the launcher
  float lora_scale;
  int first_cta;
};

struct LoraDownBatch {
  LoraDownLayer l[kMaxW4Layers];
  int count;
  int32_t* status;
};

cudaError_t launch_lora_down_tc(LoraDownBatch& b, cudaStream_t stream);

// Decode prologue (decode_prologue.cu), at most 64 tokens: per layer one
// cluster of CTAs over K slices writes x16 / pexp and t' (the cluster sums
// its slices through distributed shared memory), and the launch clears the
// GEMM's split-K tile counters.
struct DecodeProLayer {
  const uint16_t* x;  // bf16 [M, K]
  const uint16_t* A;  // LoRA A bf16 [r, K] (r > 0)
  __half* x16;        // f16 [M, K], or null when `planes` is set
  uint8_t* planes;    // E2M1 digit planes [kXPlanes * ms, K/2] (see kXPlanes below), or null
  int ms;             // token rows per plane (planes only)
  int* pexp;          // [M]
  __nv_bfloat16* t;   // [M, t_cols] (r > 0)
  const float* tensor_scale;
  int M, K, r, R, t_cols;  // R: r rounded up to a multiple of 16 (0 without an adapter)
  float lora_scale;
  int first_cta;  // set by the launcher
};

struct DecodeProBatch {
  DecodeProLayer l[kMaxW4Layers];
  int count;
  uint32_t* clear;  // words zeroed by the launch (the GEMM's tile counters), or null
  int clear_words;
  int32_t* status;
  int xr, stages, ks;  // set by the launcher
};

cudaError_t launch_decode_prologue(DecodeProBatch& b, cudaStream_t stream);

// ---- decode on the native NVFP4 MMA (w4_decode_nvf4.cu) ----
// Each token's activations, scaled by the power of two 2^-e_m that brings
// max_k |x[m, k]| into (3, 6], are written as kXPlanes E2M1 digit planes
// d_0 .. d_5 with x 2^-e = sum_p d_p 6^-p + rest, |rest| <= 6^-5: d_p is the
// round-to-nearest-even E2M1 value of the running residual, which is then
// (residual - d_p) 6 (each step exact or within an fp32 rounding).  Plane
// row p * ms + m holds token m's digits of plane p, packed like the weight
// codes (element k in the low nibble of byte k / 2 when k is even).
constexpr int kXPlanes = 6;

// Launch geometry of the plane decode for M tokens, the same on host and
// device: ms token rows per plane (1, else M rounded up to 8); rows = the
// plane rows of a stage (kXPlanes * ms rounded up to 16, to 32 when they are
// split), taken by nh MMAs of N = nmma each (N <= 256); bn = token rows of
// the t' box (the LoRA MMA's N); the stage layout (x/t' slot of xb bytes,
// then 16 KB of codes and 2 KB of block scales); and the tensor-memory map
// (nd accumulators of `rows` columns, 64 columns of LoRA A, 16 of B scales,
// then sf_slots groups of 16 columns of A scales).
struct Nvf4Geo {
  int ms, rows, nh, nmma, bn, xb, stage, stages, nd, lora0, sfb0, sf0, sf_slots;
};

__host__ __device__ inline Nvf4Geo nvf4_geo(int M) {
  Nvf4Geo g{};
  g.ms = M <= 1 ? 1 : (M + 7) / 8 * 8;
  g.rows = (kXPlanes * g.ms + 15) / 16 * 16;
  g.nh = g.rows > 256 ? 2 : 1;
  if (g.nh == 2) g.rows = (g.rows + 31) / 32 * 32;
  g.nmma = g.rows / g.nh;
  g.bn = M <= 16 ? 16 : M <= 32 ? 32 : 64;
  const int xrows = g.rows > 2 * g.bn ? g.rows : 2 * g.bn;
  g.xb = (xrows * 128 + 1023) / 1024 * 1024;
  g.stage = g.xb + 128 * 128 + 128 * 16;
  g.stages = (220 * 1024) / g.stage;
  g.stages = g.stages > 8 ? 8 : g.stages;
  g.nd = 2 * g.rows + 64 + 16 + 2 * 16 <= 512 ? 2 : 1;
  g.lora0 = (g.nd * g.rows + 63) / 64 * 64;
  g.sfb0 = g.lora0 + 64;
  g.sf0 = g.sfb0 + 16;
  g.sf_slots = (512 - g.sf0) / 16;
  g.sf_slots = g.sf_slots > 8 ? 8 : g.sf_slots;
  return g;
}

// The plane decode takes at most this many tokens (above it, the dequant
// kernel on its f16 operand path, up to 64).
constexpr int kNvf4MaxM = 8;

// Decode GEMM over the unit table in `p` (use_table set): codes and block
// scales by TMA straight into the block-scaled MMA, x as its digit planes,
// the LoRA stage as a kind::f16 MMA into plane 0's columns.
cudaError_t launch_w4_decode_nvf4(const W4Params& p, cudaStream_t stream);

int w4_bn_for(int64_t M);
int w4_bk_for(int64_t M);
// pair: 256-token tiles run on 2-CTA clusters, each cluster two adjacent
// 128-row tiles (every layer's n_tiles even; x / t' maps with 128-row boxes).
cudaError_t launch_w4a16_tc(W4Params& p, int bn, bool f16, bool pair, bool after_prologue, cudaStream_t stream);

struct Fp8GemmArgs {
  const uint8_t* qa;  // [M, K]
  const float* sa;    // [M, K/128]
  const uint8_t* qw;  // [N, K]
  const float* sw;    // [ceil(N/128), K/128]
  void* y;            // bf16 [M, N]
  int64_t M, N, K;
};

cudaError_t launch_fp8_gemm_tc(const Fp8GemmArgs& a, int32_t* status, cudaStream_t stream);
// power-of-two scales on the native block-scaled MMA (gemm_fp8_mx.cu)
cudaError_t launch_fp8_gemm_mx(const Fp8GemmArgs& a, int32_t* status, cudaStream_t stream);

// ---- bf16 GEMM with an extra contraction block (gemm_bf16_tc.cu) ----
// y[m, c] = g (sum_n A[m, n] B[c, n] + sum_j A2[m, j] B2[c, j]); all K-major
// bf16, y bf16 [M, C]; K, K2 multiples of 64, C a multiple of 128.
struct Bf16GemmArgs {
  const void* A;   // [M, K]
  const void* B;   // [C, K]
  const void* A2;  // [M, K2] or null (K2 = 0)
  const void* B2;  // [C, K2]
  const float* g;  // device scalar (1 when null or 0)
  void* y;
  int64_t M, C, K, K2;
};
cudaError_t launch_gemm_bf16_tc(const Bf16GemmArgs& a, int32_t* status, cudaStream_t stream);

// ---- LoRA backward helpers (lora_bwd.cu) ----
cudaError_t launch_lora_backward_prep(const uint8_t* codes, const uint8_t* scales, const void* A, const void* B,
                                      int N, int K, int r, int t_cols, __nv_bfloat16* wt, uint16_t* at2, uint16_t* bt,
                                      cudaStream_t stream);
int lora_grad_slices(int64_t M, int64_t C);
cudaError_t launch_lora_grad(const void* X, const uint16_t* tp, int M, int C, int r, int t_cols,
                             const float* tensor_scale, bool transposed, float* part, float* out,
                             cudaStream_t stream);

// ---- FP8 key/value cache and decode attention (attention_fp8.cu) ----
int attn_splits(int Lmax);
cudaError_t launch_kv_append_fp8(const void* k_new, const void* v_new, int B, int Hkv, const int32_t* pos, int Lmax,
                                 uint8_t* kc, float* ksc, uint8_t* vc, float* vsc, int mode, int32_t* status,
                                 cudaStream_t stream);
cudaError_t launch_attention_decode_fp8(const void* q, const uint8_t* kc, const float* ksc, const uint8_t* vc,
                                        const float* vsc, const int32_t* lens, int B, int Hq, int Hkv, int Lmax,
                                        void* out, float* pm, float* pl, float* po, int32_t* status,
                                        cudaStream_t stream);

// ---- token log-probabilities and importance-sampling weights (rollout_is.cu) ----
cudaError_t launch_token_logprob_is(const void* logits, int64_t T, int64_t V, const int32_t* tokens,
                                    const float* rollout_logp, float cap, float* logp, float* w, int32_t* status,
                                    cudaStream_t stream);

// ---- probe of the bounded-wait path (probe.cu) ----
// limit: give-up time of the wait in SM clock cycles; arrive: complete the
// barrier before waiting; cycles (nullable, device): the wait's duration.
cudaError_t launch_wait_probe(long long limit, int arrive, int32_t* status, long long* cycles, cudaStream_t stream);
// A TMA stream of [128 x 128 B] boxes over a byte matrix with no arithmetic (probe.cu).
cudaError_t launch_stream_probe(const void* data, int64_t rows, int64_t row_bytes, int32_t* status,
                                cudaStream_t stream);

}  // namespace qrr

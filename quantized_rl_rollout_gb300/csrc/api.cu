// C ABI of the library (include/qrr.h): host-side validation, workspace
// carving and dispatch to the kernels.  Nothing here allocates device memory,
// and only qrr_get_last_device_status (the explicit sync point) synchronizes
// with the host.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include <algorithm>

#include "linear.cuh"
#include "quant.cuh"
#include "tc.cuh"

#include <cuda_fp16.h>

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

// One layer of a (grouped) linear call, as the caller describes it.
struct LinIn {
  const void* x;
  int64_t N, K;
  const uint8_t* codes;
  const uint8_t* scales;
  const float* tensor_scale;
  const void* A;
  const void* B;
  int32_t r;  // effective rank (0 = no adapter)
  float alpha;
  void* y;
};

// How a linear call runs: operand type, token tile, per-layer split-K and the
// workspace carve-up.  Every layer of a call shares the token count M.
struct LinPlan {
  bool f16;
  bool pair;  // 256-token tiles on CTA pairs (2-CTA clusters), each pair two 128-row tiles
  int bn, bk, m_tiles, count;
  bool sk;  // decode with a stream-K table (else one unit per tile)
  bool nvf4;  // decode on the native NVFP4 MMA with x as E2M1 digit planes (the stream-K sizes)
  struct Layer {
    int n_tiles, splits, kcps, lora_chunks;
    size_t t_off, x16_off, p_off, part_off, cnt_off;
  } l[kMaxW4Layers];
  size_t cnt_begin, cnt_bytes, total;
};

// Decode (<= 64 tokens) takes the f16 operand path.  Up to 32 tokens the
// stages of all its tiles are cut into one contiguous range per SM
// (stream-K): a tile split across CTAs writes fp32 partials, one slot per
// piece, and the piece that finishes last sums them in piece order.  At more
// tokens a partial costs as much as a few stages, so K is split per layer by
// a length that fills whole waves of the SMs (each layer's partials capped at
// about a quarter of its weight bytes) and the units go to the CTAs longest
// first.  Prefill runs one unit per tile.
LinPlan plan_linear(int64_t M, const LinIn* in, int count) {
  LinPlan p{};
  const bool decode = M <= 64;
  p.f16 = decode;
  p.bn = w4_bn_for(M);
  p.bk = w4_bk_for(M);
  p.m_tiles = static_cast<int>((M + p.bn - 1) / p.bn);
  p.count = count;
  int kc[kMaxW4Layers], cap[kMaxW4Layers], maxkc = 1;
  for (int j = 0; j < count; ++j) {
    p.l[j].n_tiles = static_cast<int>(in[j].N / 128);
    p.l[j].lora_chunks = in[j].r > 0 ? static_cast<int>((2 * in[j].r + 63) / 64) : 0;
    kc[j] = std::max(1, static_cast<int>(in[j].K / p.bk));
    cap[j] = decode ? std::max<int>(1, static_cast<int>(0.035 * static_cast<double>(in[j].K) /
                                                        static_cast<double>(std::max<int64_t>(M, 1))))
                    : 1;
    maxkc = std::max(maxkc, kc[j]);
    p.l[j].splits = 1;
    p.l[j].kcps = kc[j];
  }
  // Prefill tiles of 256 tokens run on CTA pairs when every layer has an even
  // number of 128-row tiles: the pair's MMA reads each CTA's half of the
  // token tile, so each SM streams half of x.
  p.pair = !decode && p.bn == 256;
  for (int j = 0; j < count; ++j) p.pair = p.pair && p.l[j].n_tiles % 2 == 0;
  if (decode && M <= 32) {
    // the layers the launch will carry (those with N and K), as it will
    int skc[kMaxW4Layers], nl[kMaxW4Layers], nt[kMaxW4Layers], mt[kMaxW4Layers], pieces[kMaxW4Layers];
    int idx[kMaxW4Layers];
    int n = 0;
    for (int j = 0; j < count; ++j) {
      if (in[j].N == 0 || in[j].K == 0) continue;
      skc[n] = static_cast<int>(in[j].K / p.bk);
      nl[n] = in[j].r > 0 ? 1 : 0;
      nt[n] = p.l[j].n_tiles;
      mt[n] = p.m_tiles;
      idx[n++] = j;
    }
    p.sk = stream_k_units(skc, nl, nt, mt, n, decode_grid(), nullptr, pieces) >= 0;
    if (p.sk)
      for (int i = 0; i < n; ++i) p.l[idx[i]].splits = pieces[i];  // partial slots
    p.nvf4 = p.sk && M <= kNvf4MaxM;
  }
  if (decode && !p.sk) {
    // Cost model in pipeline stages: a unit costs its K stages plus its
    // epilogue (about half a stage, or three when it writes a split-K partial
    // and may run the reduction); units go round-robin to the SMs, so the
    // makespan is bounded by waves x the costliest unit.
    double best = -1.0;
    for (int ul = maxkc; ul >= 1; --ul) {
      double work = 0.0, worst = 0.0;
      int units = 0;
      int sp[kMaxW4Layers];
      for (int j = 0; j < count; ++j) {
        int s = std::min((kc[j] + ul - 1) / ul, std::min(cap[j], kc[j]));
        const int kcps = (kc[j] + s - 1) / s;
        s = (kc[j] + kcps - 1) / kcps;
        sp[j] = s;
        const int base = p.l[j].n_tiles * p.m_tiles;
        units += base * s;
        work += static_cast<double>(base) * kc[j];
        worst = std::max(worst, kcps + (s > 1 ? 3.0 : 0.5));
      }
      const int waves = (units + kSMs - 1) / kSMs;
      const double eff = work / (static_cast<double>(kSMs) * waves * worst);
      if (eff > best + 1e-9) {
        best = eff;
        for (int j = 0; j < count; ++j) {
          p.l[j].splits = sp[j];
          p.l[j].kcps = (kc[j] + sp[j] - 1) / sp[j];
        }
      }
    }
  }
  size_t off = 0;
  for (int j = 0; j < count; ++j) {
    LinPlan::Layer& L = p.l[j];
    L.t_off = off;
    off += round_up(static_cast<size_t>(M) * 64 * L.lora_chunks * 2);
    L.x16_off = off;  // the f16 image of x, or its digit planes
    if (p.nvf4)
      off += round_up(static_cast<size_t>(kXPlanes) * nvf4_geo(static_cast<int>(M)).ms *
                      static_cast<size_t>(in[j].K) / 2);
    else if (p.f16)
      off += round_up(static_cast<size_t>(M) * static_cast<size_t>(in[j].K) * 2);
    L.p_off = off;
    if (p.f16) off += round_up(static_cast<size_t>(M) * 4);
    L.part_off = off;
    if (L.splits > 1) off += round_up(static_cast<size_t>(L.splits) * M * in[j].N * 4);
  }
  // split-K tile counters: one block, cleared per call by the decode prologue
  p.cnt_begin = off;
  for (int j = 0; j < count; ++j) {
    p.l[j].cnt_off = off;
    off += static_cast<size_t>(p.m_tiles) * p.l[j].n_tiles * 4;
  }
  p.cnt_bytes = off - p.cnt_begin;
  p.total = round_up(off) + kAlign;
  return p;
}

// Host-side checks shared by the single and grouped linear calls.
qrr_status check_linear(const LinIn& a, int64_t M, const void* A_in, const void* B_in, int32_t r_in) {
  if (a.N < 0 || a.K < 0 || r_in < 0) return QRR_ERR_INVALID_ARG;
  if (!a.tensor_scale) return QRR_ERR_INVALID_ARG;
  if (M * a.N > 0 && !a.y) return QRR_ERR_INVALID_ARG;
  if (M * a.K > 0 && !a.x) return QRR_ERR_INVALID_ARG;
  if (a.N * a.K > 0 && (!a.codes || !a.scales)) return QRR_ERR_INVALID_ARG;
  if (a.K % 256 != 0 || a.N % 128 != 0) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (a.N > INT32_MAX || a.K > INT32_MAX) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (a.r > 0 && (a.r > 64 || a.r % 8 != 0)) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a.x) || !aligned16(a.codes) || !aligned16(a.scales) ||
      (reinterpret_cast<uintptr_t>(a.tensor_scale) & 3u) || !aligned16(a.y) ||
      (a.r > 0 && (!aligned16(A_in) || !aligned16(B_in))))
    return QRR_ERR_MISALIGNED;
  return QRR_OK;
}

qrr_status run_linear(const LinIn* in, int count, int64_t M, void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, cudaStream_t s) {
  const LinPlan pl = plan_linear(M, in, count);
  if (!workspace || workspace_bytes < pl.total) return QRR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  if (M == 0) return QRR_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // layers with K == 0 produce zeros; layers with N == 0 produce nothing
  W4Params p{};
  LoraDownBatch lb{};    // prefill: the adapter's down projection
  DecodeProBatch db{};   // decode: x16, p and t' in one cluster launch
  lb.status = dev_status;
  db.status = dev_status;
  p.status = dev_status;
  bool any_split = false;
  for (int j = 0; j < count; ++j) {
    const LinIn& a = in[j];
    const LinPlan::Layer& pj = pl.l[j];
    if (a.N == 0) continue;
    if (a.K == 0) {
      if (cudaMemsetAsync(a.y, 0, static_cast<size_t>(M * a.N) * 2, s) != cudaSuccess) return QRR_ERR_CUDA;
      continue;
    }
    __nv_bfloat16* tbuf = reinterpret_cast<__nv_bfloat16*>(ws + pj.t_off);
    __half* x16 = reinterpret_cast<__half*>(ws + pj.x16_off);
    int* pexp = reinterpret_cast<int*>(ws + pj.p_off);
    const int R = (a.r + 15) / 16 * 16;
    if (pl.f16) {
      DecodeProLayer& dl = db.l[db.count++];
      dl.x = static_cast<const uint16_t*>(a.x);
      dl.A = static_cast<const uint16_t*>(a.A);
      dl.x16 = pl.nvf4 ? nullptr : x16;
      dl.planes = pl.nvf4 ? reinterpret_cast<uint8_t*>(x16) : nullptr;
      dl.ms = nvf4_geo(static_cast<int>(M)).ms;
      dl.pexp = pexp;
      dl.t = tbuf;
      dl.tensor_scale = a.tensor_scale;
      dl.M = static_cast<int>(M);
      dl.K = static_cast<int>(a.K);
      dl.r = a.r;
      dl.R = a.r > 0 ? R : 0;
      dl.t_cols = 64 * pj.lora_chunks;
      dl.lora_scale = a.r > 0 ? a.alpha / static_cast<float>(a.r) : 0.0f;
    } else if (a.r > 0) {
      // prologue: the LoRA down projection on the tensor cores, one CTA per
      // 128-token tile over the whole K
      LoraDownLayer& ld = lb.l[lb.count++];
      if (!make_tmap_2d(&ld.tx, a.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, M, a.K, a.K * 2, 128, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
          !make_tmap_2d(&ld.ta, a.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.r, a.K, a.K * 2, R, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return QRR_ERR_CUDA;
      ld.t = tbuf;
      ld.tensor_scale = a.tensor_scale;
      ld.tpart = nullptr;
      ld.tickets = nullptr;
      ld.x = static_cast<const uint16_t*>(a.x);
      ld.x16 = nullptr;
      ld.pexp = nullptr;
      ld.M = static_cast<int>(M);
      ld.K = static_cast<int>(a.K);
      ld.r = a.r;
      ld.R = R;
      ld.t_cols = 64 * pj.lora_chunks;
      ld.ks = 1;
      ld.slice_steps = static_cast<int>(a.K / 64);
      ld.lora_scale = a.alpha / static_cast<float>(a.r);
    }
    W4Layer& L = p.layer[p.count++];
    const void* xsrc = pl.f16 ? static_cast<const void*>(x16) : a.x;
    const CUtensorMapDataType xt = pl.f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t box_m = pl.pair ? pl.bn / 2 : pl.bn;  // token rows one CTA loads
    if (pl.nvf4) {
      const Nvf4Geo geo = nvf4_geo(static_cast<int>(M));
      if (!make_tmap_2d(&L.tp, x16, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<uint64_t>(kXPlanes) * geo.ms, a.K / 2,
                        a.K / 2, static_cast<uint32_t>(geo.nmma), 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return QRR_ERR_CUDA;
    }
    if ((!pl.nvf4 && !make_tmap_2d(&L.tx, xsrc, xt, M, a.K, a.K * 2, box_m, 64, CU_TENSOR_MAP_SWIZZLE_128B)) ||
        !make_tmap_2d(&L.tcodes, a.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, a.K / 2, a.K / 2, 128, pl.bk / 2,
                      pl.bk == 256 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_tmap_2d(&L.tscales, a.scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.N, a.K / 16, a.K / 16, 128, 16,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
      return QRR_ERR_CUDA;
    if (a.r > 0) {
      if (!make_tmap_2d(&L.tt, tbuf, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, M, 64 * pj.lora_chunks,
                        64 * pj.lora_chunks * 2, box_m, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return QRR_ERR_CUDA;
      if (pl.f16 && !make_tmap_2d(&L.tb, a.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.N, a.r, a.r * 2, 128,
                                  static_cast<uint32_t>(a.r), CU_TENSOR_MAP_SWIZZLE_NONE))
        return QRR_ERR_CUDA;
    } else {
      L.tt = L.tx;  // never read without an adapter
    }
    L.scales = a.scales;
    L.tensor_scale = a.tensor_scale;
    L.B = static_cast<const uint16_t*>(a.B);
    L.pexp = pl.f16 ? pexp : nullptr;
    L.y = static_cast<__nv_bfloat16*>(a.y);
    L.partial = reinterpret_cast<float*>(ws + pj.part_off);
    L.counters = reinterpret_cast<uint32_t*>(ws + pj.cnt_off);
    L.M = static_cast<int>(M);
    L.N = static_cast<int>(a.N);
    L.K = static_cast<int>(a.K);
    L.r = a.r;
    L.lora_chunks = pj.lora_chunks;
    L.n_tiles = pj.n_tiles;
    L.m_tiles = pl.m_tiles;
    L.splits = pj.splits;
    L.kcps = pj.kcps;
    any_split = any_split || pj.splits > 1;
  }
  if (p.count == 0) return QRR_OK;
  if (pl.f16 && pl.sk) {
    int kc[kMaxW4Layers], nl[kMaxW4Layers], nt[kMaxW4Layers], mt[kMaxW4Layers], pieces[kMaxW4Layers];
    for (int j = 0; j < p.count; ++j) {
      kc[j] = p.layer[j].K / pl.bk;
      nl[j] = p.layer[j].r > 0 ? 1 : 0;
      nt[j] = p.layer[j].n_tiles;
      mt[j] = p.layer[j].m_tiles;
    }
    if (stream_k_units(kc, nl, nt, mt, p.count, decode_grid(), &p, pieces) < 0) return QRR_ERR_UNSUPPORTED_SHAPE;
  } else if (pl.f16) {
    lpt_units(p, pl.bk, decode_grid());  // no table (round-robin) when it does not fit
  }
  if (pl.f16) {
    // split tiles occur on the decode path only, and their counters are
    // cleared by the prologue, which the GEMM waits for before it touches them
    if (any_split) {
      db.clear = reinterpret_cast<uint32_t*>(ws + pl.cnt_begin);
      db.clear_words = static_cast<int>(pl.cnt_bytes / 4);
    }
    if (launch_decode_prologue(db, s) != cudaSuccess) return QRR_ERR_CUDA;
    if (pl.nvf4) return from_cuda(launch_w4_decode_nvf4(p, s));
    return from_cuda(launch_w4a16_tc(p, pl.bn, pl.f16, pl.pair, true, s));
  }
  if (lb.count > 0 && launch_lora_down_tc(lb, s) != cudaSuccess) return QRR_ERR_CUDA;
  return from_cuda(launch_w4a16_tc(p, pl.bn, pl.f16, pl.pair, lb.count > 0, s));
}

LinIn make_in(const void* x, int64_t N, int64_t K, const uint8_t* codes, const uint8_t* scales, const float* ts,
              const void* A, const void* B, int32_t r, float alpha, void* y) {
  const bool lora = r > 0 && A && B;
  return LinIn{x, N, K, codes, scales, ts, A, B, lora ? r : 0, alpha, y};
}

size_t linear_ws_bytes(int64_t M, int64_t N, int64_t K, int32_t r) {
  if (M < 0 || N < 0 || K < 0 || r < 0) return 0;
  const LinIn in{nullptr, N, K, nullptr, nullptr, nullptr, nullptr, nullptr, r, 0.0f, nullptr};
  return plan_linear(M, &in, 1).total;
}

// ---- scratch for qrr_linear_nvfp4_lora_noalloc ----------------------------
//
// A fixed block of device memory that the library owns, for callers that
// cannot allocate device memory themselves.  It is a file-scope __device__
// array, so every GPU that loads the library holds it until the process
// exits.  In host code its name is only a host-side stand-in: the device
// address comes from cudaGetSymbolAddress, taken once per device (with that
// device current) on the first call.
static __device__ __align__(256) uint8_t g_noalloc_scratch[QRR_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mutex;
constexpr int kMaxDevices = 64;
void* g_noalloc_addr[kMaxDevices] = {};

qrr_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QRR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) return QRR_ERR_CUDA;
    g_noalloc_addr[dev] = addr;
  }
  *out = g_noalloc_addr[dev];
  return QRR_OK;
}

// ---- LoRA backward: workspace plan ----
struct BwdPlan {
  int t_cols, slice, ks_u, ks_t;
  size_t wt_off, at2_off, bt_off, tu_off, tt_off, pu_off, pt_off, tick_off, tick_bytes, gpart_off, total;
};

BwdPlan plan_backward(int64_t M, int64_t N, int64_t K, int32_t r) {
  BwdPlan p{};
  p.t_cols = r > 0 ? 64 * static_cast<int>((2 * r + 63) / 64) : 0;
  p.slice = 2048;  // contraction slice of the rank projections (32 steps of 64)
  p.ks_u = static_cast<int>((N + p.slice - 1) / p.slice);
  p.ks_t = static_cast<int>((K + p.slice - 1) / p.slice);
  size_t off = 0;
  p.wt_off = off;
  off += round_up(static_cast<size_t>(K) * N * 2);
  p.at2_off = off;
  off += round_up(static_cast<size_t>(K) * p.t_cols * 2);
  p.bt_off = off;
  off += round_up(static_cast<size_t>(r) * N * 2);
  p.tu_off = off;
  off += round_up(static_cast<size_t>(M) * p.t_cols * 2);
  p.tt_off = off;
  off += round_up(static_cast<size_t>(M) * p.t_cols * 2);
  p.pu_off = off;
  off += round_up(static_cast<size_t>((p.ks_u + 3) & ~3) * M * r * 4);
  p.pt_off = off;
  off += round_up(static_cast<size_t>((p.ks_t + 3) & ~3) * M * r * 4);
  p.tick_off = off;
  p.tick_bytes = 2 * static_cast<size_t>((M + 127) / 128) * 4;
  off += round_up(p.tick_bytes);
  p.gpart_off = off;
  if (r > 0 && M > 0) {
    const size_t ga = static_cast<size_t>(lora_grad_slices(M, K)) * r * K;
    const size_t gb = static_cast<size_t>(lora_grad_slices(M, N)) * r * N;
    off += round_up((ga > gb ? ga : gb) * 4);
  }
  p.total = round_up(off) + kAlign;
  return p;
}

}  // namespace

extern "C" {

size_t qrr_lora_backward_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r) {
  if (M < 0 || N < 0 || K < 0 || r < 0 || r > 64) return 0;
  return plan_backward(M, N, K, r).total;
}

qrr_status qrr_lora_backward_nvfp4(const void* dy, int64_t M, int64_t N, const void* x, int64_t K,
                                   const uint8_t* codes, const uint8_t* scales, const float* tensor_scale,
                                   const void* lora_A, const void* lora_B, int32_t r, float alpha, void* dx, float* dA,
                                   float* dB, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                   void* stream) {
  if (M < 0 || N < 0 || K < 0 || r < 0) return QRR_ERR_INVALID_ARG;
  const bool lora = r > 0 && lora_A && lora_B;
  if (!lora) r = 0;
  if (!tensor_scale) return QRR_ERR_INVALID_ARG;
  if (M * N > 0 && !dy) return QRR_ERR_INVALID_ARG;
  if (M * K > 0 && (!dx || (lora && !x))) return QRR_ERR_INVALID_ARG;
  if (N * K > 0 && (!codes || !scales)) return QRR_ERR_INVALID_ARG;
  if (lora && ((K > 0 && !dA) || (N > 0 && !dB))) return QRR_ERR_INVALID_ARG;
  if (K % 256 != 0 || N % 128 != 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (r > 64 || (r > 0 && r % 8 != 0)) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(dx) ||
      (reinterpret_cast<uintptr_t>(tensor_scale) & 3u) ||
      (lora && (!aligned16(lora_A) || !aligned16(lora_B) || !aligned16(dA) || !aligned16(dB))))
    return QRR_ERR_MISALIGNED;
  const BwdPlan pl = plan_backward(M, N, K, r);
  if (!workspace || workspace_bytes < pl.total) return QRR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  cudaStream_t s = as_stream(stream);
  // degenerate sizes: sums over nothing are zero
  if (M == 0 || N == 0 || K == 0) {
    if (M * K > 0 && cudaMemsetAsync(dx, 0, static_cast<size_t>(M * K) * 2, s) != cudaSuccess) return QRR_ERR_CUDA;
    if (lora && K > 0 && cudaMemsetAsync(dA, 0, static_cast<size_t>(r) * K * 4, s) != cudaSuccess) return QRR_ERR_CUDA;
    if (lora && N > 0 && cudaMemsetAsync(dB, 0, static_cast<size_t>(N) * r * 4, s) != cudaSuccess) return QRR_ERR_CUDA;
    return QRR_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* wt = reinterpret_cast<__nv_bfloat16*>(ws + pl.wt_off);
  uint16_t* at2 = reinterpret_cast<uint16_t*>(ws + pl.at2_off);
  uint16_t* bt = reinterpret_cast<uint16_t*>(ws + pl.bt_off);
  __nv_bfloat16* tu = reinterpret_cast<__nv_bfloat16*>(ws + pl.tu_off);
  __nv_bfloat16* tt = reinterpret_cast<__nv_bfloat16*>(ws + pl.tt_off);
  if (launch_lora_backward_prep(codes, scales, lora_A, lora_B, static_cast<int>(N), static_cast<int>(K), r, pl.t_cols,
                                wt, at2, bt, s) != cudaSuccess)
    return QRR_ERR_CUDA;
  if (lora) {
    // u' = (alpha/r) (dY . B) / g and t' = (alpha/r) (x . A^T) / g, split over
    // 2048-wide contraction slices with a ticket per 128-token tile
    if (cudaMemsetAsync(ws + pl.tick_off, 0, pl.tick_bytes, s) != cudaSuccess) return QRR_ERR_CUDA;
    LoraDownBatch lb{};
    lb.status = dev_status;
    const int m_tiles = static_cast<int>((M + 127) / 128);
    const void* src_x[2] = {dy, x};
    const void* src_a[2] = {bt, lora_A};
    const int64_t kk[2] = {N, K};
    __nv_bfloat16* outs[2] = {tu, tt};
    const size_t poff[2] = {pl.pu_off, pl.pt_off};
    const int ksv[2] = {pl.ks_u, pl.ks_t};
    for (int i = 0; i < 2; ++i) {
      LoraDownLayer& ld = lb.l[lb.count++];
      if (!make_tmap_2d(&ld.tx, src_x[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, M, kk[i], kk[i] * 2, 128, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
          !make_tmap_2d(&ld.ta, src_a[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, r, kk[i], kk[i] * 2, (r + 15) / 16 * 16, 64,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return QRR_ERR_CUDA;
      ld.t = outs[i];
      ld.tensor_scale = tensor_scale;
      ld.tpart = reinterpret_cast<float*>(ws + poff[i]);
      ld.tickets = reinterpret_cast<uint32_t*>(ws + pl.tick_off) + i * m_tiles;
      ld.x = static_cast<const uint16_t*>(src_x[i]);
      ld.x16 = nullptr;
      ld.pexp = nullptr;
      ld.M = static_cast<int>(M);
      ld.K = static_cast<int>(kk[i]);
      ld.r = r;
      ld.R = (r + 15) / 16 * 16;
      ld.t_cols = pl.t_cols;
      ld.ks = ksv[i];
      ld.slice_steps = pl.slice / 64;
      ld.lora_scale = alpha / static_cast<float>(r);
    }
    if (launch_lora_down_tc(lb, s) != cudaSuccess) return QRR_ERR_CUDA;
  }
  // dX = g (dY . W_q + u' . A)
  Bf16GemmArgs ga{dy, wt, lora ? tu : nullptr, lora ? at2 : nullptr, tensor_scale, dx, M, K, N,
                  lora ? pl.t_cols : 0};
  if (launch_gemm_bf16_tc(ga, dev_status, s) != cudaSuccess) return QRR_ERR_CUDA;
  if (lora) {
    float* gpart = reinterpret_cast<float*>(ws + pl.gpart_off);
    if (launch_lora_grad(x, reinterpret_cast<const uint16_t*>(tu), static_cast<int>(M), static_cast<int>(K), r,
                         pl.t_cols, tensor_scale, false, gpart, dA, s) != cudaSuccess ||
        launch_lora_grad(dy, reinterpret_cast<const uint16_t*>(tt), static_cast<int>(M), static_cast<int>(N), r,
                         pl.t_cols, tensor_scale, true, gpart, dB, s) != cudaSuccess)
      return QRR_ERR_CUDA;
  }
  return QRR_OK;
}


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
  batch.job[0] = Nvfp4Job{static_cast<const uint16_t*>(W), codes, scales, tensor_scale, N, K, 0, 0, 0u};
  batch.amax_bits = static_cast<uint32_t*>(workspace);
  batch.status = dev_status;
  return from_cuda(launch_nvfp4(batch, as_stream(stream)));
}

qrr_status qrr_linear_nvfp4_lora(const void* x, int64_t M, int64_t K, const uint8_t* codes, const uint8_t* scales,
                                 const float* tensor_scale, int64_t N, const void* lora_A, const void* lora_B,
                                 int32_t r, float alpha, void* y, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, void* stream) {
  if (M < 0 || M > INT32_MAX) return M < 0 ? QRR_ERR_INVALID_ARG : QRR_ERR_UNSUPPORTED_SHAPE;
  const LinIn in = make_in(x, N, K, codes, scales, tensor_scale, lora_A, lora_B, r, alpha, y);
  qrr_status st = check_linear(in, M, lora_A, lora_B, r);
  if (st != QRR_OK) return st;
  return run_linear(&in, 1, M, workspace, workspace_bytes, dev_status, as_stream(stream));
}

size_t qrr_linear_nvfp4_lora_grouped_workspace_bytes(const qrr_linear_desc* descs, int32_t count, int64_t M) {
  if (!descs || count <= 0 || count > kMaxW4Layers || M < 0) return 0;
  LinIn in[kMaxW4Layers];
  for (int j = 0; j < count; ++j)
    in[j] = make_in(descs[j].x, descs[j].N, descs[j].K, descs[j].codes, descs[j].scales, descs[j].tensor_scale,
                    descs[j].lora_A, descs[j].lora_B, descs[j].r, descs[j].alpha, descs[j].y);
  return plan_linear(M, in, count).total;
}

qrr_status qrr_linear_nvfp4_lora_grouped(const qrr_linear_desc* descs, int32_t count, int64_t M, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (count < 0 || (count > 0 && !descs) || M < 0) return QRR_ERR_INVALID_ARG;
  if (count > kMaxW4Layers || M > INT32_MAX) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (count == 0) return QRR_OK;
  LinIn in[kMaxW4Layers];
  for (int j = 0; j < count; ++j) {
    const qrr_linear_desc& d = descs[j];
    in[j] = make_in(d.x, d.N, d.K, d.codes, d.scales, d.tensor_scale, d.lora_A, d.lora_B, d.r, d.alpha, d.y);
    qrr_status st = check_linear(in[j], M, d.lora_A, d.lora_B, d.r);
    if (st != QRR_OK) return st;
  }
  return run_linear(in, count, M, workspace, workspace_bytes, dev_status, as_stream(stream));
}

size_t qrr_noalloc_scratch_bytes(void) { return QRR_NOALLOC_SCRATCH_BYTES; }

qrr_status qrr_linear_nvfp4_lora_noalloc(const void* x, int64_t M, int64_t K, const uint8_t* codes,
                                         const uint8_t* scales, const float* tensor_scale, int64_t N,
                                         const void* lora_A, const void* lora_B, int32_t r, float alpha, void* y,
                                         int32_t* dev_status, void* stream) {
  if (M < 0 || M > INT32_MAX) return M < 0 ? QRR_ERR_INVALID_ARG : QRR_ERR_UNSUPPORTED_SHAPE;
  const LinIn in = make_in(x, N, K, codes, scales, tensor_scale, lora_A, lora_B, r, alpha, y);
  qrr_status st = check_linear(in, M, lora_A, lora_B, r);
  if (st != QRR_OK) return st;
  // too large for the built-in scratch: refused before anything is launched
  if (linear_ws_bytes(M, N, K, in.r) > QRR_NOALLOC_SCRATCH_BYTES) return QRR_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != QRR_OK) return st;
  return run_linear(&in, 1, M, scratch, QRR_NOALLOC_SCRATCH_BYTES, dev_status, as_stream(stream));
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
  batch.job[0] = Fp8WJob{static_cast<const uint16_t*>(W), q, scales, N, K, 0, 0u};
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
  // power-of-two scales run on the native block-scaled MMA (UE8M0 scale
  // bytes, no promotion); FP32 scales promote each 128-K block sum in fp32
  if (scale_mode == QRR_SCALE_POW2) return from_cuda(launch_fp8_gemm_mx(a, dev_status, s));
  return from_cuda(launch_fp8_gemm_tc(a, dev_status, s));
}

static qrr_status requantize(const qrr_weight_desc* descs, int32_t count, int32_t format, int32_t scale_mode,
                             const AqnParams& aqn, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             void* stream) {
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
      batch.aqn = aqn;
      for (int i = 0; i < n; ++i) {
        const qrr_weight_desc& d = descs[g + i];
        batch.job[i] = Nvfp4Job{static_cast<const uint16_t*>(d.W), d.codes, static_cast<uint8_t*>(d.scales),
                                d.tensor_scale, d.N, d.K, 0, 0, static_cast<uint32_t>(g + i)};
      }
      e = launch_nvfp4(batch, s);
    } else {
      Fp8WBatch batch{};
      batch.count = n;
      batch.mode = scale_mode;
      batch.status = dev_status;
      batch.aqn = aqn;
      for (int i = 0; i < n; ++i) {
        const qrr_weight_desc& d = descs[g + i];
        batch.job[i] = Fp8WJob{static_cast<const uint16_t*>(d.W), d.codes, static_cast<float*>(d.scales), d.N, d.K, 0,
                               static_cast<uint32_t>(g + i)};
      }
      e = launch_fp8_w128(batch, s);
    }
    if (e != cudaSuccess) return QRR_ERR_CUDA;
  }
  return QRR_OK;
}

qrr_status qrr_kv_append_fp8(const void* k_new, const void* v_new, int32_t B, int32_t Hkv, const int32_t* pos,
                             uint8_t* k_cache, float* k_scales, uint8_t* v_cache, float* v_scales, int32_t Lmax,
                             int32_t scale_mode, int32_t* dev_status, void* stream) {
  if (B < 0 || Hkv < 0 || Lmax < 0 || !is_fp8_mode(scale_mode)) return QRR_ERR_INVALID_ARG;
  if (B * Hkv > 0 && (!k_new || !v_new || !pos || !k_cache || !k_scales || !v_cache || !v_scales))
    return QRR_ERR_INVALID_ARG;
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if ((reinterpret_cast<uintptr_t>(k_new) & 7u) || (reinterpret_cast<uintptr_t>(v_new) & 7u) || !a4(pos) ||
      !aligned16(k_cache) || !aligned16(v_cache) || !a4(k_scales) || !a4(v_scales))
    return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  return from_cuda(launch_kv_append_fp8(k_new, v_new, B, Hkv, pos, Lmax, k_cache, k_scales, v_cache, v_scales,
                                        scale_mode, dev_status, as_stream(stream)));
}

size_t qrr_attention_decode_fp8_workspace_bytes(int32_t B, int32_t Hq, int32_t Lmax) {
  if (B < 0 || Hq < 0 || Lmax < 0) return 0;
  return round_up(static_cast<size_t>(B) * Hq * attn_splits(Lmax) * (2 + 128) * 4) + kAlign;
}

qrr_status qrr_attention_decode_fp8(const void* q, int32_t B, int32_t Hq, int32_t Hkv, const uint8_t* k_cache,
                                    const float* k_scales, const uint8_t* v_cache, const float* v_scales,
                                    const int32_t* lens, int32_t Lmax, void* out, void* workspace,
                                    size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (B < 0 || Hq < 0 || Hkv <= 0 || Lmax < 0) return QRR_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return QRR_ERR_UNSUPPORTED_SHAPE;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (Lmax % 4 != 0) return QRR_ERR_UNSUPPORTED_SHAPE;
  if (B * Hq > 0 && (!q || !k_cache || !k_scales || !v_cache || !v_scales || !lens || !out)) return QRR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(k_scales) || !aligned16(v_cache) || !aligned16(v_scales) ||
      !aligned16(out) || (reinterpret_cast<uintptr_t>(lens) & 3u))
    return QRR_ERR_MISALIGNED;
  const size_t need = qrr_attention_decode_fp8_workspace_bytes(B, Hq, Lmax);
  if (!workspace || workspace_bytes < need) return QRR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  const size_t rows = static_cast<size_t>(B) * Hq * attn_splits(Lmax);
  float* pm = static_cast<float*>(workspace);
  float* pl = pm + rows;
  float* po = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + round_up(rows * 8));
  return from_cuda(launch_attention_decode_fp8(q, k_cache, k_scales, v_cache, v_scales, lens, B, Hq, Hkv, Lmax, out,
                                               pm, pl, po, dev_status, as_stream(stream)));
}

qrr_status qrr_token_logprobs_is(const void* logits, int64_t T, int64_t V, const int32_t* tokens,
                                 const float* rollout_logp, float cap, float* logp, float* w, int32_t* dev_status,
                                 void* stream) {
  if (T < 0 || V < 1) return QRR_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !tokens || !logp || (rollout_logp && !w))) return QRR_ERR_INVALID_ARG;
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!aligned16(logits) || !a4(tokens) || !a4(logp) || !a4(rollout_logp) || !a4(w)) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  return from_cuda(
      launch_token_logprob_is(logits, T, V, tokens, rollout_logp, cap, logp, w, dev_status, as_stream(stream)));
}

qrr_status qrr_get_last_device_status(int32_t* host_out, const int32_t* dev_status, void* stream) {
  if (!host_out || !dev_status) return QRR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(dev_status) & 3u) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  cudaStream_t s = as_stream(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return QRR_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return QRR_ERR_CUDA;
  *host_out = v;
  return QRR_OK;
}

size_t qrr_workspace_bytes(int32_t op, int64_t M, int64_t N, int64_t K, int32_t r) {
  switch (op) {
    case QRR_OP_QUANTIZE_NVFP4: return qrr_quantize_nvfp4_workspace_bytes();
    case QRR_OP_LINEAR_NVFP4_LORA: return qrr_linear_nvfp4_lora_workspace_bytes(M, N, K, r);
    case QRR_OP_REQUANTIZE_WEIGHTS:
      return M < 0 || M > INT32_MAX ? 0 : qrr_requantize_workspace_bytes(static_cast<int32_t>(M));
    case QRR_OP_QUANTIZE_FP8:
    case QRR_OP_GEMM_FP8: return 0;
    case QRR_OP_LORA_BACKWARD: return qrr_lora_backward_workspace_bytes(M, N, K, r);
    default: return 0;
  }
}

int64_t qrr_plan_decode_units(int64_t M, int32_t count, const int64_t* N, const int64_t* K, const int32_t* r,
                              int32_t grid, uint32_t* units, int32_t max_units, uint16_t* offsets,
                              int32_t* grid_used) {
  if (!N || !K || !r || !units || !offsets || !grid_used || max_units < 0) return -QRR_ERR_INVALID_ARG;
  if (M < 1 || M > 64 || count < 1 || count > kMaxW4Layers || grid < 1 || grid > kMaxTableCtas)
    return -QRR_ERR_INVALID_ARG;
  LinIn in[kMaxW4Layers];
  for (int j = 0; j < count; ++j) {
    if (N[j] <= 0 || K[j] <= 0 || N[j] % 128 != 0 || K[j] % 256 != 0 || N[j] > INT32_MAX || K[j] > INT32_MAX)
      return -QRR_ERR_UNSUPPORTED_SHAPE;
    if (r[j] < 0 || r[j] > 64 || r[j] % 8 != 0) return -QRR_ERR_UNSUPPORTED_SHAPE;
    in[j] = LinIn{nullptr, N[j], K[j], nullptr, nullptr, nullptr, nullptr, nullptr, r[j], 0.0f, nullptr};
  }
  // the decode launch's own planning (run_linear): per-layer splits, then the table
  const LinPlan pl = plan_linear(M, in, count);
  W4Params p{};
  p.count = count;
  int kc[kMaxW4Layers], nl[kMaxW4Layers], nt[kMaxW4Layers], mt[kMaxW4Layers], pieces[kMaxW4Layers];
  for (int j = 0; j < count; ++j) {
    W4Layer& L = p.layer[j];
    L.M = static_cast<int>(M);
    L.N = static_cast<int>(N[j]);
    L.K = static_cast<int>(K[j]);
    L.r = r[j];
    L.lora_chunks = pl.l[j].lora_chunks;
    L.n_tiles = pl.l[j].n_tiles;
    L.m_tiles = pl.m_tiles;
    L.splits = pl.l[j].splits;
    L.kcps = pl.l[j].kcps;
    kc[j] = L.K / pl.bk;
    nl[j] = r[j] > 0 ? 1 : 0;
    nt[j] = L.n_tiles;
    mt[j] = L.m_tiles;
  }
  if (pl.sk) {
    if (stream_k_units(kc, nl, nt, mt, count, grid, &p, pieces) < 0) return -QRR_ERR_UNSUPPORTED_SHAPE;
  } else {
    lpt_units(p, pl.bk, grid);
    if (!p.use_table) return -QRR_ERR_UNSUPPORTED_SHAPE;
  }
  if (p.total_units > max_units) return -QRR_ERR_WORKSPACE;
  memcpy(units, p.unit, sizeof(uint32_t) * 2 * static_cast<size_t>(p.total_units));
  memcpy(offsets, p.unit_off, sizeof(uint16_t) * static_cast<size_t>(p.table_grid + 1));
  *grid_used = p.table_grid;
  return p.total_units;
}

qrr_status qrr_wait_probe(int64_t limit_cycles, int32_t arrive, int32_t* dev_status, int64_t* cycles, void* stream) {
  if (limit_cycles <= 0 || limit_cycles > kWaitLimitCycles || (arrive != 0 && arrive != 1)) return QRR_ERR_INVALID_ARG;
  if (!dev_status) return QRR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_status) & 3u) || (reinterpret_cast<uintptr_t>(cycles) & 7u))
    return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  return from_cuda(launch_wait_probe(limit_cycles, arrive, dev_status, reinterpret_cast<long long*>(cycles),
                                     as_stream(stream)));
}

qrr_status qrr_stream_probe(const void* data, int64_t rows, int64_t row_bytes, int32_t* dev_status, void* stream) {
  if (rows < 0 || row_bytes < 0 || (rows * row_bytes > 0 && !data)) return QRR_ERR_INVALID_ARG;
  if (rows % 128 != 0 || row_bytes % 128 != 0 || rows > INT32_MAX || row_bytes > INT32_MAX)
    return QRR_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(data) || (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  if (rows == 0 || row_bytes == 0) return QRR_OK;
  return from_cuda(launch_stream_probe(data, rows, row_bytes, dev_status, as_stream(stream)));
}

qrr_status qrr_requantize_weights(const qrr_weight_desc* descs, int32_t count, int32_t format, int32_t scale_mode,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return requantize(descs, count, format, scale_mode, aqn_params(0.0f, 0u, 0ull), workspace, workspace_bytes,
                    dev_status, stream);
}

qrr_status qrr_requantize_weights_aqn(const qrr_weight_desc* descs, int32_t count, int32_t format,
                                      int32_t scale_mode, float sigma, uint64_t seed, int32_t step, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (!(sigma >= 0.0f) || sigma == INFINITY || step < 0) return QRR_ERR_INVALID_ARG;
  return requantize(descs, count, format, scale_mode, aqn_params(sigma, static_cast<uint32_t>(step), seed), workspace,
                    workspace_bytes, dev_status, stream);
}

float qrr_aqn_sigma(int32_t step, int32_t steps, double sigma_start, double sigma_end) {
  if (steps <= 1 || step >= steps - 1) return static_cast<float>(sigma_end);
  if (step <= 0) return static_cast<float>(sigma_start);
  return static_cast<float>(sigma_start * pow(sigma_end / sigma_start, static_cast<double>(step) / (steps - 1)));
}

qrr_status qrr_aqn_noise_probe(float* out, int64_t n, int64_t start, uint64_t seed, int32_t tensor, int32_t step,
                               void* stream) {
  if (n < 0 || start < 0 || tensor < 0 || step < 0 || (n > 0 && !out)) return QRR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out) & 3u) return QRR_ERR_MISALIGNED;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  return from_cuda(launch_aqn_noise_probe(out, n, start, static_cast<uint32_t>(tensor),
                                          aqn_params(1.0f, static_cast<uint32_t>(step), seed), as_stream(stream)));
}

qrr_status qrr_round_probe(const float* in, int64_t n, int32_t fmt, uint8_t* out, void* stream) {
  if (n < 0 || (fmt != 0 && fmt != 1)) return QRR_ERR_INVALID_ARG;
  if (n > 0 && (!in || !out)) return QRR_ERR_INVALID_ARG;
  if (injected_cuda_fault()) return QRR_ERR_CUDA;
  return from_cuda(launch_round_probe(in, n, fmt, out, as_stream(stream)));
}

}  // extern "C"

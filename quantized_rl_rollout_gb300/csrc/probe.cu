// Probe of the bounded-wait path that every tensor-core pipeline of the
// library relies on: one CTA allocates tensor memory, then waits on an
// mbarrier through the same bounded wait the pipelines use, with a short
// limit.  When nothing arrives, the wait gives up, the CTA raises
// QRR_DEV_TIMEOUT in the status word, releases its tensor memory and exits,
// and the context stays usable; when the barrier is completed first, the wait
// returns at once and nothing is flagged.
#include "tc.cuh"

namespace qrr {

__global__ void __launch_bounds__(64) wait_probe_kernel(long long limit, int arrive, int32_t* status,
                                                        long long* cycles) {
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem;
  __shared__ int abort;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem, 32);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 32) {
    if (arrive) mbar_arrive(&bar);  // completes phase 0 before anyone waits
    const long long t0 = clock64();
    mbar_wait(&bar, 0, &abort, status, limit);
    if (cycles) *cycles = clock64() - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

cudaError_t launch_wait_probe(long long limit, int arrive, int32_t* status, long long* cycles, cudaStream_t stream) {
  wait_probe_kernel<<<1, 64, 0, stream>>>(limit, arrive, status, cycles);
  return cudaGetLastError();
}



// Memory-system floor of one decode pass: a TMA stream with no arithmetic.
// Every SM's CTA takes a contiguous range of [128 rows x 128 B] boxes of a
// byte matrix (row tiles outer, 128-byte column tiles inner: the order and
// shape in which the decode kernels read a weight's packed codes) and pulls
// them through an 8-stage shared-memory ring; the consumer only waits for
// each box to land.  Its time after the same L2 flush bounds what any single
// pass over that many bytes can reach on this GPU, at any arithmetic cost.
namespace {
constexpr int kSpStages = 8;
constexpr int kSpBox = 128 * 128;  // bytes per box
struct StreamProbeParams {
  CUtensorMap map;  // u8 [rows, row_bytes], box [128, 128], 128-byte swizzle
  int64_t row_tiles, col_tiles;
  int32_t* status;
};
}  // namespace

__global__ void __launch_bounds__(64, 1) stream_probe_kernel(const __grid_constant__ StreamProbeParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kSpStages], empty[kSpStages];
  __shared__ int abort;
  const int64_t total = p.row_tiles * p.col_tiles;
  const int64_t b = blockIdx.x, G = gridDim.x;
  const int64_t s0 = total * b / G, s1 = total * (b + 1) / G;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSpStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t issued = 0;
    for (int64_t s = s0; s < s1; ++s) {
      const int64_t i = s - s0;
      const int slot = static_cast<int>(i % kSpStages);
      const uint32_t use = static_cast<uint32_t>(i / kSpStages);
      if (use > 0 && !mbar_wait(&empty[slot], (use - 1) & 1, &abort, p.status)) break;
      mbar_arrive_expect_tx(&full[slot], kSpBox);
      tma_load_2d(&p.map, &full[slot], ring + slot * kSpBox, static_cast<int>((s % p.col_tiles) * 128),
                  static_cast<int>((s / p.col_tiles) * 128));
      issued = i + 1;
    }
    // every issued copy has landed before the CTA exits
    volatile int no_abort = 0;
    for (int64_t k = issued - 1; k >= 0 && k >= issued - kSpStages; --k)
      mbar_wait(&full[k % kSpStages], static_cast<uint32_t>(k / kSpStages) & 1, &no_abort, p.status);
  } else if (threadIdx.x == 32) {
    for (int64_t s = s0; s < s1; ++s) {
      const int64_t i = s - s0;
      const int slot = static_cast<int>(i % kSpStages);
      if (!mbar_wait(&full[slot], static_cast<uint32_t>(i / kSpStages) & 1, &abort, p.status)) break;
      mbar_arrive(&empty[slot]);
    }
  }
  __syncthreads();
}

cudaError_t launch_stream_probe(const void* data, int64_t rows, int64_t row_bytes, int32_t* status,
                                cudaStream_t stream) {
  static bool attr = false;
  constexpr int smem = 1024 + kSpStages * kSpBox;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(stream_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  StreamProbeParams p{};
  if (!make_tmap_2d(&p.map, data, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<uint64_t>(rows),
                    static_cast<uint64_t>(row_bytes), static_cast<uint64_t>(row_bytes), 128, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  p.row_tiles = rows / 128;
  p.col_tiles = row_bytes / 128;
  p.status = status;
  int dev = 0, sms = kSMs;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t total = p.row_tiles * p.col_tiles;
  const int grid = static_cast<int>(total < sms ? total : sms);
  stream_probe_kernel<<<grid, 64, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace qrr

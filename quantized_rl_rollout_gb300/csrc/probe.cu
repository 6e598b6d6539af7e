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

}  // namespace qrr

// Blackwell (sm_103a) building blocks written as inline PTX: mbarriers with
// bounded waits, TMA tile loads, tensor-memory (TMEM) allocation / load /
// store, tcgen05.mma issue and commit, and the shared-memory / instruction
// descriptors the MMA reads.
//
// Every wait here is bounded: a wait that does not complete within
// kWaitLimitCycles sets `*abort` (a per-CTA shared flag) and the kernel's
// QRR_DEV_TIMEOUT status bit, and all later waits of the CTA return at once,
// so a broken pipeline ends the kernel instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace qrr {

constexpr long long kWaitLimitCycles = 4000000000ll;  // about 2 s at the GB300's 2 GHz SM clock
constexpr int32_t kDevTimeout = 0x2;                         // status bit of a timed-out wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


// ---- mbarrier -------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same, but a thread whose phase is still open is parked by the hardware until
// the phase completes or about `ns` nanoseconds pass, instead of spinning: a
// spinning waiter takes issue slots from the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

constexpr uint32_t kWaitSliceNs = 1u << 20;  // about 1 ms per parked try

// Bounded wait for the phase with the given parity to complete.  Returns
// false (and raises the abort flag) on timeout or when another wait of the
// CTA already timed out.  `limit` is the give-up time in SM clock cycles; the
// pipelines use the default, a test of the timeout path passes a short one.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  // the SM cycle counter is cheap to read (a global timer read costs about a
  // microsecond, which would add that much latency to every hand-off)
  const long long t0 = clock64();
  while (true) {
#ifdef QRR_WAIT_SPIN
    if (mbar_try_wait(bar, parity)) return true;
#else
    if (mbar_try_wait_sleep(bar, parity, limit < kWaitLimitCycles ? 1000u : kWaitSliceNs)) return true;
#endif
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      flag(status, kDevTimeout);
      return false;
    }
  }
}

// ---- programmatic dependent launch ------------------------------------------

// In a kernel launched as the programmatic dependent of the previous kernel in
// its stream: wait until that kernel has completed and its writes are
// visible.  Without such a dependency it returns at once.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// In the earlier kernel: let the dependent kernel be scheduled (its CTAs start
// once every CTA of this grid has executed this or exited).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- TMA ------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tile load into shared memory, completion counted on `bar` in bytes.
// x is the innermost (contiguous) coordinate in elements, y the row.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Contiguous bulk copy global -> shared (TMA, no tensor map): both addresses
// 16-byte aligned, `bytes` a multiple of 16; completes `bytes` on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ---- TMEM -----------------------------------------------------------------

// Allocate `ncols` (power of two >= 32) TMEM columns; the base address is
// written to `*dst` in shared memory.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 columns of 32-bit: thread i of the warp gets TMEM lane
// (lane base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 4 columns of 32-bit from registers.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

// 32 lanes x 8 columns of 32-bit from registers.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(r[0]),
      "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- descriptors ------------------------------------------------------------

// Shared-memory matrix descriptor of a K-major operand tile stored in the
// 128-byte-swizzled layout TMA writes (rows of 128 bytes, 8-row groups of
// 1024 bytes).  Bits: start address >> 4 [0,14), leading byte offset >> 4
// [16,30) (unused for swizzled K-major), stride byte offset >> 4 [32,46),
// version 1 [46,48), base offset [49,52), swizzle mode [61,64) (2 = 128 B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Shared-memory matrix descriptor of an MN-major operand tile in the
// 128-byte-swizzled layout TMA writes when it loads boxes of 64 MN-contiguous
// 16-bit elements: each 128-byte row is one K index, 8 rows (1024 bytes) form
// a swizzle atom along K (stride byte offset), and the next 64 MN elements
// start `mn_stride` bytes later (leading byte offset).  Measured on GB300
// with a probe of small-integer matrices: exact results with these roles,
// wrong ones with the two offsets swapped.  A K16 MMA step advances the start
// address by 16 rows (2048 bytes).
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t smem_addr, uint32_t mn_stride) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor: D fp32, A/B formats, both K-major, shape M x N.
// Bits: D format [4,6) (1 = f32), A format [7,10), B format [10,13),
// A/B major [15], [16] (0 = K-major), N >> 3 [17,23), M >> 4 [24,29).
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_fmt, uint32_t b_fmt, uint32_t m, uint32_t n) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// The same with A and/or B MN-major (bits 15 and 16).
__host__ __device__ constexpr uint32_t make_idesc_major(uint32_t a_fmt, uint32_t b_fmt, uint32_t m, uint32_t n,
                                                        bool a_mn, bool b_mn) {
  return make_idesc(a_fmt, b_fmt, m, n) | (a_mn ? 1u << 15 : 0u) | (b_mn ? 1u << 16 : 0u);
}

constexpr uint32_t kFmtBF16 = 1;  // kind::f16 operand format
constexpr uint32_t kFmtE4M3 = 0;  // kind::f8f6f4 operand format

// D[tmem] (+)= A[smem] x B[smem]^T, kind::f16 (bf16 operands), cta_group::1.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with A read from TMEM.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four / eight kind::f16 MMAs with A from TMEM, issued back to back from one
// asm block: A chunk k sits 8 columns after chunk k - 1, `b[k]` are the B
// descriptors, only the first MMA takes `accumulate` (the others always add).
// The MMA pipe accepts an instruction about every 46 cycles; operand setup
// between single MMAs, on a sub-partition busy with other warps, would
// leave it idle.
__device__ __forceinline__ void mma4_ts(uint32_t d_tmem, uint32_t a_tmem, const uint64_t (&b)[4], uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 a1, a2, a3;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.eq.b32 q, %6, %6;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %7, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], %3, %7, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], %4, %7, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], %5, %7, q;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(accumulate), "r"(idesc)
      : "memory");
}

__device__ __forceinline__ void mma8_ts(uint32_t d_tmem, uint32_t a_tmem, const uint64_t (&b)[8], uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
      "setp.ne.b32 p, %10, 0;\n\tsetp.eq.b32 q, %10, %10;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\tadd.u32 a4, %1, 32;\n\t"
      "add.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\tadd.u32 a7, %1, 56;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %11, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], %3, %11, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], %4, %11, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], %5, %11, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], %6, %11, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], %7, %11, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], %8, %11, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], %9, %11, q;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]),
      "r"(accumulate), "r"(idesc)
      : "memory");
}

// The same four MMAs for a CTA pair (cta_group::2, M = 256): issued by one
// thread of the even CTA of a 2-CTA cluster; A is read from both CTAs' TMEM
// at a_tmem (128 rows each), B from both CTAs' shared memory at each
// descriptor's address (the even CTA holds rows [0, N/2) of B, the odd CTA
// rows [N/2, N)), and each CTA's TMEM at d_tmem receives its 128 rows of D
// over all N columns.
__device__ __forceinline__ void mma4_ts_pair(uint32_t d_tmem, uint32_t a_tmem, const uint64_t (&b)[4], uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 a1, a2, a3;\n\t"
      "setp.ne.b32 p, %6, 0;\n\tsetp.eq.b32 q, %6, %6;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %7, p;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a1], %3, %7, q;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a2], %4, %7, q;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [a3], %5, %7, q;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(accumulate), "r"(idesc)
      : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, kind::f8f6f4 (E4M3 operands).
__device__ __forceinline__ void mma_fp8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, kind::mxf8f6f4 with block scaling
// (E4M3 operands, one UE8M0 scale per 32 K of each row of A and of B): the
// scale bytes come from tensor memory at `sfa` / `sfb`, the byte within each
// 32-bit cell chosen by the scale ids of `idesc` (see make_idesc_mx).
// Layout for M = 128, cta_group::1 (measured on GB300 with a probe of
// encoded scale bytes): the scale of row m of A is lane m, column
// sfa + m / 32; the scale of row n of B is column sfb + n / 32, lane
// n % 32 of the lane quarter of the output row being formed, so every lane
// quarter holds a copy.
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::mxf8f6f4 with UE8M0 scales: E4M3 A and B,
// both K-major, D fp32, shape M x N; a_sf / b_sf pick the scale byte (0..3)
// of each 32-bit tensor-memory cell.  Bits: B scale id [4,6), A format
// [7,10), B format [10,13), N >> 3 [17,23), scale type [23] (1 = UE8M0),
// M >> 4 [24,29), A scale id [29,31).
__host__ __device__ constexpr uint32_t make_idesc_mx(uint32_t m, uint32_t n, uint32_t a_sf, uint32_t b_sf) {
  return (b_sf << 4) | (kFmtE4M3 << 7) | (kFmtE4M3 << 10) | ((n >> 3) << 17) | (1u << 23) | ((m >> 4) << 24) |
         (a_sf << 29);
}

// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Arrive on `bar` (same shared-memory offset) in each CTA of `cta_mask`
// once every cta_group::2 MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// ---- CTA pairs (2-CTA clusters) --------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster; orders shared-memory writes
// (release) before the peer's later reads (acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its cluster address (this CTA's or a
// peer's) with relaxed ordering.  A release at cluster scope would make the
// arriving thread wait until all its earlier memory operations are visible to
// the whole cluster (measured: about a thousand cycles per arrive, which
// halved the dequant rate of a CTA pair); the hand-offs that use this one
// carry tensor-memory state only, completed by tcgen05.wait::st / ::ld and
// ordered by tcgen05.fence::before_thread_sync before the arrive, and the
// waiter orders its own tcgen05 work after the wait with
// tcgen05.fence::after_thread_sync.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

// TMEM allocation shared by a CTA pair: one warp of each CTA executes it,
// and each CTA gets the same columns of its own TMEM.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 2-D tile load into this CTA's shared memory whose completion is counted on
// an mbarrier given by its cluster address, which may sit in the peer CTA of
// the pair.
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap* map, uint32_t bar_cluster, void* dst, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
  return pred;
}

// ---- host: tensor maps ------------------------------------------------------

// 2-D row-major tensor [rows, cols] of `elem_bytes`-byte elements with the
// given row pitch; box [box_rows, box_cols]; 128-byte swizzle; zero fill
// outside.  Returns false if the driver rejects the map.
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, uint64_t rows, uint64_t cols,
                  uint64_t row_pitch_bytes, uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle);

}  // namespace qrr

namespace qrr {

// 32 lanes x 16 columns of 32-bit.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 32 lanes x 32 columns of 32-bit from registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

constexpr uint32_t kFmtF16 = 0;  // kind::f16 operand format

// D[tmem] (+)= A[tmem] x B[smem]^T with an explicit instruction descriptor
// (the operand format is part of `idesc`, so f16 and bf16 MMAs can feed the
// same accumulator).
__device__ __forceinline__ void mma_f16kind_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  mma_bf16_ts(d_tmem, a_tmem, b_desc, idesc, accumulate);
}

// 32 lanes x 8 columns of 32-bit.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

// 32 lanes x 16 columns of 32-bit from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, kind::mxf4nvf4 with block scaling:
// packed E2M1 operands (two per byte, K-major, 64 K per MMA = 32 bytes of a
// row) and one UE4M3 scale per 16 K of every row of A and of B, the four
// scales of a row for the MMA's 64 K in one 32-bit tensor-memory cell (byte
// i for K [16 i, 16 i + 16)).  Cells are addressed as for kind::mxf8f6f4
// (row m of A: lane m, column sfa + m / 32; row n of B: column sfb + n / 32).
__device__ __forceinline__ void mma_nvf4_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B (format 1 of the
// fp4 kinds, bits [7,10) and [10,12)), UE4M3 scales (bit 23 clear), both
// K-major, D fp32, shape M x N, scale ids 0 (the whole cell is used).
__host__ __device__ constexpr uint32_t make_idesc_nvf4(uint32_t m, uint32_t n) {
  return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Named barrier over `count` threads (id 1..15; id 0 is __syncthreads).
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace qrr

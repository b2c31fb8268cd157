// Device-side building blocks for the sm_103a kernels: mbarriers with bounded waits, TMA
// tile loads, and the tcgen05 (5th-generation tensor core) instructions with their shared
// memory / instruction descriptors.  Everything here is hand-written inline PTX.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>

namespace sa2 {

// Device error codes written into the library's status word (same values as sa2_status).
constexpr unsigned kDevErrTimeout = 6u;
constexpr unsigned kDevErrBounds = 7u;
constexpr unsigned kDevErrRange = 8u;

// Default limit of a wait on an mbarrier, in nanoseconds of %globaltimer; legitimate waits
// in these kernels last microseconds.  The limit of the waits that make progress can be
// lowered at run time (ShapeArgs::wait_ns); the drains below always use this one.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Makes this thread's generic-proxy shared-memory writes visible to the async proxy (TMA,
// tensor core) once the threads synchronise.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void report_error(unsigned* status, unsigned code) {
  if (status) atomicCAS(status, 0u, code);
}

// ------------------------------------------------------------------------- mbarriers

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// What a CTA's waits share: its abort flag (in shared memory) and the time limit of its
// waits that make progress.
struct WaitCtl {
  volatile int* abort;
  unsigned long long limit_ns;
};

// A wait that makes progress: returns true once the phase with the given parity has
// completed.  Returns false, and raises the CTA's abort flag, once limit_ns have passed;
// returns false at once when another thread of the CTA has already raised the flag (the
// phase is tested first, so a completed phase is always seen).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (global_timer_ns() - t0 > w.limit_ns) {
      *w.abort = 1;
      return false;
    }
  }
}

// A drain: waits for a copy or an MMA this CTA has already issued to complete, so that no
// asynchronous operation still writes its shared memory when it exits, or reads or writes
// tensor memory when it is freed.  It ignores the abort flag -- an issued operation
// completes by itself -- and gives up only after kWaitLimitNs, raising the flag.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      return false;
    }
  }
}

// Test hook of the failure path: the calling warps sleep for stall_ns (bounded, in steps of
// at most 1 ms), so that waits of other warps on them expire when the wait limit is lower.
__device__ __forceinline__ void stall_for(unsigned long long stall_ns) {
  const unsigned long long t0 = global_timer_ns();
  while (global_timer_ns() - t0 < stall_ns) __nanosleep(1000000u);
}

// ------------------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled load (coordinates innermost first) completing on an mbarrier.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Plain (untiled) bulk copy of `bytes` from global to shared memory, completing on an
// mbarrier.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ----------------------------------------------------------------------------- tcgen05

// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"): start address, leading
// and stride byte offsets (16-byte units), descriptor version 1, swizzle mode in bits
// 61-63 (2 = 128-byte swizzle).  Base offset 0: every swizzle atom starts 1024-aligned.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode = 2) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swizzle_mode & 7u) << 61;
  return d;
}

// Instruction descriptor of kind::f16 with an fp32 accumulator; A and B are both bf16
// (bf16 = true) or both fp16.  a_mn / b_mn select the MN-major ("transposed") operand
// layouts.
__host__ __device__ constexpr uint32_t idesc_f32acc(int M, int N, bool a_mn, bool b_mn, bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return idesc_f32acc(M, N, a_mn, b_mn, true);
}
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn, bool b_mn) {
  return idesc_f32acc(M, N, a_mn, b_mn, false);
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T, one instruction issued by one thread.
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem)^T.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Descriptor offset (16-byte units) of k-step kk (16 elements of 2 bytes) in a K-major
// 128-byte-swizzled tile whose channel panels hold `rows` rows each.
__host__ __device__ constexpr uint64_t kmajor_kstep(int kk, int rows) {
  return (uint64_t)(((kk >> 2) * rows * 128 + (kk & 3) * 32) >> 4);
}

// The k-steps of one product, unrolled at compile time so every descriptor offset and
// accumulate flag is an immediate and the MMAs issue back to back.
// SS form, A and B K-major (A_ROWS / B_ROWS rows per channel panel); the first k-step
// overwrites D.
template <uint32_t IDESC, int A_ROWS, int B_ROWS, int KSTEPS, int KK = 0>
__device__ __forceinline__ void mma_ss_kmajor(uint32_t d, uint64_t a, uint64_t b) {
  umma_ss(d, a + kmajor_kstep(KK, A_ROWS), b + kmajor_kstep(KK, B_ROWS), IDESC, KK > 0 ? 1u : 0u);
  if constexpr (KK + 1 < KSTEPS) mma_ss_kmajor<IDESC, A_ROWS, B_ROWS, KSTEPS, KK + 1>(d, a, b);
}
// The same product accumulated onto D from the first k-step on.
template <uint32_t IDESC, int A_ROWS, int B_ROWS, int KSTEPS, int KK = 0>
__device__ __forceinline__ void mma_ss_kmajor_acc(uint32_t d, uint64_t a, uint64_t b) {
  umma_ss(d, a + kmajor_kstep(KK, A_ROWS), b + kmajor_kstep(KK, B_ROWS), IDESC, 1u);
  if constexpr (KK + 1 < KSTEPS) mma_ss_kmajor_acc<IDESC, A_ROWS, B_ROWS, KSTEPS, KK + 1>(d, a, b);
}
// TS form: A from TMEM (8 columns of fp16 pairs per k-step), B MN-major with 16 rows
// (2048 bytes) per k-step.  The first k-step overwrites D when `fresh`, else accumulates.
template <uint32_t IDESC, int KSTEPS, int KK = 0>
__device__ __forceinline__ void mma_ts_bmn(uint32_t d, uint32_t a, uint64_t b, bool fresh) {
  umma_ts(d, a + KK * 8, b + (uint64_t)(KK * 128), IDESC, KK > 0 ? 1u : (fresh ? 0u : 1u));
  if constexpr (KK + 1 < KSTEPS) mma_ts_bmn<IDESC, KSTEPS, KK + 1>(d, a, b, fresh);
}

// TS form with B K-major (B_ROWS rows per channel panel): A from TMEM, 8 columns (16 16-bit
// elements) per k-step; the first k-step overwrites D.
template <uint32_t IDESC, int B_ROWS, int KSTEPS, int KK = 0>
__device__ __forceinline__ void mma_ts_bkmajor(uint32_t d, uint32_t a, uint64_t b) {
  umma_ts(d, a + KK * 8, b + kmajor_kstep(KK, B_ROWS), IDESC, KK > 0 ? 1u : 0u);
  if constexpr (KK + 1 < KSTEPS) mma_ts_bkmajor<IDESC, B_ROWS, KSTEPS, KK + 1>(d, a, b);
}

// Arrive (once) on an mbarrier when every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM cells: thread t of the warp gets lane (base + t),
// columns col .. col+31.
#define SA2_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define SA2_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
#define SA2_P8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : SA2_R8(0), SA2_R8(8), SA2_R8(16), SA2_R8(24)
      : "r"(taddr));
}

// Waits for this thread's tcgen05.ld results; the registers pass through the asm so no use
// of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : SA2_P8(0), SA2_P8(8), SA2_P8(16), SA2_P8(24)::"memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      SA2_W8(0), SA2_W8(8), SA2_W8(16), SA2_W8(24)
      : "memory");
}

// 32 lanes x 16 columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16};" ::"r"(taddr),
      SA2_W8(0), SA2_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ int elect_lane0() { return (threadIdx.x & 31) == 0; }

// elect.sync: true in exactly one lane of a converged warp.  tcgen05.mma issued this way,
// with the whole warp running the issuing loop, issues markedly faster than from a lane
// the rest of its warp has branched away from.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}\n" : "=r"(pred));
  return pred != 0;
}

}  // namespace sa2

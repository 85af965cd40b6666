// Device helpers shared by the tcgen05 kernels (attention, QKV projection): mbarrier waits
// bounded in time, TMA tensor loads, tcgen05 MMA issue / commit / fences, shared-memory and
// instruction descriptors. Internal linkage: each translation unit gets its own copy.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace cb {
namespace {

constexpr unsigned long long kTimeoutNs = 2000000000ull;  // every mbarrier wait gives up after 2 s
constexpr unsigned long long kProbeTimeoutNs = 100000ull;  // the wait-timeout probe's limit: 100 us
constexpr uint32_t kSuspendHintNs = 200000;  // a sleeping waiter re-checks abort and time at least this often

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the thread sleep (up to the hint, in ns) until the phase completes, so
// waiting warps do not take issue slots from the softmax warps on their sub-partition.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Slow path of mbar_wait: sleep-wait with a time limit. A few plain try_waits come first: reading
// %globaltimer takes hundreds of cycles, so the clock for the limit starts only for a long wait.
// The body is force-inlined for kernels whose warpgroups change their register counts
// (setmaxnreg), where a call to an out-of-line function cannot be register-allocated.
__device__ __forceinline__ bool mbar_wait_slow_body(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                    int32_t* err, int site, bool honour_abort, uint64_t limit_ns) {
  for (int n = 0; n < 16; ++n)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if ((n & 7u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (global_timer() - t0 > limit_ns) {
        *abort_flag = 1;
        record_error(err, kErrTimeout, site);
        return false;
      }
    }
  }
}

__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                            int site, bool honour_abort, uint64_t limit_ns) {
  return mbar_wait_slow_body(bar, parity, abort_flag, err, site, honour_abort, limit_ns);
}

// Non-blocking test: true once the phase of parity `parity` has completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Busy-wait for the waits on the tile loop's critical path: a thread suspended in try_wait
// resumes several hundred cycles after the phase completes, a polling one within tens.
// Same limit and abort behaviour as mbar_wait. Poll without the clock first (reading
// %globaltimer takes hundreds of cycles and would delay noticing a phase that completes within
// the first few polls); then with the time limit.
__device__ __forceinline__ bool mbar_spin_slow_body(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                    int32_t* err, int site, uint64_t limit_ns) {
  for (int n = 0; n < 512; ++n)
    if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_test(bar, parity)) return true;
    if ((n & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_timer() - t0 > limit_ns) {
        *abort_flag = 1;
        record_error(err, kErrTimeout, site);
        return false;
      }
    }
  }
}

__device__ __noinline__ bool mbar_spin_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                            int site, uint64_t limit_ns) {
  return mbar_spin_slow_body(bar, parity, abort_flag, err, site, limit_ns);
}

__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                          int site, uint64_t limit_ns = kTimeoutNs) {
  if (mbar_test(bar, parity)) return true;
  return mbar_spin_slow(bar, parity, abort_flag, err, site, limit_ns);
}

// The same waits with the slow paths inlined (for kernels that use setmaxnreg).
__device__ __forceinline__ bool mbar_spin_inl(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                              int site, uint64_t limit_ns = kTimeoutNs) {
  if (mbar_test(bar, parity)) return true;
  return mbar_spin_slow_body(bar, parity, abort_flag, err, site, limit_ns);
}
__device__ __forceinline__ bool mbar_wait_inl(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                              int site, bool honour_abort = true, uint64_t limit_ns = kTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow_body(bar, parity, abort_flag, err, site, honour_abort, limit_ns);
}

// Wait for the phase of parity `parity` to complete; false on abort or timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int32_t* err,
                                          int site, bool honour_abort = true, uint64_t limit_ns = kTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, err, site, honour_abort, limit_ns);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// True in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (8-row x 128-byte atoms).
// lbo / sbo in bytes: K-major operands use sbo = 1024 (next 8 rows); MN-major
// operands also use lbo = distance between 64-element blocks of the MN dimension.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for the sm_100 family
  d |= (uint64_t)2 << 61;  // swizzle: 128 bytes
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, A K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

}  // namespace
}  // namespace cb

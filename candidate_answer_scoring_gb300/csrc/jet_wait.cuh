// mbarrier helpers and the bounded wait used by every spin-wait in the
// library's kernels.  A wait gives up after `limit_ns` of %globaltimer time:
// it raises the CTA's abort flag and records JET_ERR_TIMEOUT and the wait's
// location in the error word, so the kernel can drain and return instead of
// hanging the GPU.
#pragma once

#include "jet_head.cuh"

namespace jet {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Bounded wait for the phase of `bar` with the given parity.  Returns false if
// another role raised *abort_flag or if the wait exceeded limit_ns (then it
// raises the flag itself and, when err is given, records JET_ERR_TIMEOUT and
// `where` in err[2]).  The spinning part is out of line; mbar_wait below
// tries the barrier once inline first.
__device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                                            int where, unsigned long long limit_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        if (err != nullptr && atomicCAS(err, 0, JET_ERR_TIMEOUT) == 0) err[2] = where;
        return false;
      }
    }
  }
}

// A phase that has already completed (the common case for the MMA thread
// and the producer) costs one try_wait and no call (measured: multitoken
// head 2% faster than with the call on every wait).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                                          int where, unsigned long long limit_ns) {
  if (mbar_try_wait(smem_u32(bar), parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, err, where, limit_ns);
}

}  // namespace
}  // namespace jet

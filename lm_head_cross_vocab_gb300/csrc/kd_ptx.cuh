// Inline-PTX wrappers shared by the TMA / mbarrier kernels: shared-memory
// addresses, mbarriers (with time-bounded waits), bulk copies, fences.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kd_common.cuh"

namespace kd {
namespace ptx {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
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
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`
// (both addresses 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Lane 0 waits (bounded in time), the outcome is broadcast to the warp, and
// then every lane tests the completed phase itself: a successful try_wait is
// what gives a thread acquire ordering on the data the barrier guards (the
// bulk copies' bytes), which the broadcast alone does not.  On expiry the wait
// sets *abort and the status bit; later waits that see *abort give up at once.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status, bool honour_abort = true) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    if (!mbar_try(bar, parity)) {
      const uint64_t t0 = globaltimer();
      ok = 0;
      for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) {
          ok = 1;
          break;
        }
        if ((it & 63) == 0) {
          if (honour_abort && *abort) break;
          if (globaltimer() - t0 > kWaitLimitNs) {
            *abort = 1;
            set_status(status, KD_DEV_TIMEOUT);
            break;
          }
        }
      }
    }
  }
  const bool done = __shfl_sync(0xffffffffu, ok, 0) != 0;
  if (done) mbar_try(bar, parity);  // completed phase: succeeds at once, with acquire
  return done;
}

}  // namespace ptx
}  // namespace kd

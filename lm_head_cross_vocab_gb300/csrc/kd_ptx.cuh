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

// Every lane tests the phase (each successful try_wait gives that lane acquire
// ordering on the data the barrier guards, the bulk copies' bytes) and the warp
// leaves together once all lanes have seen it complete; the phase stays
// complete until this warp itself takes part in the next one.  Bounded in
// time: lane 0 checks the clock every 64 rounds; on expiry it sets *abort and
// the status bit and the warp gives up together; later waits that see *abort
// give up at once.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status, bool honour_abort = true,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
    if ((it & 63) == 0) {
      int give_up = 0;
      if ((threadIdx.x & 31) == 0) {
        if (honour_abort && *abort) {
          give_up = 1;
        } else if (globaltimer() - t0 > limit_ns) {
          *abort = 1;
          set_status(status, KD_DEV_TIMEOUT);
          give_up = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
  }
}

}  // namespace ptx
}  // namespace kd

// tma.cuh -- bulk-copy (TMA) staging for the streaming passes:
// mbarrier waits bounded by the global timer, 1-D bulk copies from global
// to shared memory with an L2 evict-first hint, and the once-per-device
// raise of a kernel's dynamic shared-memory limit.
#pragma once

#include <atomic>
#include <string>

#include "kernels.cuh"

namespace dopt {

constexpr unsigned long long kWaitNs = 1000000000ull;  // give up a wait after 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Polls an mbarrier phase for at most kWaitNs nanoseconds.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  if constexpr (DOPT_TMA_EVICT_FIRST) {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"((unsigned long long)__cvta_generic_to_global(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
  } else {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"((unsigned long long)__cvta_generic_to_global(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
  }
}

// Raises a kernel's dynamic shared-memory limit once per device (a later
// call, e.g. inside a stream capture, then issues nothing but the launch);
// `done` is one bit per device, owned by the caller per kernel.
template <typename K>
int allow_dynamic_smem(K kern, size_t smem, std::atomic<uint64_t>& done, const char* what) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (!bit || !(done.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
      return fail(DOPT_E_CUDA, std::string(what) + " smem attribute: " + cudaGetErrorString(e));
    done.fetch_or(bit);
  }
  return DOPT_OK;
}

}  // namespace dopt

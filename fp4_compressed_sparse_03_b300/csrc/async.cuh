// Asynchronous-copy building blocks shared by the TMA-fed kernels (sm_103a):
// mbarriers with bounded waits, 2D TMA tile loads, and host-side tensor-map encoding.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace csa2 {

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(saddr(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase.  Returns false when the iteration limit expires
// (then *abort is raised and CSA2_DEV_TIMEOUT reported) or when another thread of the
// CTA has already raised *abort.
__device__ __forceinline__ bool mbar_wait(volatile int* abort, uint64_t* b, uint32_t parity,
                                          int32_t* st, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try(b, parity)) return true;
    if ((i & 1023u) == 1023u && *abort) return false;
  }
  *abort = 1;
  report(st, CSA2_DEV_TIMEOUT);
  return false;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, uint64_t* bar, int x,
                                            int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(saddr(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(saddr(bar))
      : "memory");
}

// Host: 2D bf16 tensor map over a row-major [rows][cols] array, boxes of
// [box_rows][box_cols] with 128-byte swizzle (box_cols * 2 must be <= 128).
bool make_bf16_map(CUtensorMap* tm, const void* ptr, int64_t rows, int64_t cols, int box_cols,
                   int box_rows);

}  // namespace csa2

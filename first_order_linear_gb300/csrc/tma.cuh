// tma.cuh -- tensor-memory-accelerator tile copies and shared-memory barriers
// for the bulk time-major driver, plus the per-translation-unit device status
// word that bounded waits report to.
//
// A time-major [T, E] input is a 2-D tensor (E innermost).  One
// cp.async.bulk.tensor.2d copy moves a whole [rows, EW] tile of it -- EW
// consecutive environments over `rows` consecutive steps -- from global into
// shared memory, dense in [step][environment] order, and signals completion
// by the byte count on a shared-memory mbarrier.  Tiles reaching past E or T
// are zero-filled and still count their whole box.
#pragma once

#include <cuda.h>  // CUtensorMap (a 128-byte opaque descriptor)

#include <cstdint>

#include "scan_core.cuh"  // g_tu_status

namespace rlca {

// The tensor maps of one call: float inputs, then flag inputs, in the
// order of the estimator's staged_io() list (unused entries stay zero).
struct TmaSet {
  CUtensorMap f[4];
  CUtensorMap b[2];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// make the barrier initialisation visible to the async (TMA) proxy
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// this thread's arrival, announcing `bytes` of transactions still to land
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase of `bar` with the given parity to complete, for at most
// kWaitLimitNs of wall time; false (and the timeout bit in the status word)
// when it gave up.  A copy that never lands cannot hang the kernel.
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 0.2 s: thousands of times any healthy copy
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_tu_status, kStatusWaitTimeout);
      return false;
    }
  }
}

// one [rows, EW] tile at (x = first environment, y = first step) of a 2-D map
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace rlca

// Device wrappers for the asynchronous copy path of the sm_103a kernels:
// mbarriers, TMA tensor and bulk copies, shared-memory loads of 128-byte
// swizzled tiles, and L1-cached scale loads.  Every wait is bounded.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "../../include/moe_decode.h"

namespace moe {

constexpr unsigned long long kWaitNs = 200ull * 1000ull * 1000ull;  // bound of every device-side wait

MOE_DEV uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
MOE_DEV void mbar_init(uint64_t* b, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
MOE_DEV void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
MOE_DEV void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
MOE_DEV bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(su32(b)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait for the phase of `parity` to complete; false (and the status
// word set) when it did not within kWaitNs or when another wait already failed.
MOE_DEV bool mbar_wait(uint64_t* b, uint32_t parity, int* status) {
  if (mbar_try_wait(b, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (long it = 1; it < (1l << 26); ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 63) == 0) {
      if (*(volatile int*)status != 0) return false;
      if (globaltimer_ns() - t0 > kWaitNs) break;
    }
  }
  atomicExch(status, MOE_ERR_DEVICE_TIMEOUT);
  return false;
}
// Wait for copies this CTA has issued, bounded by time only: unlike mbar_wait
// it does not give up when another wait of the grid has failed, because issued
// copies always land and the CTA may not leave while one still writes into its
// shared memory.  False (and the status word set) only when the bound ran out.
MOE_DEV bool mbar_wait_landed(uint64_t* b, uint32_t parity, int* status) {
  if (mbar_try_wait(b, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (long it = 1; it < (1l << 26); ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 63) == 0 && globaltimer_ns() - t0 > kWaitNs) break;
  }
  atomicExch(status, MOE_ERR_DEVICE_TIMEOUT);
  return false;
}
MOE_DEV void tma_load_5d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(su32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(c2),
      "r"(c3), "r"(c4), "r"(su32(bar))
      : "memory");
}
MOE_DEV void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(su32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(su32(bar))
      : "memory");
}
MOE_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(su32(bar))
      : "memory");
}
MOE_DEV void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(su32(dst)), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(su32(bar))
      : "memory");
}
MOE_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
      "l"(src), "r"(bytes), "r"(su32(bar))
      : "memory");
}
MOE_DEV uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
// 16-byte chunk `c` of 128-byte row `f` of a tile written by TMA with the
// 128-byte swizzle (chunk index XOR row index mod 8, rows 1024-byte aligned).
MOE_DEV uint32_t swz(uint32_t base, int f, int c) { return base + f * 128 + ((c ^ (f & 7)) << 4); }

// L1-cached load of a block scale.  Weight and x scales are never written in
// this kernel; an h-scale row is read only after its expert's ready signal and
// is alone in its 128-byte line, so no stale line can be cached before it.
MOE_DEV float ld_ca(const float* p) {
  float v;
  asm volatile("ld.global.ca.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}


}  // namespace moe

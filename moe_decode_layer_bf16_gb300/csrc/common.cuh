// Device helpers shared by the sm_103a kernels of libmoe_decode.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

constexpr float kFp8Max = 448.f; // largest finite E4M3 magnitude

// ---------------------------------------------------------------- loads
// Weights are streamed once: read-only path, no L1 allocation.
MOE_DEV uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
// Data written earlier in the same kernel by another CTA: bypass L1.
MOE_DEV uint4 ld_l2(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
MOE_DEV float ld_l2f(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}
MOE_DEV float4 ld_l2f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p) : "memory");
  return v;
}
MOE_DEV int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Counter updates that publish (release) what this thread, and through a
// preceding CTA barrier its CTA, wrote before, and (acq_rel) acquire what the
// earlier updaters published: one instruction instead of fence + atomic.
MOE_DEV int atom_add_acq_rel(int* p, int v) {
  int r;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(r) : "l"(p), "r"(v) : "memory");
  return r;
}
MOE_DEV unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned r;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(r) : "l"(p), "r"(v) : "memory");
  return r;
}
MOE_DEV void red_add_release(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while its predecessor is still running; it waits
// here before touching the predecessor's results.  A no-op otherwise.
MOE_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream be scheduled before this one ends.
MOE_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
MOE_DEV unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- MMA
// D(16x8, f32) += A(16x32, e4m3, row) * B(32x8, e4m3, col)
MOE_DEV void mma_e4m3(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                      uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
MOE_DEV void mma_bf16(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                      uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64-byte span of a 16-row tile: thread (g = lane/4, q = lane%4) holds the
// 16 bytes at offset 16q of rows g (w0) and g+8 (w1), and the same 16 bytes of
// column n = g of the B operand (b).  The 64-byte span is two MMA k-steps.
// Any fixed permutation of k is allowed as long as A and B share it; this one
// lets every operand come straight from one 128-bit load per row.
MOE_DEV void mma_span_e4m3(float* c, const uint4& w0, const uint4& w1, const uint4& b) {
  mma_e4m3(c, w0.x, w1.x, w0.y, w1.y, b.x, b.y);
  mma_e4m3(c, w0.z, w1.z, w0.w, w1.w, b.z, b.w);
}
MOE_DEV void mma_span_bf16(float* c, const uint4& w0, const uint4& w1, const uint4& b) {
  mma_bf16(c, w0.x, w1.x, w0.y, w1.y, b.x, b.y);
  mma_bf16(c, w0.z, w1.z, w0.w, w1.w, b.z, b.w);
}

// ---------------------------------------------------------------- FP8 codes
// Four floats to four E4M3 codes (round to nearest even, saturating).
MOE_DEV uint32_t f32x4_to_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  // the first source goes to the upper byte of the pair
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Scale of one activation group: amax / 448 in IEEE fp32 (rounded up to a power
// of two for e8m0); 1 for an all-zero group.
MOE_DEV float group_scale(float amax, bool e8m0) {
  if (amax == 0.f) return 1.f;
  float s = __fdiv_rn(amax, kFp8Max);
  if (e8m0) {
    uint32_t bits = __float_as_uint(s);
    if (bits & 0x7fffffu) bits = ((bits >> 23) + 1u) << 23;
    s = __uint_as_float(bits);
  }
  return s;
}

MOE_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
MOE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

MOE_DEV float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
MOE_DEV float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
MOE_DEV uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 p = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&p);
}

}  // namespace moe

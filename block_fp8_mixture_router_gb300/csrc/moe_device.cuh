// Device helpers: warp-level MMA wrappers, streaming loads, conversions.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// ---- loads ------------------------------------------------------------------
// Weights are read once per forward: stream them past L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Activations written earlier in the same forward (possibly by another kernel
// of the chain or another CTA): read at L2.
__device__ __forceinline__ uint4 ld_cg16(const void* p) {
  return __ldcg(reinterpret_cast<const uint4*>(p));
}

// ---- programmatic dependent launch -------------------------------------------
// Without the launch attribute both are no-ops, so the same kernel serves
// plain and chained launches.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Ask L2 to fetch [p, p + bytes) (16-byte aligned, multiple of 16); no wait.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}

// Prefetch share `part` of `parts` equal shares of [p, p + bytes), in pieces.
__device__ __forceinline__ void prefetch_l2_share(const void* p, size_t bytes, int part, int parts) {
  const size_t per = ((bytes + parts - 1) / parts + 15) & ~(size_t)15;
  size_t lo = per * part;
  size_t hi = lo + per < bytes ? lo + per : bytes;
  const char* c = static_cast<const char*>(p);
  while (lo < hi) {
    uint32_t n = (uint32_t)((hi - lo) < 65536 ? (hi - lo) : 65536);
    n &= ~15u;
    if (n == 0) break;
    prefetch_l2(c + lo, n);
    lo += n;
  }
}

// ---- warp MMAs ------------------------------------------------------------
// D(16x8, f32) += A(16x32, e4m3, row) * B(32x8, e4m3, col)
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64-byte slice of K for a 16-row e4m3 tile, read straight from global.
//
// The dot products do not depend on the order of K, so K is relabelled: lane
// (g = lane/4, q = lane%4) loads 16 contiguous bytes at byte offset 16*q of the
// slice from rows g and g+8, and the same 16 bytes of its token g's row.  Its
// bytes 0-3/4-7 serve as the first MMA's k-labels 4q..4q+3 / 16+4q..16+4q+3 and
// bytes 8-11/12-15 as the second MMA's.  A and B use the same relabelling, so
// each MMA pair covers the slice's 64 k exactly once.
__device__ __forceinline__ void mma_e4m3_k64(float (&d)[4], const uint4& a_lo, const uint4& a_hi,
                                             const uint4& b) {
  mma_e4m3(d, a_lo.x, a_hi.x, a_lo.y, a_hi.y, b.x, b.y);
  mma_e4m3(d, a_lo.z, a_hi.z, a_lo.w, a_hi.w, b.z, b.w);
}

// The bf16 analogue over a 32-element slice: lane loads 8 elements at element
// offset 8*q; elements 0-1/2-3 feed the first MMA's labels 2q..2q+1 /
// 8+2q..8+2q+1, elements 4-5/6-7 the second MMA's.
__device__ __forceinline__ void mma_bf16_k32(float (&d)[4], const uint4& a_lo, const uint4& a_hi,
                                             const uint4& b) {
  mma_bf16(d, a_lo.x, a_hi.x, a_lo.y, a_hi.y, b.x, b.y);
  mma_bf16(d, a_lo.z, a_hi.z, a_lo.w, a_hi.w, b.z, b.w);
}

// ---- conversions ------------------------------------------------------------
__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// e4m3 codes of four values, first value in the lowest byte: the hardware
// conversion, round to nearest even, saturating to +-448, NaN to the NaN code.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(lo) : "f"(v1), "f"(v0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(hi) : "f"(v3), "f"(v2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Quantise four values of a group with scale s: codes of v/s (IEEE division).
__device__ __forceinline__ uint32_t quant4(float v0, float v1, float v2, float v3, float s) {
  return e4m3x4(__fdiv_rn(v0, s), __fdiv_rn(v1, s), __fdiv_rn(v2, s), __fdiv_rn(v3, s));
}

// silu(z) = z / (1 + e^-z) with the fast exponential and divide; the
// exponent is clamped so the divisor stays finite (silu(z) is then ~0).
__device__ __forceinline__ float silu_f32(float z) {
  return __fdividef(z, 1.0f + __expf(fminf(-z, 80.0f)));
}

// Logistic sigmoid with the fast exponential and divide.
__device__ __forceinline__ float sigmoid_f32(float v) {
  return __fdividef(1.0f, 1.0f + __expf(fminf(-v, 80.0f)));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Scale of one quantisation group from its amax: amax / 448 (IEEE division),
// 1 for an all-zero group.
__device__ __forceinline__ float group_scale(float amax) {
  return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

}  // namespace moe

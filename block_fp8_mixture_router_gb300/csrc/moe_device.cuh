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
// v rounded to bf16 (nearest even) and back, with integer operations: the
// same value as the conversion for every finite v and infinity, on the
// full-rate integer pipe rather than the conversion unit.  NaN stays NaN.
__device__ __forceinline__ float bf16_round(float v) {
  const uint32_t u = __float_as_uint(v);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return v;
  return __uint_as_float((u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u);
}

// e4m3 codes of four values, first value in the lowest byte: the hardware
// conversion, round to nearest even, saturating to +-448, NaN to the NaN code.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(lo) : "f"(v1), "f"(v0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(hi) : "f"(v3), "f"(v2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Reciprocal of a divisor for div_shared: RN(1/s) when s is a normal number
// in [2^-125, 2^126), else 0, which sends div_shared to the IEEE division.
__device__ __forceinline__ float div_recip(float s) {
  const uint32_t es = (__float_as_uint(s) >> 23) & 0xFFu;
  return (es >= 2u && es <= 252u) ? __frcp_rn(s) : 0.0f;
}

// The IEEE division kept out of line, so that the rare operands div_shared
// hands to it do not grow the code of every call site.
static __device__ __noinline__ float div_ieee(float v, float s) { return __fdiv_rn(v, s); }

// v / s rounded to nearest even, bit for bit the IEEE quotient, for a divisor
// shared by many dividends (y = div_recip(s)).  One Newton step from v*y
// leaves q within an ulp of v/s; for such a q the FMA remainder r = v - q*s
// is exact (the property Markstein's division rests on), so comparing |r|
// with s times half the ulp of q -- the ulp below when q is a power of two
// and v/s lies below it -- decides between q and its neighbour.  Dividends
// below 2^-95 or near overflow, and quotients below 2^-63, whose remainder or
// half-ulp product could leave the normal range, take the IEEE division.
__device__ __forceinline__ float div_shared_fast(float v, float s, float y, bool& rare) {
  const uint32_t ev = (__float_as_uint(v) >> 23) & 0xFFu;
  rare = (y == 0.0f) | (ev > 252u) | ((ev < 32u) & (v != 0.0f));
  float q = v * y;
  if (ev < 32u) return q;  // a signed zero
  q = fmaf(fmaf(-q, s, v), y, q);
  const float r = fmaf(-q, s, v);
  const uint32_t qb = __float_as_uint(q);
  const uint32_t e = (qb >> 23) & 0xFFu;
  rare |= (e < 64u) | (e > 253u);
  const float half = s * __uint_as_float((e - 24u) << 23);
  const bool down = (r < 0.0f) != (q < 0.0f);
  const float h = (down && (qb & 0x7FFFFFu) == 0u) ? 0.5f * half : half;
  const float ar = fabsf(r);
  if (ar < h || (ar == h && !(qb & 1u))) return q;
  return __uint_as_float(down ? qb - 1u : qb + 1u);
}

// (div_shared_fast sets `rare` where the steps above cannot decide and the
// IEEE division must; its result is then not to be used.  Callers that
// divide several values at once take the fast path for all of them first and
// the rare fallback after, so no out-of-line call splits their code.)
__device__ __forceinline__ float div_shared(float v, float s, float y) {
  bool rare;
  const float q = div_shared_fast(v, s, y, rare);
  return rare ? div_ieee(v, s) : q;
}

// Codes of v/s through the IEEE quotients, out of line (the rare groups
// quant4 cannot settle from the product).
static __device__ __noinline__ uint32_t quant4_exact(float v0, float v1, float v2, float v3,
                                                     float s) {
  const float y = div_recip(s);
  return e4m3x4(div_shared(v0, s, y), div_shared(v1, s, y), div_shared(v2, s, y),
                div_shared(v3, s, y));
}

// Does the e4m3 rounding of a quotient need more than the product q = v*y
// (y within a few ulps of 1/s)?  q is then within 4 fp32 ulps of the IEEE
// quotient, and the two round to the same e4m3 code unless an e4m3 rounding
// midpoint lies between them: for |q| in e4m3's normal range the midpoints
// are the floats whose 20 mantissa bits below the kept 3 read 0x80000, so a
// window of 8 ulps around them is flagged, and so is e4m3's subnormal range
// (|q| < 2^-6, q != 0).  Saturation needs nothing: everything above 448
// becomes 448.
__device__ __forceinline__ bool e4m3_undecided(float q) {
  const uint32_t u = __float_as_uint(q) & 0x7FFFFFFFu;
  return (u - 1u < 0x3C800000u - 1u) | ((u & 0xFFFFFu) - 0x7FFF8u < 16u);
}

// Quantise four values of a group with scale s: the e4m3 codes of the IEEE
// quotients v/s, taken from the products v * rcp(s) wherever those decide
// them (all but a few groups in a million), else from the exact quotients.
// The codes from the products alone; `undecided` is set where quant4 would
// take the exact quotients instead (the codes returned are then not to be
// used).
__device__ __forceinline__ uint32_t quant4_fast(float v0, float v1, float v2, float v3, float s,
                                                bool& undecided) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(s));
  const float q0 = v0 * y, q1 = v1 * y, q2 = v2 * y, q3 = v3 * y;
  const uint32_t es = (__float_as_uint(s) >> 23) & 0xFFu;
  undecided = (es - 2u > 250u) | e4m3_undecided(q0) | e4m3_undecided(q1) | e4m3_undecided(q2) |
              e4m3_undecided(q3);
  return e4m3x4(q0, q1, q2, q3);
}

__device__ __forceinline__ uint32_t quant4(float v0, float v1, float v2, float v3, float s) {
  bool undecided;
  const uint32_t c = quant4_fast(v0, v1, v2, v3, s, undecided);
  return undecided ? quant4_exact(v0, v1, v2, v3, s) : c;
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
  return amax > 0.0f ? div_shared(amax, 448.0f, 0x1.24924ap-9f) : 1.0f;  // RN(1/448)
}

// group_scale without the out-of-line division: `rare` is set where
// group_scale must be called instead.
__device__ __forceinline__ float group_scale_fast(float amax, bool& rare) {
  const float q = div_shared_fast(amax, 448.0f, 0x1.24924ap-9f, rare);
  rare &= amax > 0.0f;
  return amax > 0.0f ? q : 1.0f;
}

}  // namespace moe

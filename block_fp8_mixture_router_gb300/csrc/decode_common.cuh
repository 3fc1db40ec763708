// Device helpers of the role-split decode kernels: mbarriers and 1-D bulk
// copies, bounded waits, and the launch-tagged words the CTAs exchange
// through global memory ({tag in the high 32 bits, value bits in the low}).
#pragma once

#include "moe_rowops.cuh"

namespace moe {
namespace dec {

constexpr long long kSpin = 1ll << 22;  // tries before a wait gives up

__device__ __forceinline__ uint32_t sa(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(sa(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(sa(bar)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.  The
// lines it reads are marked evict-first in L2: weights stream through once
// per launch, and without the hint they push out what every launch reuses
// (the kernel's code, x, the exchange words).
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "{\n .reg .b64 pol;\n createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n"
      " cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], pol;\n}\n" ::"r"(sa(dst)),
      "l"(src), "r"(bytes), "r"(sa(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(sa(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void copy_wait(uint64_t* bar, uint32_t parity, int* status) {
  long long it = 0;
  while (!mbar_test(bar, parity)) {
    if (++it > kSpin) {
      atomicExch(status, 1);
      break;
    }
  }
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}

// The value of a tagged word once its tag is current (bounded).
__device__ __forceinline__ float poll_tagged(const unsigned long long* p, unsigned long long tag,
                                             int* status) {
  unsigned long long v = ld_relaxed64(p);
  long long it = 0;
  while ((v & 0xFFFFFFFF00000000ull) != tag) {
    if (++it > kSpin) {
      atomicExch(status, 1);
      break;
    }
    if (it > 16) __nanosleep(32);
    v = ld_relaxed64(p);
  }
  return __uint_as_float((uint32_t)v);
}

// Values of n tagged words src[0..n) into dst[0..n) (any memory), the
// calling CTA's threads striding over them: each thread issues its loads in
// batches of eight before it looks at any (one round trip per batch), and
// re-polls only the words whose tag was not yet current.
template <int kThreadsPerCta, typename Store>
__device__ __forceinline__ void poll_range(const unsigned long long* src, int n,
                                           unsigned long long tag, int* status, Store store) {
  constexpr int kB = 8;
  for (int i0 = threadIdx.x; i0 < n; i0 += kB * kThreadsPerCta) {
    unsigned long long v[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = i0 + u * kThreadsPerCta;
      v[u] = i < n ? ld_relaxed64(src + i) : tag;
    }
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = i0 + u * kThreadsPerCta;
      if (i < n) {
        float f = __uint_as_float((uint32_t)v[u]);
        if ((v[u] & 0xFFFFFFFF00000000ull) != tag) f = poll_tagged(src + i, tag, status);
        store(i, f);
      }
    }
  }
}

// The same for n words at gathered addresses addr(i).
template <int kThreadsPerCta, typename Addr, typename Store>
__device__ __forceinline__ void poll_gather(int n, unsigned long long tag, int* status, Addr addr,
                                            Store store) {
  constexpr int kB = 8;
  for (int i0 = threadIdx.x; i0 < n; i0 += kB * kThreadsPerCta) {
    unsigned long long v[kB];
    const unsigned long long* p[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = i0 + u * kThreadsPerCta;
      p[u] = i < n ? addr(i) : nullptr;
      v[u] = i < n ? ld_relaxed64(p[u]) : tag;
    }
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int i = i0 + u * kThreadsPerCta;
      if (i < n) {
        float f = __uint_as_float((uint32_t)v[u]);
        if ((v[u] & 0xFFFFFFFF00000000ull) != tag) f = poll_tagged(p[u], tag, status);
        store(i, f);
      }
    }
  }
}

__device__ __forceinline__ void publish(unsigned long long* p, unsigned long long tag, float v) {
  st_relaxed64(p, tag | __float_as_uint(v));
}

__device__ __forceinline__ uint4 lds16(const void* p) { return *reinterpret_cast<const uint4*>(p); }

__host__ __device__ __forceinline__ size_t al16(size_t v) { return (v + 15) & ~(size_t)15; }

// [src, src + n floats) widened to 16-byte boundaries for one bulk copy (the
// scale arrays start 16-byte aligned and span whole 16-byte units).
__device__ __forceinline__ uint32_t span16(const float* src, int n, const float** lo, int* delta) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(src) & ~(uintptr_t)15;
  const uintptr_t a1 = (reinterpret_cast<uintptr_t>(src + n) + 15) & ~(uintptr_t)15;
  *lo = reinterpret_cast<const float*>(a0);
  *delta = (int)((reinterpret_cast<uintptr_t>(src) - a0) / 4);
  return (uint32_t)(a1 - a0);
}

}  // namespace dec
}  // namespace moe

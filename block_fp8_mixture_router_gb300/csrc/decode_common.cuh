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

// Tries before a poll gives up: kSpin unless the context set a limit in
// status[kPollLimitWord] (copy waits keep kSpin, so a launch never leaves a
// copy in flight).
__device__ __forceinline__ long long poll_limit(const int* status) {
  const int lim = *reinterpret_cast<const volatile int*>(status + kPollLimitWord);
  return lim > 0 ? (long long)lim : kSpin;
}

// The value of a tagged word once its tag is current (bounded).  On giving
// up it sets the status flag and returns whatever value the word holds.
__device__ __forceinline__ float poll_tagged(const unsigned long long* p, unsigned long long tag,
                                             int* status) {
  unsigned long long v = ld_relaxed64(p);
  if ((v & 0xFFFFFFFF00000000ull) == tag) return __uint_as_float((uint32_t)v);
  const long long lim = poll_limit(status);
  long long it = 0;
  while ((v & 0xFFFFFFFF00000000ull) != tag) {
    if (++it > lim) {
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

// ---- launch tags ---------------------------------------------------------------
// A launch's tag is the context's epoch + 1; the last CTA to leave publishes
// the tag as the new epoch.  A poll accepts a word whose tag equals its
// launch's, so a tag must never come back while a word written under it
// could still be read.  On the launch whose last tag reaches kTagClear the
// last CTA instead clears every exchange word and restarts the epoch at 0:
// tags then start again at 1 over words that all read 0.  (A chain launch
// uses one tag per layer, at most kMaxChain, so tags stay below kTagWrap.)
// Every CTA of that launch fences its exchange writes before it arrives at
// the exit counter, so none can land after the clear.
// Exchange words of the context (tagged logits, then the decode exchange
// words), as the context allocates them.
__device__ __forceinline__ void clear_exchange_words(const KArgs& a) {
  const size_t n_log = (size_t)kDecodeRows * a.d.E;
  const size_t n_xw = (size_t)kDecodeRows * ((size_t)a.d.k * a.d.I + (size_t)a.d.k * a.d.H +
                                             a.d.Is + a.d.H);
  for (size_t i = threadIdx.x; i < n_log; i += blockDim.x) a.w.tlog[i] = 0ull;
  for (size_t i = threadIdx.x; i < n_xw; i += blockDim.x) a.w.xw[i] = 0ull;
}

// The exit of a tagged-exchange launch; every thread of the CTA calls it.
// tag: the launch's last tag.
__device__ __forceinline__ void launch_exit(const KArgs& a, int tag) {
  int* bar_exit = a.w.done + 3;
  int* epoch = a.w.done + 4;
  __shared__ int s_last;
  __syncthreads();
  if (tag < kTagClear) {
    // The next launch reads the epoch, the outputs and the exchange words
    // only after this grid has completed, and stale words carry older tags.
    if (threadIdx.x == 0) {
      const int old = atomicAdd(bar_exit, 1);
      if (old == (int)gridDim.x - 1) {
        *bar_exit = 0;
        if (a.chain.n) a.w.done[6] = 0;  // the chain's combine counter
        *epoch = tag;
      }
    }
    return;
  }
  if (threadIdx.x == 0) {
    __threadfence();  // release: this CTA's exchange writes before its arrival
    s_last = atomicAdd(bar_exit, 1) == (int)gridDim.x - 1;
    __threadfence();  // acquire: every other CTA's writes before the clear
  }
  __syncthreads();
  if (!s_last) return;
  clear_exchange_words(a);
  __syncthreads();
  if (threadIdx.x == 0) {
    *bar_exit = 0;
    if (a.chain.n) a.w.done[6] = 0;
    *epoch = 0;
  }
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

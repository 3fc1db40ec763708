// Per-row device routines shared by the prompt and decode kernels: the
// activation quantisation with the shared-expert gate, and the top-k.
#pragma once

#include <math.h>

#include "moe_device.cuh"

namespace moe {

// ---- activation quantisation (1 x 128 groups) and the shared gate ----------
// One CTA per row (any multiple of 32 threads up to 1024).  Warp w quantises
// groups w, w + nw, ...; each lane holds 4 consecutive values of the group.
// With one scale per row (a.d.per_row) every group takes the row's scale.
// The gate dot product x . g is reduced in a fixed order (per-thread strided
// sums, then warps 0..nw-1).
// Largest |value| of four bf16 values packed in a uint2.
__device__ __forceinline__ float amax4(const uint2& raw) {
  const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
  const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
  return fmaxf(fmaxf(fabsf(__low2float(p0)), fabsf(__high2float(p0))),
               fmaxf(fabsf(__low2float(p1)), fabsf(__high2float(p1))));
}

// Scale of a whole row (one scale per row): amax over the row's H values,
// reduced over the CTA's warps (every thread calls it; it synchronises the
// CTA twice).  red: at least nw floats of shared memory.
__device__ __forceinline__ float row_scale(const bf16* xr, int H, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float m = 0.0f;
  for (int base = 4 * threadIdx.x; base < H; base += 4 * blockDim.x)
    m = fmaxf(m, amax4(*reinterpret_cast<const uint2*>(xr + base)));
  m = warp_max(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float r = 0.0f;
  for (int w = 0; w < nw; ++w) r = fmaxf(r, red[w]);
  __syncthreads();  // red is free again
  return group_scale(r);
}

__device__ __forceinline__ void quant_row_and_gate(const KArgs& a, int t) {
  __shared__ float red[32];
  const int H = a.d.H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const bf16* xr = a.x + (size_t)t * H;
  const int ngroups = H / kGroup;
  const float rs = a.d.per_row ? row_scale(xr, H, red) : 0.0f;
  for (int gi = warp; gi < ngroups; gi += nw) {
    const int base = gi * kGroup + 4 * lane;
    uint2 raw = *reinterpret_cast<const uint2*>(xr + base);
    __nv_bfloat162 p0 = *reinterpret_cast<__nv_bfloat162*>(&raw.x);
    __nv_bfloat162 p1 = *reinterpret_cast<__nv_bfloat162*>(&raw.y);
    float v[4] = {__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1)};
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    m = warp_max(m);
    const float s = a.d.per_row ? rs : group_scale(m);
    const uint32_t packed = quant4(v[0], v[1], v[2], v[3], s);
    *reinterpret_cast<uint32_t*>(a.w.xq + (size_t)t * H + base) = packed;
    if (lane == 0) a.w.sx[(size_t)t * ngroups + gi] = s;
  }
  float acc = 0.0f;
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    acc = fmaf(__bfloat162float(xr[i]), __bfloat162float(a.L.gate[i]), acc);
  acc = warp_sum(acc);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = 0.0f;
    for (int w = 0; w < nw; ++w) v += red[w];
    a.w.gamma[t] = sigmoid_f32(v);
  }
}

// ---- top-k + renormalised softmax ------------------------------------------
// One warp per row.  Logits become order-preserving 32-bit keys (-0 folded
// into +0 first, so equal values have equal keys).  Lane l holds experts
// l, l+32, ...; each round every lane offers its largest remaining key (the
// lowest expert among equal keys), and the warp takes the largest key and,
// among the lanes offering it, the lowest expert: the k largest logits, ties
// to the lower index, in rank order.  The softmax over the selected logits is
// taken with one lane per rank (k <= 32).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The logit the router selects and weighs by: the fp32 sum, or in the
// bf16-logit variant that sum rounded to bf16 (nearest, ties to even).
__device__ __forceinline__ float route_logit(float v, int rbf16) {
  return rbf16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

// kCg: read the logits at L2 (they were written by other CTAs of the same
// kernel).
// rbf16: route on the logits rounded to bf16 (route_logit).
template <bool kCg = false>
__device__ __forceinline__ void topk_row(const float* logits, int E, int k, int* idx_out,
                                         float* w_out, int rbf16 = 0) {
  const int lane = threadIdx.x & 31;
  uint32_t key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? order_key(route_logit(kCg ? __ldcg(logits + e) : logits[e], rbf16)) : 0u;
  }
  uint32_t my_key = 0u, my_e = 0u;
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool better = key[i] > bk;
      bk = better ? key[i] : bk;
      bi = better ? i : bi;
    }
    const uint32_t mx = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t win =
        __reduce_min_sync(0xffffffffu, bk == mx ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu);
    const bool mine = (int)(win & 31u) == lane;
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = (mine & (i == (int)(win >> 5))) ? 0u : key[i];
    my_key = lane == j ? mx : my_key;
    my_e = lane == j ? win : my_e;
  }
  const float top = key_value(__shfl_sync(0xffffffffu, my_key, 0));
  const float ex = lane < k ? __expf(key_value(my_key) - top) : 0.0f;
  const float den = warp_sum(ex);
  if (lane < k) {
    idx_out[lane] = (int)my_e;
    w_out[lane] = __fdividef(ex, den);
  }
}

// ---- top-k of one row with all warps of the CTA -------------------------------
// kWarps warps of 32 hold experts 0..32*kWarps-1 (E <= 32*kWarps, k <= 16).
// Level 1: each warp takes the k best of its 32 experts in k rounds; a
// round's winner is the largest key and, among equal keys, the lowest lane,
// i.e. the lowest expert.  Level 2 ranks the kWarps*k candidates against each
// other in parallel.  Both levels give the order of topk_row (larger key
// first, lower expert on equal keys).  cand_key / cand_id are shared-memory
// scratch of 2*kWarps*16 entries each; idx_out / w_out (shared memory)
// receive the experts in rank order and their softmax weights.  The caller
// synchronises the CTA afterwards.
// Barrier of the first kWarps warps of the CTA (named barrier 2): the fast
// top-k below synchronises only the warps that run it.
template <int kWarps>
__device__ __forceinline__ void topk_bar() {
  asm volatile("bar.sync 2, %0;\n" ::"n"(32 * kWarps) : "memory");
}

// lg, cand_key and cand_id must be 16-byte aligned (they are read as
// vectors).  Run by the first kWarps warps of the CTA (all of them call it).
// Fast variant for k <= 8 and a multiple of four warps: every thread ranks
// its own expert among its warp's 32 (counting the keys that beat it, read
// from shared memory as broadcast vectors, no serial rounds); the k best of
// each warp go to slots [warp][rank]; then four threads per candidate count,
// over a quarter of the lists each, the candidates that beat it, and the
// candidates ranked below k write the result.  Same order as below.
template <int kWarps>
__device__ void topk_one_row_fast(const float* lg, int E, int k, uint32_t* cand_key,
                                  uint32_t* cand_id, int* idx_out, float* w_out) {
  static_assert(kWarps % 4 == 0, "lists split in quarters");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = 32 * warp + lane;
  const uint32_t my = e < E ? order_key(lg[e]) : 0u;
  {
    int r = 0;
    const int base = 32 * warp;
    if (base + 32 <= E) {
      const float4* row = reinterpret_cast<const float4*>(lg + base);
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 v = row[j4];
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t kj = order_key(vv[c]);
          const int j = 4 * j4 + c;
          r += ((kj > my) | ((kj == my) & (j < lane))) ? 1 : 0;
        }
      }
    } else {
      for (int j = 0; j < 32; ++j) {
        const uint32_t kj = base + j < E ? order_key(lg[base + j]) : 0u;
        r += ((kj > my) | ((kj == my) & (j < lane))) ? 1 : 0;
      }
    }
    if (r < k) {
      cand_key[warp * 8 + r] = my;
      cand_id[warp * 8 + r] = (uint32_t)e;
    }
  }
  topk_bar<kWarps>();
  uint32_t* rank_key = cand_key + 8 * kWarps;
  uint32_t* rank_id = cand_id + 8 * kWarps;
  {
    const int c = threadIdx.x >> 2, part = threadIdx.x & 3;
    int rank = 0;
    uint32_t K = 0u, D = 0u;
    const bool have = c < 8 * kWarps;
    if (have) {
      K = cand_key[c];
      D = cand_id[c];
      constexpr int kPer = kWarps / 4;
#pragma unroll
      for (int w = 0; w < kPer; ++w) {
        const int w2 = part * kPer + w;
        const uint4 k0 = *reinterpret_cast<const uint4*>(cand_key + w2 * 8);
        const uint4 k1 = *reinterpret_cast<const uint4*>(cand_key + w2 * 8 + 4);
        const uint4 d0 = *reinterpret_cast<const uint4*>(cand_id + w2 * 8);
        const uint4 d1 = *reinterpret_cast<const uint4*>(cand_id + w2 * 8 + 4);
        const uint32_t K8[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        const uint32_t D8[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2)
          rank += ((s2 < k) & ((K8[s2] > K) | ((K8[s2] == K) & (D8[s2] < D)))) ? 1 : 0;
      }
    }
    rank += __shfl_xor_sync(0xffffffffu, rank, 1);
    rank += __shfl_xor_sync(0xffffffffu, rank, 2);
    if (have && part == 0 && (c & 7) < k && rank < k) {
      rank_key[rank] = K;
      rank_id[rank] = D;
    }
  }
  topk_bar<kWarps>();
  if (warp == 0) {
    const uint32_t my_key = lane < k ? rank_key[lane] : 0u;
    const float top = key_value(__shfl_sync(0xffffffffu, my_key, 0));
    const float ex = lane < k ? __expf(key_value(my_key) - top) : 0.0f;
    const float den = warp_sum(ex);
    if (lane < k) {
      idx_out[lane] = (int)rank_id[lane];
      w_out[lane] = __fdividef(ex, den);
    }
  }
}

template <int kWarps>
__device__ __noinline__ void topk_one_row_general(const float* lg, int E, int k,
                                                  uint32_t* cand_key, uint32_t* cand_id,
                                                  int* idx_out, float* w_out);

template <int kWarps>
__device__ __forceinline__ void topk_one_row(const float* lg, int E, int k, uint32_t* cand_key,
                                             uint32_t* cand_id, int* idx_out, float* w_out) {
  if constexpr (kWarps % 4 == 0) {
    if (k <= 8 && E <= 32 * kWarps) {
      topk_one_row_fast<kWarps>(lg, E, k, cand_key, cand_id, idx_out, w_out);
      return;
    }
  }
  topk_one_row_general<kWarps>(lg, E, k, cand_key, cand_id, idx_out, w_out);
}

// The general path (any k <= 16), out of line so that its code stays out of
// the fast path's way.
template <int kWarps>
__device__ __noinline__ void topk_one_row_general(const float* lg, int E, int k,
                                                  uint32_t* cand_key, uint32_t* cand_id,
                                                  int* idx_out, float* w_out) {
  static_assert(kWarps <= 32, "one list per lane");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    const int e = 32 * warp + lane;
    uint32_t key = e < E ? order_key(lg[e]) : 0u;
    uint32_t ck = 0u, cid = 0xFFFFFFFFu;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
      const uint32_t mx = __reduce_max_sync(0xffffffffu, key);
      const int wl = __ffs(__ballot_sync(0xffffffffu, key == mx)) - 1;
      key = lane == wl ? 0u : key;
      ck = lane == j ? mx : ck;
      cid = lane == j ? (mx ? (uint32_t)(32 * warp + wl) : 0xFFFFFFFFu) : cid;
    }
    if (lane < k) {
      cand_key[warp * kMaxTopK + lane] = ck;
      cand_id[warp * kMaxTopK + lane] = cid;
    }
  }
  __syncthreads();
  // Level 2: candidate c = (list w, place j) of the kWarps*16 slots takes
  // rank = number of valid candidates that beat it (larger key, or equal
  // key and lower expert); every thread reads all slots (broadcast loads).
  constexpr int kC = kWarps * kMaxTopK;
  static_assert(kC <= 32 * kWarps, "one thread per candidate");
  uint32_t* rank_key = cand_key + kC;  // callers provide 2*kC-entry scratch
  uint32_t* rank_id = cand_id + kC;
  if (threadIdx.x < kC) {
    const int c = threadIdx.x;
    const bool valid = (c % kMaxTopK) < k && cand_key[c] != 0u;
    const uint32_t K = cand_key[c], D = cand_id[c];
    int rank = 0;
    if (k <= 8) {
      // the first 8 slots of every list in registers (16-byte loads issued
      // together: shared loads in a dependent loop are latency-bound)
      uint4 kv[2 * kWarps], dv[2 * kWarps];
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) {
        kv[2 * w2] = *reinterpret_cast<const uint4*>(cand_key + w2 * kMaxTopK);
        kv[2 * w2 + 1] = *reinterpret_cast<const uint4*>(cand_key + w2 * kMaxTopK + 4);
        dv[2 * w2] = *reinterpret_cast<const uint4*>(cand_id + w2 * kMaxTopK);
        dv[2 * w2 + 1] = *reinterpret_cast<const uint4*>(cand_id + w2 * kMaxTopK + 4);
      }
#pragma unroll
      for (int v = 0; v < 2 * kWarps; ++v) {
        const uint32_t K4[4] = {kv[v].x, kv[v].y, kv[v].z, kv[v].w};
        const uint32_t D4[4] = {dv[v].x, dv[v].y, dv[v].z, dv[v].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const bool ok2 = 4 * (v & 1) + t < k;
          rank += (ok2 & ((K4[t] > K) | ((K4[t] == K) & (D4[t] < D)))) ? 1 : 0;
        }
      }
    } else {
      for (int w2 = 0; w2 < kWarps; ++w2)
        for (int j2 = 0; j2 < k; ++j2) {
          const uint32_t K2 = cand_key[w2 * kMaxTopK + j2], D2 = cand_id[w2 * kMaxTopK + j2];
          rank += ((K2 > K) | ((K2 == K) & (D2 < D))) ? 1 : 0;
        }
    }
    if (valid && rank < k) {
      rank_key[rank] = K;
      rank_id[rank] = D;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t my_key = lane < k ? rank_key[lane] : 0u;
    const float top = key_value(__shfl_sync(0xffffffffu, my_key, 0));
    const float ex = lane < k ? __expf(key_value(my_key) - top) : 0.0f;
    const float den = warp_sum(ex);
    if (lane < k) {
      idx_out[lane] = (int)rank_id[lane];
      w_out[lane] = __fdividef(ex, den);
    }
  }
}

}  // namespace moe

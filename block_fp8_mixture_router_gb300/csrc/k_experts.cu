// Routed block-FP8 SwiGLU experts, the bf16 shared expert, and the combine.
//
// Expert arithmetic: PR #939 "Fish Audio Drama 3 text to speech on one CUDA
// GPU", sections "What it adds" (drama3_fp8.cu: FP8 experts on FP8 rows with
// per-row scales) and "Precision" (dynamic e4m3 activations, amax / 448).
// SwiGLU outputs: commit "one SwiGLU launch for the routed and shared
// experts" (routed rows stored as their FP8 quantisation, shared rows bf16).
// Combine: commit "MoE combine on 8-wide vectors" (16-byte loads, 8 outputs
// per thread, every sum keeps its order).
//
// Work units.  A routed gate/up unit is (expert chunk of <= 16 rows, 16 gate
// rows + the 16 matching up rows); its MMA tiles put 8 gate rows over the 8
// matching up rows so one thread ends up holding both halves of a SwiGLU.  A
// 128-column group of the SwiGLU output is finished by 8 units; the last of
// them to arrive (an arrival counter, reset by that unit) quantises the group,
// so the result never depends on which CTA ran which unit.  K is split over
// the 8 warps in 64-byte slices; each slice's MMA partial is scaled by its
// 128-block's weight scale times the row's activation scale, and the warps'
// sums are added in warp order.
#include <math.h>

#include "moe_device.cuh"

namespace moe {

namespace {

constexpr int kWarps = 8;

constexpr int kMaxNbh = 4096 / kGroup;  // 128-wide K groups of H at most

struct __align__(16) Smem {
  float red[kWarps][2][2][4][32];  // [warp][tile][n-tile][c][lane]
  float sxs[kChunk][kMaxNbh];      // a routed unit's token scales [row][K group]
  float swg[kMaxNbh], swu[kMaxNbh];  // its gate and up weight-block scales
  int flag;
};

__device__ __forceinline__ float& red_at(Smem& s, int w, int tile, int nt, int c, int lane) {
  return s.red[w][tile][nt][c][lane];
}

// ---- routed gate/up ----------------------------------------------------------
__device__ void gateup_routed(const KArgs& a, Smem& sm, int chunk_id, int mp) {
  const int H = a.d.H, I = a.d.I, k = a.d.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, q = lane & 3;
  const int4 ch = a.w.chunks[chunk_id];
  const int e = ch.x, s0 = ch.y, ntok = ch.z;
  const int n0 = 16 * mp;
  const int nbh = H / kGroup;
  const uint8_t* W = a.L.w13 + (size_t)e * 2 * I * H;
  const float* S = a.L.s13 + (size_t)e * (2 * I / kGroup) * nbh;
  const float* Sg = S + (size_t)(n0 / kGroup) * nbh;
  const float* Su = S + (size_t)((I + n0) / kGroup) * nbh;
  const uint8_t* rg0 = W + (size_t)(n0 + g) * H;
  const uint8_t* ru0 = W + (size_t)(I + n0 + g) * H;
  const uint8_t* rg1 = W + (size_t)(n0 + 8 + g) * H;
  const uint8_t* ru1 = W + (size_t)(I + n0 + 8 + g) * H;

  const uint8_t* xb[2];
  bool bval[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    int tb = 8 * nt + g;
    bval[nt] = tb < ntok;
    int t = bval[nt] ? a.w.pair_of_slot[s0 + tb] / k : 0;
    xb[nt] = a.w.xq + (size_t)t * H;
  }
  // the unit's scales into shared memory once (coalesced), instead of
  // scattered loads inside the K loop; hidden sizes beyond kMaxNbh groups
  // keep the direct loads
  const bool staged = nbh <= kMaxNbh;
  const float* sxc[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int tc = 8 * nt + 2 * q + c;
      sxc[nt][c] = !staged && tc < ntok
                       ? a.w.sx + (size_t)(a.w.pair_of_slot[s0 + tc] / k) * nbh
                       : nullptr;
    }
  if (staged) {
    for (int i = threadIdx.x; i < ntok * nbh; i += blockDim.x) {
      const int tok = i / nbh, kbb = i - tok * nbh;
      sm.sxs[tok][kbb] = __ldcg(a.w.sx + (size_t)(a.w.pair_of_slot[s0 + tok] / k) * nbh + kbb);
    }
    for (int i = threadIdx.x; i < nbh; i += blockDim.x) {
      sm.swg[i] = __ldg(Sg + i);
      sm.swu[i] = __ldg(Su + i);
    }
  }
  __syncthreads();
  const int n_nt = ntok > 8 ? 2 : 1;

  float acc[2][2][4] = {};
  const int nblk = H / 64;
  // unrolled so the loads of several K slices are in flight together
#pragma unroll 4
  for (int b = warp; b < nblk; b += kWarps) {
    const int kb = (b * 64) / kGroup;
    const int off = b * 64 + 16 * q;
    const uint4 ag0 = ld_stream16(rg0 + off), au0 = ld_stream16(ru0 + off);
    const uint4 ag1 = ld_stream16(rg1 + off), au1 = ld_stream16(ru1 + off);
    const float sg = staged ? sm.swg[kb] : __ldg(Sg + kb);
    const float su = staged ? sm.swu[kb] : __ldg(Su + kb);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (nt >= n_nt) break;
      const uint4 bx = bval[nt] ? ld_cg16(xb[nt] + off) : make_uint4(0u, 0u, 0u, 0u);
      const int tc0 = 8 * nt + 2 * q;
      float sa, sb;
      if (staged) {
        sa = tc0 < ntok ? sm.sxs[tc0][kb] : 0.0f;
        sb = tc0 + 1 < ntok ? sm.sxs[tc0 + 1][kb] : 0.0f;
      } else {
        sa = sxc[nt][0] ? __ldcg(sxc[nt][0] + kb) : 0.0f;
        sb = sxc[nt][1] ? __ldcg(sxc[nt][1] + kb) : 0.0f;
      }
      float p0[4] = {}, p1[4] = {};
      mma_e4m3_k64(p0, ag0, au0, bx);
      mma_e4m3_k64(p1, ag1, au1, bx);
      acc[0][nt][0] = fmaf(p0[0], sg * sa, acc[0][nt][0]);
      acc[0][nt][1] = fmaf(p0[1], sg * sb, acc[0][nt][1]);
      acc[0][nt][2] = fmaf(p0[2], su * sa, acc[0][nt][2]);
      acc[0][nt][3] = fmaf(p0[3], su * sb, acc[0][nt][3]);
      acc[1][nt][0] = fmaf(p1[0], sg * sa, acc[1][nt][0]);
      acc[1][nt][1] = fmaf(p1[1], sg * sb, acc[1][nt][1]);
      acc[1][nt][2] = fmaf(p1[2], su * sa, acc[1][nt][2]);
      acc[1][nt][3] = fmaf(p1[3], su * sb, acc[1][nt][3]);
    }
  }
#pragma unroll
  for (int tile = 0; tile < 2; ++tile)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) red_at(sm, warp, tile, nt, c, lane) = acc[tile][nt][c];
  __syncthreads();
  if (warp < 4) {
    const int tile = warp >> 1, nt = warp & 1;
    if (nt < n_nt) {
      float z[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v = 0.0f;
        for (int w = 0; w < kWarps; ++w) v += red_at(sm, w, tile, nt, c, lane);
        z[c] = v;
      }
      const int n = n0 + 8 * tile + g;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int tok = 8 * nt + 2 * q + c;
        if (tok < ntok) {
          const float zg = bf16_round(z[c]), zu = bf16_round(z[2 + c]);
          a.w.hbuf[(size_t)(s0 + tok) * I + n] = silu_f32(zg) * zu;
        }
      }
    }
  }
  __threadfence();
  __syncthreads();
  const int grp = n0 / kGroup;
  if (threadIdx.x == 0) {
    int* cnt = &a.w.gcount[(size_t)chunk_id * (I / kGroup) + grp];
    const int old = atomicAdd(cnt, 1);
    const int last = old == kGroup / 16 - 1;
    if (last) *cnt = 0;
    sm.flag = last;
  }
  __syncthreads();
  if (sm.flag) {
    __threadfence();
    const int nbi = I / kGroup;
    for (int tok = warp; tok < ntok; tok += kWarps) {
      const int slot = s0 + tok;
      const float4 v = __ldcg(reinterpret_cast<const float4*>(a.w.hbuf + (size_t)slot * I +
                                                              grp * kGroup + 4 * lane));
      float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
      m = warp_max(m);
      const float s = group_scale(m);
      const uint32_t packed = quant4(v.x, v.y, v.z, v.w, s);
      *reinterpret_cast<uint32_t*>(a.w.hq + (size_t)slot * I + grp * kGroup + 4 * lane) = packed;
      if (lane == 0) a.w.sh[(size_t)slot * nbi + grp] = s;
    }
  }
  __syncthreads();
}

// ---- shared gate/up (bf16) ---------------------------------------------------
__device__ void gateup_shared(const KArgs& a, Smem& sm, int tchunk, int ms) {
  const int H = a.d.H, Is = a.d.Is, T = a.d.T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, q = lane & 3;
  const int t0 = tchunk * kChunk;
  const int ntok = min(kChunk, T - t0);
  const bf16* rg = a.L.ws13 + (size_t)(8 * ms + g) * H;
  const bf16* ru = a.L.ws13 + (size_t)(Is + 8 * ms + g) * H;
  const bf16* xb[2];
  bool bval[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    bval[nt] = 8 * nt + g < ntok;
    xb[nt] = a.x + (size_t)(bval[nt] ? t0 + 8 * nt + g : 0) * H;
  }
  const int n_nt = ntok > 8 ? 2 : 1;
  float acc[2][4] = {};
  const int nblk = H / 32;
  for (int b = warp; b < nblk; b += kWarps) {
    const int off = b * 32 + 8 * q;
    const uint4 ag = ld_stream16(rg + off), au = ld_stream16(ru + off);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (nt >= n_nt) break;
      const uint4 bx = bval[nt] ? ld_cg16(xb[nt] + off) : make_uint4(0u, 0u, 0u, 0u);
      mma_bf16_k32(acc[nt], ag, au, bx);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) red_at(sm, warp, 0, nt, c, lane) = acc[nt][c];
  __syncthreads();
  if (warp < 2 && warp < n_nt) {
    const int nt = warp;
    float z[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v = 0.0f;
      for (int w = 0; w < kWarps; ++w) v += red_at(sm, w, 0, nt, c, lane);
      z[c] = v;
    }
    const int n = 8 * ms + g;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int tok = 8 * nt + 2 * q + c;
      if (tok < ntok) {
        const float zg = bf16_round(z[c]), zu = bf16_round(z[2 + c]);
        a.w.hs[(size_t)(t0 + tok) * Is + n] = __float2bfloat16_rn(silu_f32(zg) * zu);
      }
    }
  }
  __syncthreads();
}

}  // namespace

namespace {

// L2 prefetch of the weight rows one gate/up unit reads (two contiguous runs).
__device__ void prefetch_gateup_unit(const KArgs& a, int u, int n_routed, int total) {
  if (u >= total) return;
  const int H = a.d.H, I = a.d.I, Is = a.d.Is;
  if (u < n_routed) {
    const int mpp = I / 16;
    const int e = a.w.chunks[u / mpp].x, n0 = 16 * (u % mpp);
    const uint8_t* W = a.L.w13 + (size_t)e * 2 * I * H;
    prefetch_l2(W + (size_t)n0 * H, 16u * H);
    prefetch_l2(W + (size_t)(I + n0) * H, 16u * H);
  } else {
    const int ms = (u - n_routed) % (Is / 8);
    prefetch_l2(a.L.ws13 + (size_t)(8 * ms) * H, 8u * H * 2);
    prefetch_l2(a.L.ws13 + (size_t)(Is + 8 * ms) * H, 8u * H * 2);
  }
}

}  // namespace

// Down-projection weights of the selected experts are prefetched into L2 by
// the decode gate/up kernel when they fit this budget (for the next kernel).
constexpr size_t kDownPrefetchBudget = 48u << 20;

template <bool kDecode>
__global__ void __launch_bounds__(256) k_gateup(KArgs a) {
  __shared__ Smem sm;
  if (kDecode) {
    pdl_wait();
    pdl_trigger();
  }
  const int n_routed = *a.w.n_chunks * (a.d.I / 16);
  const int n_tchunks = (a.d.T + kChunk - 1) / kChunk;
  const int ms_per = a.d.Is / 8;
  const int total = n_routed + n_tchunks * ms_per;
  if (kDecode && threadIdx.x == 0) {
    prefetch_gateup_unit(a, blockIdx.x, n_routed, total);
    prefetch_gateup_unit(a, blockIdx.x + gridDim.x, n_routed, total);
    const int U = *a.w.n_chunks;
    const size_t per = (size_t)a.d.H * a.d.I;
    if ((size_t)U * per <= kDownPrefetchBudget)
      for (int c = 0; c < U; ++c)
        prefetch_l2_share(a.L.w2 + (size_t)a.w.chunks[c].x * per, per, blockIdx.x, gridDim.x);
  }
  for (int u = blockIdx.x; u < total; u += gridDim.x) {
    if (kDecode && threadIdx.x == 0) prefetch_gateup_unit(a, u + 2 * gridDim.x, n_routed, total);
    if (u < n_routed) {
      gateup_routed(a, sm, u / (a.d.I / 16), u % (a.d.I / 16));
    } else {
      const int v = u - n_routed;
      gateup_shared(a, sm, v / ms_per, v % ms_per);
    }
  }
}

cudaError_t launch_gateup(const KArgs& a, int grid, cudaStream_t s) {
  k_gateup<false><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gateup_decode(const KArgs& a, int grid, bool pdl, cudaStream_t s) {
  return launch_pdl(k_gateup<true>, dim3(grid), dim3(256), 0, s, pdl, a);
}

// ---- down projections ------------------------------------------------------
namespace {

__device__ void down_routed(const KArgs& a, Smem& sm, int chunk_id, int mt) {
  const int H = a.d.H, I = a.d.I;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, q = lane & 3;
  const int4 ch = a.w.chunks[chunk_id];
  const int e = ch.x, s0 = ch.y, ntok = ch.z;
  const int m0 = 16 * mt;
  const int nbi = I / kGroup;
  const uint8_t* W = a.L.w2 + (size_t)e * H * I;
  const float* S = a.L.s2 + (size_t)e * (H / kGroup) * nbi + (size_t)(m0 / kGroup) * nbi;
  const uint8_t* r0 = W + (size_t)(m0 + g) * I;
  const uint8_t* r1 = W + (size_t)(m0 + 8 + g) * I;
  const uint8_t* hb[2];
  bool bval[2];
  const float* shc[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int tb = 8 * nt + g;
    bval[nt] = tb < ntok;
    hb[nt] = a.w.hq + (size_t)(s0 + (bval[nt] ? tb : 0)) * I;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int tc = 8 * nt + 2 * q + c;
      shc[nt][c] = tc < ntok ? a.w.sh + (size_t)(s0 + tc) * nbi : nullptr;
    }
  }
  const int n_nt = ntok > 8 ? 2 : 1;
  float acc[2][4] = {};
  const int nblk = I / 64;
  for (int b = warp; b < nblk; b += kWarps) {
    const int kb = (b * 64) / kGroup;
    const int off = b * 64 + 16 * q;
    const uint4 a0 = ld_stream16(r0 + off), a1 = ld_stream16(r1 + off);
    const float sw = __ldg(S + kb);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (nt >= n_nt) break;
      const uint4 bx = bval[nt] ? ld_cg16(hb[nt] + off) : make_uint4(0u, 0u, 0u, 0u);
      const float sa = shc[nt][0] ? __ldcg(shc[nt][0] + kb) : 0.0f;
      const float sb = shc[nt][1] ? __ldcg(shc[nt][1] + kb) : 0.0f;
      float p[4] = {};
      mma_e4m3_k64(p, a0, a1, bx);
      acc[nt][0] = fmaf(p[0], sw * sa, acc[nt][0]);
      acc[nt][1] = fmaf(p[1], sw * sb, acc[nt][1]);
      acc[nt][2] = fmaf(p[2], sw * sa, acc[nt][2]);
      acc[nt][3] = fmaf(p[3], sw * sb, acc[nt][3]);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) red_at(sm, warp, 0, nt, c, lane) = acc[nt][c];
  __syncthreads();
  if (warp < 2 && warp < n_nt) {
    const int nt = warp;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v = 0.0f;
      for (int w = 0; w < kWarps; ++w) v += red_at(sm, w, 0, nt, c, lane);
      const int tok = 8 * nt + 2 * q + (c & 1);
      const int m = m0 + g + (c >> 1) * 8;
      if (tok < ntok) a.w.dbuf[(size_t)(s0 + tok) * H + m] = __float2bfloat16_rn(v);
    }
  }
  __syncthreads();
}

__device__ void down_shared(const KArgs& a, Smem& sm, int tchunk, int mt) {
  const int H = a.d.H, Is = a.d.Is, T = a.d.T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, q = lane & 3;
  const int t0 = tchunk * kChunk;
  const int ntok = min(kChunk, T - t0);
  const int m0 = 16 * mt;
  const bf16* r0 = a.L.ws2 + (size_t)(m0 + g) * Is;
  const bf16* r1 = a.L.ws2 + (size_t)(m0 + 8 + g) * Is;
  const bf16* hb[2];
  bool bval[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    bval[nt] = 8 * nt + g < ntok;
    hb[nt] = a.w.hs + (size_t)(bval[nt] ? t0 + 8 * nt + g : 0) * Is;
  }
  const int n_nt = ntok > 8 ? 2 : 1;
  float acc[2][4] = {};
  const int nblk = Is / 32;
  for (int b = warp; b < nblk; b += kWarps) {
    const int off = b * 32 + 8 * q;
    const uint4 a0 = ld_stream16(r0 + off), a1 = ld_stream16(r1 + off);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (nt >= n_nt) break;
      const uint4 bx = bval[nt] ? ld_cg16(hb[nt] + off) : make_uint4(0u, 0u, 0u, 0u);
      mma_bf16_k32(acc[nt], a0, a1, bx);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) red_at(sm, warp, 0, nt, c, lane) = acc[nt][c];
  __syncthreads();
  if (warp < 2 && warp < n_nt) {
    const int nt = warp;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float v = 0.0f;
      for (int w = 0; w < kWarps; ++w) v += red_at(sm, w, 0, nt, c, lane);
      const int tok = 8 * nt + 2 * q + (c & 1);
      const int m = m0 + g + (c >> 1) * 8;
      if (tok < ntok) a.w.ds[(size_t)(t0 + tok) * H + m] = __float2bfloat16_rn(v);
    }
  }
  __syncthreads();
}

}  // namespace

__global__ void __launch_bounds__(256) k_down(KArgs a) {
  __shared__ Smem sm;
  const int mt_per = a.d.H / 16;
  const int n_routed = *a.w.n_chunks * mt_per;
  const int n_tchunks = (a.d.T + kChunk - 1) / kChunk;
  const int total = n_routed + n_tchunks * mt_per;
  for (int u = blockIdx.x; u < total; u += gridDim.x) {
    if (u < n_routed) {
      down_routed(a, sm, u / mt_per, u % mt_per);
    } else {
      const int v = u - n_routed;
      down_shared(a, sm, v / mt_per, v % mt_per);
    }
  }
}

cudaError_t launch_down(const KArgs& a, int grid, cudaStream_t s) {
  k_down<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ---- combine ---------------------------------------------------------------
// y[t, m..m+7] = bf16( sum_j w[t,j] d[slot(t,j), m..m+7] + gamma[t] ds[t, m..m+7] ),
// routed terms in rank order, the shared term last.
__global__ void __launch_bounds__(256) k_combine(KArgs a) {
  const int H = a.d.H, k = a.d.k;
  const int per_row = H / 8;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.d.T * per_row) return;
  const int t = i / per_row, m = (i % per_row) * 8;
  pdl_wait();
  pdl_trigger();
  float acc[8] = {};
  for (int j = 0; j < k; ++j) {
    const int slot = __ldcg(a.w.slot_of_pair + t * k + j);
    const float w = __ldcg(a.w.wts + t * k + j);
    const uint4 raw = ld_cg16(a.w.dbuf + (size_t)slot * H + m);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      acc[2 * h] = fmaf(w, __low2float(p[h]), acc[2 * h]);
      acc[2 * h + 1] = fmaf(w, __high2float(p[h]), acc[2 * h + 1]);
    }
  }
  const float gm = __ldcg(a.w.gamma + t);
  const uint4 raw = ld_cg16(a.w.ds + (size_t)t * H + m);
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
  uint4 out;
  __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float y0 = fmaf(gm, __low2float(p[h]), acc[2 * h]);
    const float y1 = fmaf(gm, __high2float(p[h]), acc[2 * h + 1]);
    o[h] = __floats2bfloat162_rn(y0, y1);
  }
  *reinterpret_cast<uint4*>(a.y + (size_t)t * H + m) = out;
}

cudaError_t launch_combine(const KArgs& a, cudaStream_t s, bool pdl) {
  const int n = a.d.T * (a.d.H / 8);
  return launch_pdl(k_combine, dim3((n + 255) / 256), dim3(256), 0, s, pdl, a);
}

// ---- re-quantised SwiGLU rows by (row, rank), for checking -----------------
__global__ void k_gather_hq(KArgs a, uint8_t* hq, float* sh) {
  const int p = blockIdx.x;  // pair t*k + j
  const int slot = a.w.slot_of_pair[p];
  const int I = a.d.I, nbi = I / kGroup;
  for (int i = threadIdx.x; i < I; i += blockDim.x) hq[(size_t)p * I + i] = a.w.hq[(size_t)slot * I + i];
  for (int i = threadIdx.x; i < nbi; i += blockDim.x) sh[(size_t)p * nbi + i] = a.w.sh[(size_t)slot * nbi + i];
}

cudaError_t launch_gather_hq(const KArgs& a, uint8_t* hq, float* sh, cudaStream_t s) {
  if (a.d.T * a.d.k == 0) return cudaSuccess;
  k_gather_hq<<<a.d.T * a.d.k, 128, 0, s>>>(a, hq, sh);
  return cudaGetLastError();
}

// The e4m3 codes and group scales of x that each (row, rank) pair's expert
// read in the most recent forward: from the row-major workspace copy (decode
// kernels, warp-MMA prompt kernels) or from the pair's slot of the
// slot-ordered operand of the tcgen05 gate/up GEMM.
__global__ void k_gather_codes(KArgs a, const uint8_t* xg, const float* sxg, int slot_order,
                               uint8_t* codes, float* scales) {
  const int p = blockIdx.x;  // pair t*k + j
  const int t = p / a.d.k;
  const int H = a.d.H, nbh = H / kGroup;
  const uint8_t* src = a.w.xq + (size_t)t * H;
  const float* ssrc = a.w.sx + (size_t)t * nbh;
  if (slot_order) {
    const int slot = a.w.slot_of_pair[p];
    src = xg + (size_t)slot * H;
    ssrc = sxg + (size_t)slot * nbh;
  }
  for (int i = threadIdx.x; i < H; i += blockDim.x) codes[(size_t)p * H + i] = src[i];
  for (int i = threadIdx.x; i < nbh; i += blockDim.x) scales[(size_t)p * nbh + i] = ssrc[i];
}

cudaError_t launch_gather_codes(const KArgs& a, const uint8_t* xg, const float* sxg,
                                bool slot_order, uint8_t* codes, float* scales, cudaStream_t s) {
  if (a.d.T * a.d.k == 0) return cudaSuccess;
  k_gather_codes<<<a.d.T * a.d.k, 256, 0, s>>>(a, xg, sxg, slot_order ? 1 : 0, codes, scales);
  return cudaGetLastError();
}

}  // namespace moe

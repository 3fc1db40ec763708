// Decode path (rows <= 16): router + top-k + schedule in one launch, and the
// down projections fused with the combine.  With the gate/up kernel between
// them the layer is three launches chained by programmatic dependent launch.
//
// Chaining and prefetch follow PR #927 "backbone chain launches with PDL"
// (section "What this changes": kernels wait before touching their
// predecessor's data; immutable weights may be fetched before the wait).  The
// one-row layer is bound by reading weights, so every kernel starts the
// weight traffic it can before it waits: the router kernel fetches its router
// rows and asks L2 for the shared expert, the gate/up kernel asks L2 for the
// selected experts' down weights, and the layer's HBM reads overlap the
// launch and dependency latencies.
//
// Router and top-k: PR #939 "Fish Audio Drama 3 text to speech on one CUDA
// GPU", sections "What it adds" (the router in drama3.cu) and "Fidelity
// against the PyTorch oracle" (near-tied 8th/9th experts: ties go to the
// lower index).  Combine: commit "MoE combine on 8-wide vectors" (every sum
// keeps its order: routed terms in rank order, then the shared term).
#include <math.h>

#include "moe_rowops.cuh"

namespace moe {

namespace {

// Block-wide exclusive prefix sum over the CTA's threads (one value each,
// up to 32 warps).
__device__ int block_exscan(int v, int* total, int* scratch /*[32]*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  int base = 0, all = 0;
  for (int w = 0; w < nw; ++w) {
    if (w < warp) base += scratch[w];
    all += scratch[w];
  }
  __syncthreads();
  *total = all;
  return base + inc - v;
}

// The schedule in the layout the expert kernels read (slots sorted by
// (expert, row); one chunk per selected expert, since an expert holds at
// most 16 rows here), from every row's top-k in a.w.idx.
__device__ void decode_schedule(const KArgs& a) {
  __shared__ int s_idx[kDecodeRows * kMaxTopK];
  __shared__ uint32_t s_tok[kMaxExperts];
  __shared__ int s_scan[32];
  const int T = a.d.T, k = a.d.k, E = a.d.E;
  for (int e = threadIdx.x; e < kMaxExperts; e += blockDim.x) s_tok[e] = 0u;
  __threadfence_block();
  __syncthreads();
  // an index outside [0, E) (possible only after a wait gave up and the
  // status flag is set) joins no expert's rows
  for (int p = threadIdx.x; p < T * k; p += blockDim.x) {
    const int e = a.w.idx[p];
    s_idx[p] = e;
    if (e >= 0 && e < E) atomicOr(&s_tok[e], 1u << (p / k));
  }
  __syncthreads();
  const int e = threadIdx.x;
  const uint32_t mask = e < E ? s_tok[e] : 0u;
  const int cnt = __popc(mask);
  int n_slots, n_used;
  const int slot0 = block_exscan(cnt, &n_slots, s_scan);
  const int u = block_exscan(cnt > 0 ? 1 : 0, &n_used, s_scan);
  if (cnt > 0) {
    a.w.chunks[u] = make_int4(e, slot0, cnt, 0);
    uint32_t m = mask;
    for (int r = 0; m; ++r) {
      const int t = __ffs(m) - 1;
      m &= m - 1;
      int j = 0;
      while (j < k - 1 && s_idx[t * k + j] != e) ++j;
      const int p = t * k + j, slot = slot0 + r;
      a.w.pair_of_slot[slot] = p;
      a.w.slot_of_pair[p] = slot;
    }
  }
  if (e < E) a.w.counts[e] = cnt;
  if (threadIdx.x == 0) *a.w.n_chunks = n_used;
}

}  // namespace

constexpr long long kRouteSpin = 1ll << 22;  // tries before the logit wait gives up

// ---- D1: router logits, x quantisation, top-k, schedule ---------------------
// CTAs [0, n_router): two experts each; warp w covers expert 2b + w/4 over the
// K quarter w%4; each counts itself done (done[0]) once its logits are out.
// CTAs [n_router, n_router + T): row t's quantisation and shared gate, then,
// once every router CTA is done (a bounded wait: all CTAs of this grid are
// resident together), row t's top-k with the whole CTA; the last of them
// (done[1]) builds the schedule and resets both counters.
constexpr int kRtWarps = 16;  // warps per router CTA: K in eighths of two experts

__global__ void __launch_bounds__(32 * kRtWarps) k_route_decode(KArgs a) {
  __shared__ float red[kRtWarps][kDecodeRows];
  __shared__ int s_last;
  // the top-k reads these as 16-byte vectors
  __shared__ __align__(16) float s_lg[kMaxExperts];
  __shared__ __align__(16) uint32_t s_ck[2 * kRtWarps * kMaxTopK];
  __shared__ __align__(16) uint32_t s_cid[2 * kRtWarps * kMaxTopK];
  __shared__ int s_idx1[kMaxTopK];
  __shared__ float s_w1[kMaxTopK];
  const int T = a.d.T, H = a.d.H, E = a.d.E, k = a.d.k;
  const int n_router = (E + 1) / 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // immutable weights first: ask L2 for this CTA's share of the shared expert
  if (threadIdx.x == 0) {
    const size_t b13 = (size_t)2 * a.d.Is * H * 2, b2 = (size_t)H * a.d.Is * 2;
    prefetch_l2_share(a.L.ws13, b13, blockIdx.x, gridDim.x);
    prefetch_l2_share(a.L.ws2, b2, blockIdx.x, gridDim.x);
  }
  if (blockIdx.x >= n_router) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x - n_router;
    quant_row_and_gate(a, t);
    if (threadIdx.x == 0) {
      long long it = 0;
      for (;;) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(a.w.done) : "memory");
        if (v >= n_router) break;
        if (++it > kRouteSpin) {
          atomicExch(a.w.status, 1);
          break;
        }
        __nanosleep(32);
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
      s_lg[e] = route_logit(__ldcg(a.w.logits + (size_t)t * E + e), a.d.rbf16);
    __syncthreads();
    // the top-k on the first 8 warps (named barrier), the rest wait below
    if (k <= 8 && E <= 256) {
      if (warp < 8) topk_one_row_fast<8>(s_lg, E, k, s_ck, s_cid, s_idx1, s_w1);
    } else {
      topk_one_row<kRtWarps>(s_lg, E, k, s_ck, s_cid, s_idx1, s_w1);
    }
    __syncthreads();
    if (threadIdx.x < k) {
      a.w.idx[(size_t)t * k + threadIdx.x] = s_idx1[threadIdx.x];
      a.w.wts[(size_t)t * k + threadIdx.x] = s_w1[threadIdx.x];
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&a.w.done[1], 1) == T - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    decode_schedule(a);
    __syncthreads();
    if (threadIdx.x == 0) {
      a.w.done[0] = 0;
      a.w.done[1] = 0;
    }
    return;
  }

  constexpr int kParts = kRtWarps / 2;  // K parts per expert
  const int e = 2 * blockIdx.x + warp / kParts;
  const int quarter = H / kParts;
  const int k0 = (warp % kParts) * quarter;
  const bool valid = e < E;
  const float* wrow = a.L.wr + (size_t)(valid ? e : 0) * H + k0;
  // router rows do not depend on the previous kernel: load before waiting
  constexpr int kMaxV = 8;  // float4 per lane, up to H = 4096
  const int nv = (quarter + 127) / 128;
  float4 wv[kMaxV];
#pragma unroll
  for (int i = 0; i < kMaxV; ++i) {
    wv[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (i < nv && 128 * i + 4 * lane < quarter)
      wv[i] = __ldg(reinterpret_cast<const float4*>(wrow + 128 * i + 4 * lane));
  }
  pdl_wait();
  pdl_trigger();

  float acc[kDecodeRows];
#pragma unroll
  for (int t = 0; t < kDecodeRows; ++t) acc[t] = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxV; ++i) {
    if (i >= nv) break;
    if (128 * i + 4 * lane >= quarter) continue;
    const int kk = k0 + 128 * i + 4 * lane;
    // every row's x for this slice in flight at once (one round trip per
    // slice instead of one per row)
    uint2 raw[kDecodeRows];
#pragma unroll
    for (int t = 0; t < kDecodeRows; ++t)
      raw[t] = t < T ? __ldcg(reinterpret_cast<const uint2*>(a.x + (size_t)t * H + kk))
                     : make_uint2(0u, 0u);
#pragma unroll
    for (int t = 0; t < kDecodeRows; ++t) {
      const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw[t].x);
      const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw[t].y);
      float s = acc[t];
      s = fmaf(__low2float(p0), wv[i].x, s);
      s = fmaf(__high2float(p0), wv[i].y, s);
      s = fmaf(__low2float(p1), wv[i].z, s);
      s = fmaf(__high2float(p1), wv[i].w, s);
      acc[t] = s;
    }
  }
#pragma unroll
  for (int t = 0; t < kDecodeRows; ++t) {
    if (t >= T) break;
    const float v = warp_sum(acc[t]);
    if (lane == 0) red[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < 2 * T) {
    const int h = threadIdx.x / T, t = threadIdx.x % T;
    const int ee = 2 * blockIdx.x + h;
    if (ee < E) {
      float v = 0.0f;
      for (int pp = 0; pp < kParts; ++pp) v += red[kParts * h + pp][t];  // K parts in order
      a.w.logits[(size_t)t * E + ee] = v;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd(&a.w.done[0], 1);
}

cudaError_t launch_route_decode(const KArgs& a, bool pdl, cudaStream_t s) {
  const int grid = (a.d.E + 1) / 2 + a.d.T;
  return launch_pdl(k_route_decode, dim3(grid), dim3(32 * kRtWarps), 0, s, pdl, a);
}

// ---- D3: down projections + combine -----------------------------------------
// One CTA per 16 output rows.  Work items: every selected expert (its rows'
// 16 x I slice of the down weights against those rows' re-quantised SwiGLU
// codes) and the shared expert's slice in two K halves.  Items go to warps
// round-robin, each covering its full K, so no cross-warp reduction is needed.
// 16 warps: every item is a chain of dependent loads, so the more items run
// side by side in a CTA the more of that latency is hidden.
constexpr int kDcWarps = 16;

__global__ void __launch_bounds__(32 * kDcWarps) k_down_combine_decode(KArgs a) {
  __shared__ float s_d[kDecodeRows * kMaxTopK][16];
  __shared__ float s_ds[2][kDecodeRows][16];
  const int T = a.d.T, H = a.d.H, I = a.d.I, Is = a.d.Is, k = a.d.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, q = lane & 3;
  const int m0 = 16 * blockIdx.x;
  const int nbi = I / kGroup;
  pdl_wait();
  pdl_trigger();
  const int U = *a.w.n_chunks;
  for (int it = warp; it < U + 2; it += kDcWarps) {
    if (it < U) {
      const int4 ch = a.w.chunks[it];
      const int e = ch.x, s0 = ch.y, ntok = ch.z;
      const uint8_t* W = a.L.w2 + (size_t)e * H * I;
      const float* S = a.L.s2 + ((size_t)e * (H / kGroup) + m0 / kGroup) * nbi;
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
      // unrolled so the loads of several K slices are in flight together
#pragma unroll 8
      for (int b = 0; b < I / 64; ++b) {
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
        for (int c = 0; c < 4; ++c) {
          const int tok = 8 * nt + 2 * q + (c & 1);
          if (nt < n_nt && tok < ntok) s_d[s0 + tok][g + 8 * (c >> 1)] = bf16_round(acc[nt][c]);
        }
    } else {
      const int half = it - U;
      const int kh = Is / 2;
      const bf16* r0 = a.L.ws2 + (size_t)(m0 + g) * Is + half * kh;
      const bf16* r1 = a.L.ws2 + (size_t)(m0 + 8 + g) * Is + half * kh;
      const bf16* hb[2];
      bool bval[2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        bval[nt] = 8 * nt + g < T;
        hb[nt] = a.w.hs + (size_t)(bval[nt] ? 8 * nt + g : 0) * Is + half * kh;
      }
      const int n_nt = T > 8 ? 2 : 1;
      float acc[2][4] = {};
#pragma unroll 8
      for (int b = 0; b < kh / 32; ++b) {
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
        for (int c = 0; c < 4; ++c) {
          const int tok = 8 * nt + 2 * q + (c & 1);
          if (nt < n_nt && tok < T) s_ds[half][tok][g + 8 * (c >> 1)] = acc[nt][c];
        }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * 16; i += blockDim.x) {
    const int t = i >> 4, r = i & 15;
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int slot = __ldcg(a.w.slot_of_pair + t * k + j);
      acc = fmaf(__ldcg(a.w.wts + t * k + j), s_d[slot][r], acc);
    }
    const float ds = bf16_round(s_ds[0][t][r] + s_ds[1][t][r]);
    a.y[(size_t)t * H + m0 + r] = __float2bfloat16_rn(fmaf(__ldcg(a.w.gamma + t), ds, acc));
  }
}

cudaError_t launch_down_combine_decode(const KArgs& a, bool pdl, cudaStream_t s) {
  return launch_pdl(k_down_combine_decode, dim3(a.d.H / 16), dim3(32 * kDcWarps), 0, s, pdl, a);
}

}  // namespace moe

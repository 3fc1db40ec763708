// Router logits, activation quantisation + shared gate, top-k, and the
// token-to-expert schedule.
//
// Router and top-k: PR #939 "Fish Audio Drama 3 text to speech on one CUDA
// GPU", section "What it adds" (drama3.cu holds the router) and section
// "Fidelity against the PyTorch oracle" (8th/9th experts 6e-5 apart or tied).
// Activation quantisation: PR #939 section "Precision" (e4m3 per row and per
// 128 inputs, amax / 448) and the "Drama 3 text backbone" commit of PR #925
// (dynamic 1 x 128 FP8 activation quantization).
#include <math.h>

#include "moe_rowops.cuh"

namespace moe {

// ---- router logits: [T][E] = x[T][H] . Wr[E][H]^T, fp32 -------------------
// 32 rows x 64 experts per CTA, K in slices of 32 through shared memory.
__global__ void __launch_bounds__(256) k_router(KArgs a) {
  __shared__ float xs[32][33];
  __shared__ float ws[64][33];
  const int T = a.d.T, H = a.d.H, E = a.d.E;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int e0 = blockIdx.x * 64, t0 = blockIdx.y * 32;
  float acc[2][4] = {};
  for (int k0 = 0; k0 < H; k0 += 32) {
    for (int i = tid; i < 32 * 32; i += 256) {
      int r = i >> 5, c = i & 31, t = t0 + r;
      xs[r][c] = t < T ? __bfloat162float(a.x[(size_t)t * H + k0 + c]) : 0.0f;
    }
    for (int i = tid; i < 64 * 32; i += 256) {
      int r = i >> 5, c = i & 31, e = e0 + r;
      ws[r][c] = e < E ? __ldg(a.L.wr + (size_t)e * H + k0 + c) : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float x0 = xs[2 * ty][kk], x1 = xs[2 * ty + 1][kk];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float w = ws[tx + 16 * j][kk];
        acc[0][j] = fmaf(x0, w, acc[0][j]);
        acc[1][j] = fmaf(x1, w, acc[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    int t = t0 + 2 * ty + r;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = e0 + tx + 16 * j;
      if (e < E) a.w.logits[(size_t)t * E + e] = acc[r][j];
    }
  }
}

cudaError_t launch_router(const KArgs& a, cudaStream_t s) {
  dim3 grid((a.d.E + 63) / 64, (a.d.T + 31) / 32);
  k_router<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ---- activation quantisation (1 x 128 groups) and the shared gate ----------
__global__ void __launch_bounds__(256) k_quant_gamma(KArgs a) { quant_row_and_gate(a, blockIdx.x); }

cudaError_t launch_quant_gamma(const KArgs& a, cudaStream_t s) {
  k_quant_gamma<<<a.d.T, 256, 0, s>>>(a);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256) k_topk(KArgs a) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= a.d.T) return;
  topk_row(a.w.logits + (size_t)t * a.d.E, a.d.E, a.d.k, a.w.idx + (size_t)t * a.d.k,
           a.w.wts + (size_t)t * a.d.k);
}

cudaError_t launch_topk(const KArgs& a, cudaStream_t s) {
  k_topk<<<(a.d.T + 7) / 8, 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ---- schedule: stable slots sorted by (expert, row), and expert chunks ----
// A pair p = t*k + j routes row t to expert e = idx[p].  Rows pick distinct
// experts, so an expert's slots in row order are its rank among the rows
// that chose it: bit t of bitmap[e] marks row t, and a running popcount over
// the bitmap words gives every rank.  One CTA; no ordering depends on timing.
__global__ void __launch_bounds__(1024) k_schedule(KArgs a) {
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_ch[kMaxExperts + 1];
  const int T = a.d.T, k = a.d.k, E = a.d.E, W = (T + 31) / 32;
  const int tid = threadIdx.x;
  uint32_t* bm = a.w.bitmap;
  for (int i = tid; i < E * W; i += blockDim.x) bm[i] = 0u;
  __syncthreads();
  for (int p = tid; p < T * k; p += blockDim.x) {
    int t = p / k, e = a.w.idx[p];
    atomicOr(&bm[(size_t)e * W + (t >> 5)], 1u << (t & 31));
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < W; ++w) {
      a.w.wprefix[(size_t)e * W + w] = run;
      run += __popc(__ldcg(&bm[(size_t)e * W + w]));
    }
    s_cnt[e] = run;
  }
  __syncthreads();
  if (tid == 0) {
    int o = 0, c = 0;
    for (int e = 0; e < E; ++e) {
      s_off[e] = o;
      s_ch[e] = c;
      o += s_cnt[e];
      c += (s_cnt[e] + kChunk - 1) / kChunk;
    }
    s_off[E] = o;
    s_ch[E] = c;
    *a.w.n_chunks = c;
  }
  __syncthreads();
  for (int p = tid; p < T * k; p += blockDim.x) {
    int t = p / k, e = a.w.idx[p];
    size_t wi = (size_t)e * W + (t >> 5);
    uint32_t below = __ldcg(&bm[wi]) & ((1u << (t & 31)) - 1u);
    int slot = s_off[e] + a.w.wprefix[wi] + __popc(below);
    a.w.pair_of_slot[slot] = p;
    a.w.slot_of_pair[p] = slot;
  }
  for (int e = tid; e < E; e += blockDim.x) {
    a.w.counts[e] = s_cnt[e];
    a.w.off[e] = s_off[e];
    int n = s_cnt[e];
    for (int c = 0; c * kChunk < n; ++c)
      a.w.chunks[s_ch[e] + c] = make_int4(e, s_off[e] + c * kChunk, min(kChunk, n - c * kChunk), 0);
  }
  if (tid == 0) a.w.off[E] = s_off[E];
}

cudaError_t launch_schedule(const KArgs& a, cudaStream_t s) {
  k_schedule<<<1, 1024, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe

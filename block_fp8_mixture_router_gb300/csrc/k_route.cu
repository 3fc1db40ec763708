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
  pdl_wait();
  pdl_trigger();
  topk_row(a.w.logits + (size_t)t * a.d.E, a.d.E, a.d.k, a.w.idx + (size_t)t * a.d.k,
           a.w.wts + (size_t)t * a.d.k, a.d.rbf16);
}

cudaError_t launch_topk(const KArgs& a, cudaStream_t s, bool pdl) {
  return launch_pdl(k_topk, dim3((a.d.T + 7) / 8), dim3(256), 0, s, pdl, a);
}

// One warp per row: logits[t][e] = sum over splits s = 0..ks-1, in that
// order, of part[s][t][e]; then the top-k of the row.
__global__ void __launch_bounds__(256) k_topk_splits(KArgs a, const float* __restrict__ part,
                                                     int ks) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= a.d.T) return;
  pdl_wait();
  pdl_trigger();
  const int E = a.d.E, lane = threadIdx.x & 31;
  float* row = a.w.logits + (size_t)t * E;
  const size_t stride = (size_t)a.d.T * E;
  const float* pr = part + (size_t)t * E;
  // lane holds experts lane + 32 i; each split's loads are issued together
  float acc[kMaxExperts / 32];
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) {
    const int e = lane + 32 * i;
    acc[i] = e < E ? __ldg(pr + e) : 0.0f;
  }
#pragma unroll 4
  for (int sp = 1; sp < ks; ++sp) {
    float v[kMaxExperts / 32];
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? __ldg(pr + sp * stride + e) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) acc[i] += v[i];
  }
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) {
    const int e = lane + 32 * i;
    if (e < E) row[e] = acc[i];
  }
  __syncwarp();
  topk_row(row, E, a.d.k, a.w.idx + (size_t)t * a.d.k, a.w.wts + (size_t)t * a.d.k, a.d.rbf16);
}

cudaError_t launch_topk_splits(const KArgs& a, const float* part, int ks, cudaStream_t s,
                               bool pdl) {
  return launch_pdl(k_topk_splits, dim3((a.d.T + 7) / 8), dim3(256), 0, s, pdl, a, part, ks);
}

// ---- schedule: stable slots sorted by (expert, row), and expert chunks ----
// A pair p = t*k + j routes row t to expert e = idx[p].  Rows pick distinct
// experts, so an expert's slots in row order are its rank among the rows
// that chose it.  Two kernels, each one CTA per block of kSchedRows rows:
//   count:  a bitmap of the block's rows per expert gives every pair its rank
//           within the block and each expert's count in the block;
//   finish: slot = (rows of all experts before e) + (rows of e in earlier
//           blocks) + (rank in the block).  Block 0 also writes the per-expert
//           counts, offsets and the chunk list of the warp-MMA kernels.
// A single block (up to kSchedRows rows) takes both steps in one kernel.
// Nothing depends on timing: every sum has a fixed order.

__global__ void __launch_bounds__(256) k_sched_count(KArgs a, int* __restrict__ rank,
                                                     int* __restrict__ blk_cnt) {
  __shared__ uint32_t bm[kMaxExperts][kSchedRows / 32];
  const int T = a.d.T, k = a.d.k, E = a.d.E, b = blockIdx.x, tid = threadIdx.x;
  const int t0 = b * kSchedRows, nt = min(kSchedRows, T - t0);
  for (int i = tid; i < E * (kSchedRows / 32); i += 256) (&bm[0][0])[i] = 0u;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int p0 = t0 * k, np = nt * k;
  for (int i = tid; i < np; i += 256) {
    const int tl = i / k, e = __ldg(a.w.idx + p0 + i);
    atomicOr(&bm[e][tl >> 5], 1u << (tl & 31));
  }
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kSchedRows / 32; ++w) c += __popc(bm[e][w]);
    blk_cnt[(size_t)b * E + e] = c;
  }
  for (int i = tid; i < np; i += 256) {
    const int tl = i / k, e = __ldg(a.w.idx + p0 + i);
    int r = __popc(bm[e][tl >> 5] & ((1u << (tl & 31)) - 1u));
    for (int w = 0; w < (tl >> 5); ++w) r += __popc(bm[e][w]);
    rank[p0 + i] = r;
  }
}

// The finishing steps for block b: slots of the block's pairs and, for
// block 0, the per-expert counts, offsets and chunk list.  counts(e, &pre,
// &tot) gives expert e's rows in earlier blocks and in all blocks; rank(p)
// the rank of pair p among its expert's rows in its block.
template <class Counts, class Rank>
__device__ __forceinline__ void sched_finish_block(const KArgs& a, int b, Counts counts,
                                                   Rank rank) {
  __shared__ int s_pre[kMaxExperts];   // rows of e in earlier blocks
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_tot[kMaxExperts];
  __shared__ int s_ch[kMaxExperts + 1];
  __shared__ int s_wsum[2][8];
  const int T = a.d.T, k = a.d.k, E = a.d.E, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  int tot = 0, chs = 0;
  if (tid < E) {
    int pre = 0;
    counts(tid, &pre, &tot);
    s_pre[tid] = pre;
    s_tot[tid] = tot;
    chs = (tot + kChunk - 1) / kChunk;
  }
  // exclusive scans over experts (thread e holds expert e): warps, then warp sums
  int ic = tot, ich = chs;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, ic, o);
    const int vh = __shfl_up_sync(0xffffffffu, ich, o);
    if (lane >= o) {
      ic += v;
      ich += vh;
    }
  }
  if (lane == 31) {
    s_wsum[0][warp] = ic;
    s_wsum[1][warp] = ich;
  }
  __syncthreads();
  int wo = 0, wch = 0;
  for (int w = 0; w < warp; ++w) {
    wo += s_wsum[0][w];
    wch += s_wsum[1][w];
  }
  if (tid < E) {
    s_off[tid] = wo + ic - tot;
    s_ch[tid] = wch + ich - chs;
  }
  if (tid == 0) {
    int o = 0, c = 0;
    for (int w = 0; w < 8; ++w) {
      o += s_wsum[0][w];
      c += s_wsum[1][w];
    }
    s_off[E] = o;
    s_ch[E] = c;
  }
  __syncthreads();
  const int p0 = b * kSchedRows * k, np = min(kSchedRows, T - b * kSchedRows) * k;
  for (int i = tid; i < np; i += 256) {
    const int p = p0 + i, e = a.w.idx[p];
    const int slot = s_off[e] + s_pre[e] + rank(p);
    a.w.pair_of_slot[slot] = p;
    a.w.slot_of_pair[p] = slot;
  }
  if (b == 0) {
    for (int e = tid; e < E; e += 256) {
      a.w.counts[e] = s_tot[e];
      a.w.off[e] = s_off[e];
    }
    if (tid == 0) {
      a.w.off[E] = s_off[E];
      *a.w.n_chunks = s_ch[E];
    }
    // expert chunks of <= kChunk rows (the warp-MMA expert kernels' work list)
    for (int e = warp; e < E; e += 8) {
      const int n = s_tot[e];
      for (int c = lane; c * kChunk < n; c += 32)
        a.w.chunks[s_ch[e] + c] =
            make_int4(e, s_off[e] + c * kChunk, min(kChunk, n - c * kChunk), 0);
    }
  }
}

__global__ void __launch_bounds__(256) k_sched_finish(KArgs a, const int* __restrict__ rank,
                                                      const int* __restrict__ blk_cnt, int nb) {
  const int b = blockIdx.x, E = a.d.E;
  pdl_wait();
  pdl_trigger();
  sched_finish_block(
      a, b,
      [&](int e, int* pre, int* tot) {
        // the blocks' counts 32 at a time: all loads of a batch are in
        // flight before its sums (integer sums: any order gives the same)
        int p = 0, tot_e = 0;
        for (int b0 = 0; b0 < nb; b0 += 32) {
          int v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            v[j] = b0 + j < nb ? __ldg(blk_cnt + (size_t)(b0 + j) * E + e) : 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            p += b0 + j < b ? v[j] : 0;
            tot_e += v[j];
          }
        }
        *pre = p;
        *tot = tot_e;
      },
      [&](int p) { return rank[p]; });
}

// Up to kSchedRows rows (one block): counting and finishing in one CTA, the
// block's bitmap kept in shared memory, one launch instead of two.
__global__ void __launch_bounds__(256) k_sched_one(KArgs a) {
  __shared__ uint32_t bm[kMaxExperts][kSchedRows / 32];
  const int T = a.d.T, k = a.d.k, E = a.d.E, tid = threadIdx.x;
  for (int i = tid; i < E * (kSchedRows / 32); i += 256) (&bm[0][0])[i] = 0u;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int np = T * k;
  for (int i = tid; i < np; i += 256) {
    const int tl = i / k, e = a.w.idx[i];
    atomicOr(&bm[e][tl >> 5], 1u << (tl & 31));
  }
  __syncthreads();
  sched_finish_block(
      a, 0,
      [&](int e, int* pre, int* tot) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kSchedRows / 32; ++w) c += __popc(bm[e][w]);
        *pre = 0;
        *tot = c;
      },
      [&](int p) {
        const int tl = p / k, e = a.w.idx[p];
        int r = __popc(bm[e][tl >> 5] & ((1u << (tl & 31)) - 1u));
        for (int w = 0; w < (tl >> 5); ++w) r += __popc(bm[e][w]);
        return r;
      });
}

cudaError_t setup_schedule() { return cudaSuccess; }

cudaError_t launch_schedule(const KArgs& a, cudaStream_t s, bool pdl) {
  const int nb = (a.d.T + kSchedRows - 1) / kSchedRows;
  if (nb == 1) return launch_pdl(k_sched_one, dim3(1), dim3(256), 0, s, pdl, a);
  int* rank = a.w.sched_rank;
  int* blk = a.w.sched_blk;
  cudaError_t e = launch_pdl(k_sched_count, dim3(nb), dim3(256), 0, s, pdl, a, rank, blk);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_sched_finish, dim3(nb), dim3(256), 0, s, pdl, a, (const int*)rank,
                    (const int*)blk, nb);
}

}  // namespace moe

// Decode layer for 2..16 rows as one kernel over every SM, split by role
// like the one-row kernel:
//   routed CTAs (128): phase 1 computes gate/up units (16 SwiGLU features of
//      one selected expert for all rows that chose it: 16 gate + 16 up rows,
//      64 KB per unit through a two-slot ring) and publishes the SwiGLU
//      values; phase 2 computes down units (64 output rows of one expert: a
//      32 KB slice warmed in L2 during phase 1) from the polled SwiGLU values,
//      quantised as they are read, and publishes the expert outputs;
//   shared gate/up CTAs (H/128): shared SwiGLU features for all rows;
//   shared down CTAs (the rest): blocks of the shared expert's output rows.
// Every CTA computes router logits for experts b and b + G, all rows, in the
// register pass that quantises x and takes the shared gates.  The routed
// CTAs then each compute the top-k of every row and the same list of
// distinct experts.  Values move between CTAs as 64-bit {launch tag, value}
// words (decode_common.cuh), indexed by pair (row, rank): no grid barrier.
// The routed CTAs finish with the combine, y = sum_j w_j d_j (rank order) +
// gamma ds, 16 output rows of one row per item.
//
// Router and top-k: PR #939 "Fish Audio Drama 3 text to speech on one CUDA
// GPU", sections "What it adds" and "Fidelity against the PyTorch oracle".
// Expert arithmetic: PR #939 section "Precision".  SwiGLU storage: commit
// "one SwiGLU launch for the routed and shared experts".  Combine order:
// commit "MoE combine on 8-wide vectors".  Launch chaining: PR #927, section
// "What this changes".  Every wait is bounded (see decode_common.cuh).
#include <math.h>

#include "decode_common.cuh"

namespace moe {

namespace {

using namespace dec;

constexpr int kW = 8;
constexpr int kThreads = 32 * kW;
constexpr int kR = kDecodeRows;   // rows at most
constexpr int kGU = 16;           // SwiGLU features per gate/up unit
constexpr int kDN = 64;           // output rows per down unit
constexpr int kSlot = 64 * 1024;  // ring slot (two slots)
constexpr int kSdnSlots = 5;
constexpr int kSdnUnit = 32;
constexpr int kMaxRowH = 2048;
constexpr size_t kDataBytes = 208 * 1024;
constexpr size_t kPrefetchBytes = 48u << 20;  // W2 warmed in L2 at most

struct Roles {
  int P, nR, nS1, nS2, Fs, R2;
};

__host__ __device__ inline Roles rows_roles(int G, int H, int Is) {
  Roles r;
  r.P = H / kGroup;
  r.nS1 = r.P;
  r.nS2 = 8;
  r.nR = G - r.nS1 - r.nS2;
  r.Fs = Is / r.nS1;
  r.R2 = ((H + r.nS2 - 1) / r.nS2 + kSdnUnit - 1) / kSdnUnit * kSdnUnit;
  return r;
}

struct Small {
  int idx[kR * kMaxTopK];
  float w[kR * kMaxTopK];
  uint32_t tok[kMaxExperts];    // rows choosing expert e (bit t)
  int uexp[kMaxExperts];        // distinct experts, id order
  uint32_t umask[kMaxExperts];  // their rows
  int uoff[kMaxExperts];        // slots before them (rows of lower experts)
  int scan[kW];
  int U;
  float gred[kW * kR];
  float gamma[kR];
  int tag;
  float gmx[2][kW * 4];  // one scale per row: each warp's amax of a row group (two buffers)
  float hmx[kR * 8];     // one scale per row: group amaxes of an expert's SwiGLU rows
};

// Row strides in shared memory (padding keeps the 8 rows an MMA reads at once
// in different banks).
__host__ __device__ inline int xq_stride(int H) { return H + 64; }
__host__ __device__ inline int xs_stride(int H) { return 2 * H + 32; }
__host__ __device__ inline int hq_stride(int I) { return I + 64; }
__host__ __device__ inline int hs_stride(int Is) { return 2 * Is + 32; }

struct Lay {
  uint8_t* data;    // role area
  float* sx;        // [kR][H/128]
  float* red;       // router partials [2][kW][kR]
  uint64_t* bar;    // [8]
  Small* sm;
};

__host__ __device__ inline size_t rows_small(int H) {
  return al16((size_t)kR * (H / kGroup) * 4) + al16((size_t)2 * kW * kR * 4) + 8 * 8 +
         al16(sizeof(Small));
}

__device__ inline Lay rows_lay(uint8_t* smem, int H) {
  Lay L;
  uint8_t* p = smem;
  L.data = p;
  p += kDataBytes;
  L.sx = reinterpret_cast<float*>(p);
  p += al16((size_t)kR * (H / kGroup) * 4);
  L.red = reinterpret_cast<float*>(p);
  p += al16((size_t)2 * kW * kR * 4);
  L.bar = reinterpret_cast<uint64_t*>(p);
  p += 8 * 8;
  L.sm = reinterpret_cast<Small*>(p);
  return L;
}

// Routed role area: [ring slot 0][ring slot 1][xq rows][hq rows][sh][scales][partials]
struct RArea {
  uint8_t* slot[2];
  uint8_t* xq;   // [kR][xq_stride]
  uint8_t* hq;   // [kR][hq_stride]
  float* sh;     // [kR][I/128]
  float* sc;     // per slot: gate scale row, up scale row (widened), 2 x 2 x 32 floats
  float* part;   // [kW][2][32][NT][4]
};

__device__ inline RArea r_area(uint8_t* data, int H, int I) {
  RArea A;
  A.slot[0] = data;
  A.slot[1] = data + kSlot;
  uint8_t* p = data + 2 * kSlot;
  A.xq = p;
  p += (size_t)kR * xq_stride(H);
  A.hq = p;
  p += (size_t)kR * hq_stride(I);
  A.sh = reinterpret_cast<float*>(p);
  p += al16((size_t)kR * (I / kGroup) * 4);
  A.sc = reinterpret_cast<float*>(p);
  p += 2 * 2 * 32 * 4;
  A.part = reinterpret_cast<float*>(p);
  return A;
}

__host__ __device__ inline size_t r_area_bytes(int H, int I) {
  return (size_t)2 * kSlot + (size_t)kR * xq_stride(H) + (size_t)kR * hq_stride(I) +
         al16((size_t)kR * (I / kGroup) * 4) + 2 * 2 * 32 * 4 + (size_t)kW * 2 * 32 * 2 * 4 * 4;
}

// Exchange words: [kR*k][I] routed h, [kR*k][H] routed d, [kR][Is] hs, [kR][H] ds.
struct Xw {
  unsigned long long *h, *d, *hs, *ds;
};

__device__ inline Xw rows_xw(unsigned long long* base, int k, int H, int I, int Is) {
  Xw x;
  x.h = base;
  x.d = x.h + (size_t)kR * k * I;
  x.hs = x.d + (size_t)kR * k * H;
  x.ds = x.hs + (size_t)kR * Is;
  return x;
}

// Block exclusive scan over the kThreads threads' values.
__device__ inline int block_exscan(int v, int* total, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  int base = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    if (w < warp) base += scratch[w];
    all += scratch[w];
  }
  __syncthreads();
  *total = all;
  return base + inc - v;
}

// Position of the n-th (0-based) set bit of m.
__device__ __forceinline__ int nth_bit(uint32_t m, int n) {
  for (int i = 0; i < n; ++i) m &= m - 1u;
  return __ffs(m) - 1;
}

// Order this thread's earlier shared-memory accesses before bulk copies
// that reuse the same bytes.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Rank of expert e in row t's selection (k <= 16).
__device__ __forceinline__ int rank_in_row(const Small* sm, int k, int t, int e) {
  int j = 0;
  while (j < k - 1 && sm->idx[t * k + j] != e) ++j;
  return j;
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) k_decode_rows(KArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int G = gridDim.x, b = blockIdx.x;
  const int T = a.d.T, H = a.d.H, E = a.d.E, k = a.d.k, I = a.d.I, Is = a.d.Is;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int nbh = H / kGroup, nbi = I / kGroup;
  const Roles R = rows_roles(G, H, Is);
  const Lay L = rows_lay(smem, H);
  Small* sm = L.sm;
  const int* epoch = a.w.done + 4;
  int* status = a.w.status;
  const Xw X = rows_xw(a.w.xw, k, H, I, Is);
  const bool is_routed = b < R.nR;
  const bool is_sgu = !is_routed && b < R.nR + R.nS1;
  const bool is_sdn = !is_routed && !is_sgu;
  const int s1 = b - R.nR, s2 = b - R.nR - R.nS1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(&L.bar[i]);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  // ---- before the wait: the shared expert's weights and the router rows ----
  const uint32_t sgu_unit = 16u * (uint32_t)H * 2u;
  const uint32_t sdn_unit = (uint32_t)kSdnUnit * (uint32_t)Is * 2u;
  const int sdn_m0 = is_sdn ? s2 * R.R2 : 0;
  const int sdn_rows = is_sdn ? max(0, min(R.R2, H - sdn_m0)) : 0;
  const int n_sdn_units = sdn_rows / kSdnUnit;
  const int n_sgu_units = R.Fs / 8;
  if (threadIdx.x == 0) {
    if (is_sgu) {
      for (int u = 0; u < n_sgu_units && u < 2; ++u) {
        const int n0 = s1 * R.Fs + 8 * u;
        mbar_expect(&L.bar[u], sgu_unit);
        bulk_copy(L.data + (size_t)u * kSlot, a.L.ws13 + (size_t)n0 * H, sgu_unit / 2, &L.bar[u]);
        bulk_copy(L.data + (size_t)u * kSlot + sgu_unit / 2, a.L.ws13 + (size_t)(Is + n0) * H,
                  sgu_unit / 2, &L.bar[u]);
      }
    } else if (is_sdn) {
      for (int u = 0; u < n_sdn_units && u < kSdnSlots; ++u) {
        mbar_expect(&L.bar[u], sdn_unit);
        bulk_copy(L.data + (size_t)u * sdn_unit, a.L.ws2 + (size_t)(sdn_m0 + kSdnUnit * u) * Is,
                  sdn_unit, &L.bar[u]);
      }
    }
  }
  const int keighth = H / 8;
  const int k0 = warp * keighth;
  constexpr int kMaxV = kMaxRowH / 8 / 128;
  const int nv = keighth / 128;
  float4 wv[2][kMaxV];
  uint2 gw[kMaxV];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int er = b + G * h;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
      wv[h][i] = (er < E && i < nv)
                     ? __ldg(reinterpret_cast<const float4*>(a.L.wr + (size_t)er * H + k0 +
                                                             128 * i + 4 * lane))
                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
#pragma unroll
  for (int i = 0; i < kMaxV; ++i)
    gw[i] = i < nv ? __ldg(reinterpret_cast<const uint2*>(a.L.gate + k0 + 128 * i + 4 * lane))
                   : make_uint2(0u, 0u);
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) sm->tag = ld_acquire(epoch) + 1;

  // ---- router logits, x quantisation and the shared gates, all rows ----------
  RArea A = r_area(L.data, H, I);
  uint8_t* xs = L.data + 2 * kSlot;  // shared gate/up: x rows (bf16)
  // Rows go through in groups of kGR, in a loop that is not unrolled: the
  // pass runs once per launch, so its code is fetched cold every time and
  // must stay small.  The next group's x loads are in flight while the
  // current group is quantised and multiplied; within a group the per-row
  // warp reductions are interleaved so their shuffle chains overlap.
  constexpr int kGR = 4;
  uint2 xc[kMaxV][kGR], xn[kMaxV][kGR];
  auto load_group = [&](uint2 (&dst)[kMaxV][kGR], int t0) {
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
#pragma unroll
      for (int j = 0; j < kGR; ++j)
        dst[i][j] = (i < nv && t0 + j < T)
                        ? __ldcg(reinterpret_cast<const uint2*>(a.x + (size_t)(t0 + j) * H + k0 +
                                                                128 * i + 4 * lane))
                        : make_uint2(0u, 0u);
  };
  load_group(xc, 0);
#pragma unroll 1
  for (int t0 = 0; t0 < T; t0 += kGR) {
    if (t0 + kGR < T) load_group(xn, t0 + kGR);
    // 1 x 128 quantisation: group amax of every (slice, row), reduced together
    float gm[kMaxV][kGR];
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
#pragma unroll
      for (int j = 0; j < kGR; ++j) {
        const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&xc[i][j].x);
        const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&xc[i][j].y);
        gm[i][j] = fmaxf(fmaxf(fabsf(__low2float(p0)), fabsf(__high2float(p0))),
                         fmaxf(fabsf(__low2float(p1)), fabsf(__high2float(p1))));
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int i = 0; i < kMaxV; ++i)
#pragma unroll
        for (int j = 0; j < kGR; ++j)
          gm[i][j] = fmaxf(gm[i][j], __shfl_xor_sync(0xffffffffu, gm[i][j], o));
    if (a.d.per_row) {
      // one scale per row: every group of a row takes the row's amax, over
      // all warps (alternate buffers, so one barrier per row group suffices)
      static_assert(kGR == 4, "gmx holds four rows per warp");
      float* gmx = sm->gmx[(t0 / kGR) & 1];
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < kGR; ++j) {
          float v = 0.0f;
#pragma unroll
          for (int i = 0; i < kMaxV; ++i) v = fmaxf(v, gm[i][j]);
          gmx[warp * kGR + j] = v;
        }
      }
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kGR; ++j) {
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kW; ++w) v = fmaxf(v, gmx[w * kGR + j]);
#pragma unroll
        for (int i = 0; i < kMaxV; ++i) gm[i][j] = v;
      }
    }
    // router dot products (experts b, b + G) and the shared gate
    float acc[3][kGR];
#pragma unroll
    for (int j = 0; j < kGR; ++j) acc[0][j] = acc[1][j] = acc[2][j] = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
      if (i >= nv) continue;
      const int kk = k0 + 128 * i + 4 * lane;
      const __nv_bfloat162 g0 = *reinterpret_cast<const __nv_bfloat162*>(&gw[i].x);
      const __nv_bfloat162 g1 = *reinterpret_cast<const __nv_bfloat162*>(&gw[i].y);
#pragma unroll
      for (int j = 0; j < kGR; ++j) {
        const int t = t0 + j;
        const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&xc[i][j].x);
        const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&xc[i][j].y);
        const float x0 = __low2float(p0), x1 = __high2float(p0), x2 = __low2float(p1),
                    x3 = __high2float(p1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float v = acc[h][j];
          v = fmaf(x0, wv[h][i].x, v);
          v = fmaf(x1, wv[h][i].y, v);
          v = fmaf(x2, wv[h][i].z, v);
          v = fmaf(x3, wv[h][i].w, v);
          acc[h][j] = v;
        }
        float gs = acc[2][j];
        gs = fmaf(x0, __low2float(g0), gs);
        gs = fmaf(x1, __high2float(g0), gs);
        gs = fmaf(x2, __low2float(g1), gs);
        gs = fmaf(x3, __high2float(g1), gs);
        acc[2][j] = gs;
        if (t < T) {
          const float sc = group_scale(gm[i][j]);
          const uint32_t packed = quant4(x0, x1, x2, x3, sc);
          if (is_routed) {
            *reinterpret_cast<uint32_t*>(A.xq + (size_t)t * xq_stride(H) + kk) = packed;
            if (lane == 0) L.sx[t * nbh + kk / kGroup] = sc;
          } else if (is_sgu) {
            *reinterpret_cast<uint2*>(xs + (size_t)t * xs_stride(H) + 2 * kk) = xc[i][j];
          }
          if (b == 0) {
            *reinterpret_cast<uint32_t*>(a.w.xq + (size_t)t * H + kk) = packed;
            if (lane == 0) a.w.sx[(size_t)t * nbh + kk / kGroup] = sc;
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int h = 0; h < 3; ++h)
#pragma unroll
        for (int j = 0; j < kGR; ++j) acc[h][j] += __shfl_xor_sync(0xffffffffu, acc[h][j], o);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < kGR; ++j) {
        const int t = t0 + j;
        if (t >= T) break;
        L.red[(0 * kW + warp) * kR + t] = acc[0][j];
        L.red[(1 * kW + warp) * kR + t] = acc[1][j];
        sm->gred[warp * kR + t] = acc[2][j];
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
#pragma unroll
      for (int j = 0; j < kGR; ++j) xc[i][j] = xn[i][j];
  }
  __syncthreads();
  const unsigned long long tag = (unsigned long long)(unsigned)sm->tag << 32;
  if (threadIdx.x < 2 * T) {
    const int h = threadIdx.x / T, t = threadIdx.x % T;
    const int ee = b + G * h;
    if (ee < E) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kW; ++w) v += L.red[(h * kW + w) * kR + t];
      st_relaxed64(a.w.tlog + (size_t)t * E + ee, tag | __float_as_uint(v));
    }
  }
  if (threadIdx.x >= 64 && threadIdx.x < 64 + T) {
    const int t = threadIdx.x - 64;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kW; ++w) v += sm->gred[w * kR + t];
    sm->gamma[t] = sigmoid_f32(v);
    if (b == 0) a.w.gamma[t] = sm->gamma[t];
  }
  __syncthreads();

  if (is_routed) {
    // ---- logits of every row, top-k per row, the distinct experts --------
    float* lg = reinterpret_cast<float*>(A.slot[1]);  // [T][E], before the ring is used
    poll_range<kThreads>(a.w.tlog, T * E, tag, status, [&](int i, float v) { lg[i] = v; });
    for (int e = threadIdx.x; e < kMaxExperts; e += kThreads) sm->tok[e] = 0u;
    __syncthreads();
    for (int t = warp; t < T; t += kW)
      topk_row(lg + (size_t)t * E, E, k, sm->idx + t * k, sm->w + t * k, a.d.rbf16);
    __syncthreads();
    for (int p = threadIdx.x; p < T * k; p += kThreads)
      atomicOr(&sm->tok[sm->idx[p]], 1u << (p / k));
    __syncthreads();
    {
      const int e = threadIdx.x;
      const uint32_t msk = e < E ? sm->tok[e] : 0u;
      int U = 0, nrow = 0;
      const int pos = block_exscan(msk ? 1 : 0, &U, sm->scan);
      const int off = block_exscan(__popc(msk), &nrow, sm->scan);
      if (msk) {
        sm->uexp[pos] = e;
        sm->umask[pos] = msk;
        sm->uoff[pos] = off;
      }
      if (threadIdx.x == 0) sm->U = U;
    }
    __syncthreads();
    const int U = sm->U;
    if (b == 0) {
      // routing and slot order (experts by id, rows in order) for the checking entry points
      for (int p = threadIdx.x; p < T * k; p += kThreads) {
        const int t = p / k, e = sm->idx[p];
        int u = 0;
        while (sm->uexp[u] != e) ++u;
        const int slot = sm->uoff[u] + __popc(sm->umask[u] & ((1u << t) - 1u));
        a.w.idx[p] = e;
        a.w.wts[p] = sm->w[p];
        a.w.slot_of_pair[p] = slot;
        a.w.pair_of_slot[slot] = p;
      }
      for (int u = threadIdx.x; u < U; u += kThreads)
        a.w.chunks[u] = make_int4(sm->uexp[u], sm->uoff[u], __popc(sm->umask[u]), 0);
      if (threadIdx.x == 0) *a.w.n_chunks = U;
    }

    // ---- phase 1: gate/up units of 16 features, two-slot ring ---------------
    const int nF = I / kGU;
    const int n1 = U * nF;
    const uint32_t uhalf = (uint32_t)kGU * H;
    auto issue_gu = [&](int v, int s) {
      const int u = v / nF, f = v % nF;
      const int e = sm->uexp[u];
      const uint8_t* W13 = a.L.w13 + (size_t)e * 2 * I * H;
      const float* S13 = a.L.s13 + (size_t)e * (2 * I / kGroup) * nbh;
      const float *lo_g, *lo_u;
      int dg, du;
      const uint32_t bg = span16(S13 + (size_t)(kGU * f / kGroup) * nbh, nbh, &lo_g, &dg);
      const uint32_t bu = span16(S13 + (size_t)((I + kGU * f) / kGroup) * nbh, nbh, &lo_u, &du);
      float* sc = A.sc + s * 64;
      mbar_expect(&L.bar[s], 2 * uhalf + bg + bu);
      bulk_copy(A.slot[s], W13 + (size_t)(kGU * f) * H, uhalf, &L.bar[s]);
      bulk_copy(A.slot[s] + uhalf, W13 + (size_t)(I + kGU * f) * H, uhalf, &L.bar[s]);
      bulk_copy(sc, lo_g, bg, &L.bar[s]);
      bulk_copy(sc + 32, lo_u, bu, &L.bar[s]);
    };
    // each CTA takes a contiguous block of units (consecutive features of
    // one expert share its rows)
    const int per1 = (n1 + R.nR - 1) / R.nR;
    const int v1a = min(n1, b * per1), v1b = min(n1, v1a + per1);
    if (threadIdx.x == 0) {
      fence_proxy_async();  // the ring held the logits
      for (int i = 0; i < 2 && v1a + i < v1b; ++i) issue_gu(v1a + i, i);
    }
    // warm this CTA's phase-2 down slices in L2 while phase 1 streams
    const int nP = H / kDN;
    const int n2 = U * nP;
    const int per2 = (n2 + R.nR - 1) / R.nR;
    const int v2a = min(n2, b * per2), v2b = min(n2, v2a + per2);
    if (warp == kW - 1 && (size_t)U * H * I <= kPrefetchBytes) {
      for (int v = v2a + lane; v < v2b; v += 32) {
        const int u = v / nP, pp = v % nP;
        prefetch_l2(a.L.w2 + ((size_t)sm->uexp[u] * H + (size_t)kDN * pp) * I,
                    (uint32_t)kDN * I);
      }
    }
    for (int i = 0; v1a + i < v1b; ++i) {
      const int v = v1a + i;
      const int s = i & 1;
      const int u = v / nF, f = v % nF;
      const uint32_t msk = sm->umask[u];
      const int nt = __popc(msk);
      copy_wait(&L.bar[s], (uint32_t)((i >> 1) & 1), status);
      // warp = K eighth; it covers both 8-feature m-tiles, so each token
      // fragment is read from shared memory once
      const uint8_t* rows = A.slot[s];
      const float* sg = A.sc + s * 64;
      const float* su = sg + 32;
      const float* lo;
      int dg, du;
      {
        const int e = sm->uexp[u];
        const float* S13 = a.L.s13 + (size_t)e * (2 * I / kGroup) * nbh;
        span16(S13 + (size_t)(kGU * f / kGroup) * nbh, nbh, &lo, &dg);
        span16(S13 + (size_t)((I + kGU * f) / kGroup) * nbh, nbh, &lo, &du);
      }
      sg += dg;
      su += du;
      // token columns: the rows of expert u, in order
      const uint8_t* xb[NT];
      const float* sxc[NT][2];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int cg = min(8 * n + g, nt - 1);
        xb[n] = A.xq + (size_t)(nth_bit(msk, cg)) * xq_stride(H);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int cc = min(8 * n + 2 * q + c, nt - 1);
          sxc[n][c] = L.sx + (size_t)(nth_bit(msk, cc)) * nbh;
        }
      }
      float acc[2][NT][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[mt][n][0] = acc[mt][n][1] = acc[mt][n][2] = acc[mt][n][3] = 0.0f;
      const int nsl = H / 64, per = nsl / kW;
#pragma unroll 2
      for (int bs = warp * per; bs < warp * per + per; ++bs) {
        const int kb = bs >> 1;
        const int off = bs * 64 + 16 * q;
        uint4 ag[2], au[2], bx[NT];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          ag[mt] = lds16(rows + (size_t)(8 * mt + g) * H + off);
          au[mt] = lds16(rows + uhalf + (size_t)(8 * mt + g) * H + off);
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) bx[n] = lds16(xb[n] + off);
        const float wgs = sg[kb], wus = su[kb];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const float sa0 = sxc[n][0][kb], sa1 = sxc[n][1][kb];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            float pp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            mma_e4m3_k64(pp, ag[mt], au[mt], bx[n]);
            acc[mt][n][0] = fmaf(pp[0], wgs * sa0, acc[mt][n][0]);
            acc[mt][n][1] = fmaf(pp[1], wgs * sa1, acc[mt][n][1]);
            acc[mt][n][2] = fmaf(pp[2], wus * sa0, acc[mt][n][2]);
            acc[mt][n][3] = fmaf(pp[3], wus * sa1, acc[mt][n][3]);
          }
        }
      }
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            A.part[(((warp * 2 + mt) * 32 + lane) * NT + n) * 4 + c] = acc[mt][n][c];
      __syncthreads();
      // the slot is free: the unit two steps ahead
      if (threadIdx.x == 0 && v1a + i + 2 < v1b) {
        fence_proxy_async();
        issue_gu(v1a + i + 2, s);
      }
      {
        // one output per thread: (m-tile, lane, token tile, column), the
        // K eighths summed in order, then SwiGLU and publish
        const int o = threadIdx.x;  // 2 * 32 * NT * 2 outputs when NT == 2
        if (o < 2 * 32 * NT * 2) {
          const int mt = o / (32 * NT * 2), rem = o % (32 * NT * 2);
          const int ln = rem / (NT * 2), n = (rem / 2) % NT, c = rem % 2;
          float zg = 0.0f, zu = 0.0f;
#pragma unroll
          for (int w8 = 0; w8 < kW; ++w8) {
            const float* pp = A.part + (((w8 * 2 + mt) * 32 + ln) * NT + n) * 4;
            zg += pp[c];
            zu += pp[2 + c];
          }
          const int col = 8 * n + 2 * (ln & 3) + c;
          if (col < nt) {
            const int e = sm->uexp[u];
            const int t = nth_bit(msk, col);
            const float h = silu_f32(bf16_round(zg)) * bf16_round(zu);
            const int pair = t * k + rank_in_row(sm, k, t, e);
            publish(X.h + (size_t)pair * I + kGU * f + 8 * mt + (ln >> 2), tag, h);
          }
        }
      }
      __syncthreads();
    }

    // ---- phase 2: down units of 64 output rows ------------------------------
    // slices through four 32 KB slots of the ring (bars 2..5)
    const uint32_t dbytes = (uint32_t)kDN * I;
    auto issue_dn = [&](int v, int s) {
      const int u = v / nP, pp = v % nP;
      mbar_expect(&L.bar[2 + s], dbytes);
      bulk_copy(A.slot[0] + (size_t)s * dbytes,
                a.L.w2 + ((size_t)sm->uexp[u] * H + (size_t)kDN * pp) * I, dbytes, &L.bar[2 + s]);
    };
    const int nds = (int)((2u * kSlot) / dbytes) < 4 ? (int)((2u * kSlot) / dbytes) : 4;
    if (threadIdx.x == 0) {
      fence_proxy_async();  // the ring held phase 1's rows
      for (int i = 0; i < nds && v2a + i < v2b; ++i) issue_dn(v2a + i, i);
    }
    int u_have = -1;  // expert whose quantised SwiGLU rows are in hq
    float* hstage = reinterpret_cast<float*>(A.xq);  // [nt][I] fp32 (x codes are done with)
    for (int i = 0; v2a + i < v2b; ++i) {
      const int v = v2a + i;
      const int s = i % nds;
      const int u = v / nP, pp = v % nP;
      const int e = sm->uexp[u];
      const uint32_t msk = sm->umask[u];
      const int nt = __popc(msk);
      // SwiGLU values of expert e for its rows, once per expert: every
      // thread's loads issued in batches into fp32 staging, then quantised
      // per (row, group) by warp w's items w, w + 8, ...
      if (u != u_have) {
        u_have = u;
        __syncthreads();  // the previous expert's rows are no longer read
        poll_gather<kThreads>(
            nt * I, tag, status,
            [&](int i2) {
              const int col = i2 / I, c = i2 - col * I;
              const int t = nth_bit(msk, col);
              return X.h + (size_t)(t * k + rank_in_row(sm, k, t, e)) * I + c;
            },
            [&](int i2, float val) { hstage[i2] = val; });
        __syncthreads();
        if (a.d.per_row) {
          // one scale per row: the group amaxes first, then each row's
          for (int it = warp; it < nt * nbi; it += kW) {
            const int col = it / nbi, grp = it % nbi;
            const float4 hv = *reinterpret_cast<const float4*>(hstage + (size_t)col * I +
                                                               grp * kGroup + 4 * lane);
            const float m =
                warp_max(fmaxf(fmaxf(fabsf(hv.x), fabsf(hv.y)), fmaxf(fabsf(hv.z), fabsf(hv.w))));
            if (lane == 0) sm->hmx[it] = m;
          }
          __syncthreads();
        }
        for (int it = warp; it < nt * nbi; it += kW) {
          const int col = it / nbi, grp = it % nbi;
          const float4 hv =
              *reinterpret_cast<const float4*>(hstage + (size_t)col * I + grp * kGroup + 4 * lane);
          float m = fmaxf(fmaxf(fabsf(hv.x), fabsf(hv.y)), fmaxf(fabsf(hv.z), fabsf(hv.w)));
          m = warp_max(m);
          if (a.d.per_row) {
            m = 0.0f;
            for (int g2 = 0; g2 < nbi; ++g2) m = fmaxf(m, sm->hmx[col * nbi + g2]);
          }
          const float sq = group_scale(m);
          const uint32_t packed = quant4(hv.x, hv.y, hv.z, hv.w, sq);
          *reinterpret_cast<uint32_t*>(A.hq + (size_t)col * hq_stride(I) + grp * kGroup +
                                       4 * lane) = packed;
          if (lane == 0) A.sh[col * nbi + grp] = sq;
          if (pp == 0) {  // the expert's first block writes its rows for the checking calls
            const int slot = sm->uoff[u] + col;
            *reinterpret_cast<uint32_t*>(a.w.hq + (size_t)slot * I + grp * kGroup + 4 * lane) =
                packed;
            if (lane == 0) a.w.sh[(size_t)slot * nbi + grp] = sq;
          }
        }
      }
      __syncthreads();
      copy_wait(&L.bar[2 + s], (uint32_t)((i / nds) & 1), status);
      const uint8_t* w2s = A.slot[0] + (size_t)s * dbytes;  // [64][I]
      const float* s2 = a.L.s2 + ((size_t)e * nbh + (size_t)(kDN * pp) / kGroup) * nbi;
      // warp = (m-tile mt of 16 rows, K half kh)
      const int mt = warp & 3, kh = warp >> 2;
      const uint8_t* hb[NT];
      const float* shc[NT][2];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int cg = min(8 * n + g, nt - 1);
        hb[n] = A.hq + (size_t)cg * hq_stride(I);
#pragma unroll
        for (int c = 0; c < 2; ++c) shc[n][c] = A.sh + min(8 * n + 2 * q + c, nt - 1) * nbi;
      }
      float acc[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
      const int nsl = I / 64, per = nsl / 2;
      const uint8_t* rows = w2s + (size_t)(16 * mt) * I;
      for (int bs = kh * per; bs < kh * per + per; ++bs) {
        const int grp = bs >> 1;
        const int off = bs * 64 + 16 * q;
        const uint4 a_lo = lds16(rows + (size_t)g * I + off);
        const uint4 a_hi = lds16(rows + (size_t)(8 + g) * I + off);
        const float ws = __ldg(s2 + grp);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const uint4 bx = lds16(hb[n] + off);
          float p4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          mma_e4m3_k64(p4, a_lo, a_hi, bx);
          const float sa0 = shc[n][0][grp], sa1 = shc[n][1][grp];
          acc[n][0] = fmaf(p4[0], ws * sa0, acc[n][0]);
          acc[n][1] = fmaf(p4[1], ws * sa1, acc[n][1]);
          acc[n][2] = fmaf(p4[2], ws * sa0, acc[n][2]);
          acc[n][3] = fmaf(p4[3], ws * sa1, acc[n][3]);
        }
      }
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) A.part[((warp * 32 + lane) * NT + n) * 4 + c] = acc[n][c];
      __syncthreads();
      if (threadIdx.x == 0 && v2a + i + nds < v2b) {
        fence_proxy_async();
        issue_dn(v2a + i + nds, s);
      }
      if (warp < 4) {  // warp mt: its 16 rows, both K halves in order
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          float dv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dv[c] = A.part[((warp * 32 + lane) * NT + n) * 4 + c] +
                    A.part[(((4 + warp) * 32 + lane) * NT + n) * 4 + c];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int col = 8 * n + 2 * q + c;
            if (col < nt) {
              const int t = nth_bit(msk, col);
              const int pair = t * k + rank_in_row(sm, k, t, e);
              const int m = kDN * pp + 16 * warp + g;
              publish(X.d + (size_t)pair * H + m, tag, bf16_round(dv[c]));
              publish(X.d + (size_t)pair * H + m + 8, tag, bf16_round(dv[2 + c]));
            }
          }
        }
      }
      __syncthreads();
    }

    // ---- combine: items (row t, 16 output rows) --------------------------------
    const int nchunk = H / 16;
    for (int it = b; it < T * nchunk; it += R.nR) {
      const int t = it / nchunk, m0 = 16 * (it % nchunk);
      float* comb = A.part;  // [k + 1][16]
      for (int i = threadIdx.x; i < (k + 1) * 16; i += kThreads) {
        const int j = i / 16, r = i % 16;
        comb[i] = j < k ? poll_tagged(X.d + (size_t)(t * k + j) * H + m0 + r, tag, status)
                        : poll_tagged(X.ds + (size_t)t * H + m0 + r, tag, status);
      }
      __syncthreads();
      if (threadIdx.x < 16) {
        float y = 0.0f;
        for (int j = 0; j < k; ++j) y = fmaf(sm->w[t * k + j], comb[j * 16 + threadIdx.x], y);
        y = fmaf(sm->gamma[t], comb[k * 16 + threadIdx.x], y);
        a.y[(size_t)t * H + m0 + threadIdx.x] = __float2bfloat16_rn(y);
      }
      __syncthreads();
    }
  } else if (is_sgu) {
    // ---- shared gate/up: units of [8 gate; 8 up] rows, all warps split K ----
    const int nsl = H / 32, per = nsl / kW;
    for (int uu = 0; uu < n_sgu_units; ++uu) {
      const int s = uu & 1;
      copy_wait(&L.bar[s], (uint32_t)((uu >> 1) & 1), status);
      const uint8_t* rows = L.data + (size_t)s * kSlot;
      const size_t row = (size_t)2 * H;
      float acc[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
      const uint8_t* xb[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) xb[n] = xs + (size_t)min(8 * n + g, T - 1) * xs_stride(H);
#pragma unroll 4
      for (int bs = warp * per; bs < warp * per + per; ++bs) {
        const int off = bs * 32 + 8 * q;  // elements
        const uint4 ag = lds16(rows + (size_t)g * row + 2 * off);
        const uint4 au = lds16(rows + (size_t)(8 + g) * row + 2 * off);
#pragma unroll
        for (int n = 0; n < NT; ++n) mma_bf16_k32(acc[n], ag, au, lds16(xb[n] + 2 * off));
      }
      float* part = reinterpret_cast<float*>(xs + (size_t)kR * xs_stride(H));
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int c = 0; c < 4; ++c) part[((warp * 32 + lane) * NT + n) * 4 + c] = acc[n][c];
      __syncthreads();
      if (threadIdx.x == 0 && uu + 2 < n_sgu_units) {
        fence_proxy_async();
        const int n0 = s1 * R.Fs + 8 * (uu + 2);
        mbar_expect(&L.bar[s], sgu_unit);
        bulk_copy(L.data + (size_t)s * kSlot, a.L.ws13 + (size_t)n0 * H, sgu_unit / 2, &L.bar[s]);
        bulk_copy(L.data + (size_t)s * kSlot + sgu_unit / 2, a.L.ws13 + (size_t)(Is + n0) * H,
                  sgu_unit / 2, &L.bar[s]);
      }
      if (warp == 0) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          for (int w = 0; w < kW; ++w)  // parts in K order
#pragma unroll
            for (int c = 0; c < 4; ++c) z[c] += part[((w * 32 + lane) * NT + n) * 4 + c];
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int t = 8 * n + 2 * q + c;
            if (t < T) {
              const float hs = bf16_round(silu_f32(bf16_round(z[c])) * bf16_round(z[2 + c]));
              publish(X.hs + (size_t)t * Is + s1 * R.Fs + 8 * uu + g, tag, hs);
            }
          }
        }
      }
      __syncthreads();
    }
  } else if (sdn_rows > 0) {
    // ---- shared down: rows [sdn_m0, +sdn_rows), 32 per unit, one warp each ----
    uint8_t* hsb = L.data + (size_t)kSdnSlots * sdn_unit;  // [kR][hs_stride] bf16
    poll_range<kThreads>(X.hs, T * Is, tag, status, [&](int i, float v) {
      const int t = i / Is, c = i % Is;
      reinterpret_cast<bf16*>(hsb + (size_t)t * hs_stride(Is))[c] = __float2bfloat16_rn(v);
    });
    __syncthreads();
    const uint8_t* hb[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) hb[n] = hsb + (size_t)min(8 * n + g, T - 1) * hs_stride(Is);
    for (int uu = warp; uu < n_sdn_units; uu += kW) {
      const int slot = uu % kSdnSlots;
      copy_wait(&L.bar[slot], (uint32_t)((uu / kSdnSlots) & 1), status);
      const uint8_t* rows = L.data + (size_t)slot * sdn_unit;
      for (int tile = 0; tile < kSdnUnit / 16; ++tile) {
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
        const uint8_t* tr = rows + (size_t)(16 * tile) * Is * 2;
#pragma unroll 4
        for (int bs = 0; bs < Is / 32; ++bs) {
          const int off = bs * 32 + 8 * q;
          const uint4 a_lo = lds16(tr + (size_t)g * Is * 2 + 2 * off);
          const uint4 a_hi = lds16(tr + (size_t)(8 + g) * Is * 2 + 2 * off);
#pragma unroll
          for (int n = 0; n < NT; ++n) mma_bf16_k32(acc[n], a_lo, a_hi, lds16(hb[n] + 2 * off));
        }
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int t = 8 * n + 2 * q + c;
            if (t < T) {
              const int m = sdn_m0 + kSdnUnit * uu + 16 * tile + g;
              publish(X.ds + (size_t)t * H + m, tag, bf16_round(acc[n][c]));
              publish(X.ds + (size_t)t * H + m + 8, tag, bf16_round(acc[n][2 + c]));
            }
          }
      }
      __syncwarp();
      const int un = uu + kSdnSlots;
      if (lane == 0 && un < n_sdn_units) {
        fence_proxy_async();
        mbar_expect(&L.bar[slot], sdn_unit);
        bulk_copy(L.data + (size_t)slot * sdn_unit,
                  a.L.ws2 + (size_t)(sdn_m0 + kSdnUnit * un) * Is, sdn_unit, &L.bar[slot]);
      }
    }
  }

  // ---- exit: the last CTA advances the launch tag (or clears the words) ----
  launch_exit(a, sm->tag);
}

}  // namespace

size_t decode_rows_smem(int H) { return kDataBytes + rows_small(H); }

bool decode_rows_fits(int G, int H, int E, int k, int I, int Is, size_t budget) {
  if (H % 1024 != 0 || H > kMaxRowH) return false;
  if (E > 2 * G || E > kMaxExperts || k > kMaxTopK) return false;
  const Roles R = rows_roles(G, H, Is);
  if (R.nR < 32 || Is % R.nS1 != 0 || R.Fs < 8 || R.Fs % 8 != 0) return false;
  if ((H / 32) % kW != 0 || (H / 64) % kW != 0) return false;
  if (I % kGU != 0 || I % kGroup != 0 || I / kGroup > 8 || (I / 64) % 2 != 0) return false;
  if (H % kDN != 0 || (size_t)kDN * I > (size_t)kSlot) return false;
  if ((size_t)2 * kGU * H > (size_t)kSlot || (size_t)16 * H * 2 > (size_t)kSlot) return false;
  if ((size_t)kSdnSlots * kSdnUnit * Is * 2 + (size_t)kR * hs_stride(Is) > kDataBytes) return false;
  if ((size_t)2 * kSlot + (size_t)kR * xs_stride(H) + (size_t)kW * 32 * 2 * 4 * 4 > kDataBytes)
    return false;
  if (r_area_bytes(H, I) > kDataBytes) return false;
  if ((size_t)kR * E * 4 > (size_t)kSlot) return false;
  if (R.R2 % kSdnUnit != 0 || (size_t)R.R2 * R.nS2 < (size_t)H) return false;
  return decode_rows_smem(H) <= budget;
}

cudaError_t setup_decode_rows(size_t max_smem) {
  cudaError_t e = cudaFuncSetAttribute(k_decode_rows<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_decode_rows<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)max_smem);
}

cudaError_t launch_decode_rows(const KArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s) {
  if (a.d.T <= 8)
    return launch_pdl(k_decode_rows<1>, dim3(grid), dim3(kThreads), smem, s, pdl, a);
  return launch_pdl(k_decode_rows<2>, dim3(grid), dim3(kThreads), smem, s, pdl, a);
}

}  // namespace moe

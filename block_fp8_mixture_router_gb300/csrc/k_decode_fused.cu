// Decode layer (rows <= 16) as one persistent kernel: one CTA per SM.
//
//   A  router logits (each CTA one or two experts), published as 64-bit
//      {launch tag, value} words; the shared expert's gate/up tile copy (one
//      [8 gate; 8 up] bf16 row tile for each of the first Is/8 CTAs) and the
//      router rows are requested before the kernel waits on its predecessor.
//   B  every CTA quantises x itself, gathers all logits (polling the tags),
//      takes the same top-k and builds the same schedule, then streams its
//      routed gate/up tiles (8 gate + 8 up e4m3 rows of one selected expert,
//      full K, plus their two block-scale rows) through a ring of shared-
//      memory stages (four 1-D bulk copies per tile) and writes SwiGLU rows.
//      Its shared tile is computed once its routed copies are in flight.  When
//      its last tile is done it copies what phase C needs (the selected
//      experts' and the shared expert's down slices, warmed in L2 during
//      phase B) into shared memory, and arrives at the grid barrier.
//   C  16 output rows per CTA: the SwiGLU rows are re-quantised (every CTA the
//      same way), the down slices are applied, and the combine writes y.
//
// The one-row layer is bound by its 33.6 MB of weights; what costs time
// beyond that is latency: dependent global round trips, long dependent
// instruction chains in one warp, and bulk-copy issue (tens of nanoseconds
// each).  Each phase therefore issues all its loads together, in few large
// copies, and waits once.
//
// Launch chaining follows PR #927 "backbone chain launches with PDL", section
// "What this changes" (wait before reading the predecessor's results;
// immutable weights may be fetched before the wait).  Router and top-k:
// PR #939 "Fish Audio Drama 3 text to speech on one CUDA GPU", sections "What
// it adds" and "Fidelity against the PyTorch oracle" (near-tied 8th/9th
// experts; the lower index wins).  Expert arithmetic: PR #939 section
// "Precision" (e4m3 inputs per row and per 128 inputs, amax/448).  SwiGLU
// storage: commit "one SwiGLU launch for the routed and shared experts".
// Combine order: commit "MoE combine on 8-wide vectors".
//
// Every wait is bounded: a poll, grid barrier or bulk copy that does not
// complete within the spin limit sets the context's status flag and the
// kernel runs to its end without waiting further (its output is then
// undefined, and the host reports MOE_ERR_DEVICE_TIMEOUT).
#include <math.h>

#include "moe_rowops.cuh"

namespace moe {

namespace {

constexpr int kW = 8;               // warps per CTA
constexpr int kThreads = 32 * kW;
constexpr int kMaxStages = 6;
constexpr int kRowPad = 64;         // bytes between staged activation rows
constexpr long long kSpinLimit = 1ll << 22;
constexpr size_t kDownPrefetchBytes = 48u << 20;

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

__device__ __forceinline__ void mbar_expect_only(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(sa(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(sa(bar)) : "memory");
}

__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(sa(dst)),
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

__device__ __forceinline__ uint4 lds16(const void* p) { return *reinterpret_cast<const uint4*>(p); }

__host__ __device__ __forceinline__ size_t al16(size_t v) { return (v + 15) & ~(size_t)15; }

// Bytes reserved for one staged scale row of n floats (room for widening).
__host__ __device__ __forceinline__ size_t scale_slot(int n) { return al16((size_t)n * 4 + 16); }

// A bulk copy must start on a 16-byte boundary and move a multiple of 16
// bytes: widen [src, src + n) to 16-byte boundaries (the scale arrays are
// 16-byte aligned at their start and a multiple of 16 bytes long, so the
// widened range stays inside them).  Returns the bytes; *lo the widened start,
// *delta the floats between *lo and src.
__device__ __forceinline__ uint32_t scale_span(const float* src, int n, const float** lo,
                                               int* delta) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(src) & ~(uintptr_t)15;
  const uintptr_t a1 = (reinterpret_cast<uintptr_t>(src + n) + 15) & ~(uintptr_t)15;
  *lo = reinterpret_cast<const float*>(a0);
  *delta = (int)((reinterpret_cast<uintptr_t>(src) - a0) / 4);
  return (uint32_t)(a1 - a0);
}

struct Sched {
  int idx[kDecodeRows * kMaxTopK];
  float w[kDecodeRows * kMaxTopK];
  int slot_of_pair[kDecodeRows * kMaxTopK];
  int pair_of_slot[kDecodeRows * kMaxTopK];
  uint32_t tok[kMaxExperts];
  int4 chunk[kMaxExperts];   // {expert, first slot, rows, 0}
  uint32_t cand_key[2 * kW * kMaxTopK];
  uint32_t cand_id[2 * kW * kMaxTopK];
  float gred[kW * kDecodeRows];
  int scan[kW];
  int n_used;
  int tag;
};

// Shared memory: [stages][red][xq rows][sx][logits][gates][mbarriers][schedule].
struct Layout {
  int n_stages, stage_bytes, xq_stride, nbh;
  uint8_t* stages;
  float* red;      // [kW][2][4][32]
  uint8_t* xq;     // [T][xq_stride]
  float* sx;       // [T][H/128]
  float* lg;       // [T][E]
  float* gam;      // [kDecodeRows]
  uint64_t* bar;   // [kMaxStages + 2]
  Sched* sc;
};

// A stage: 16 rows of K = H bytes, then the gate and up block-scale rows.
__host__ __device__ __forceinline__ size_t stage_bytes_for(int H) {
  return al16((size_t)16 * H + 2 * scale_slot(H / kGroup));
}

__host__ __device__ __forceinline__ size_t smem_after_stages(int T, int H, int E) {
  return (size_t)kW * 2 * 4 * 32 * 4 + al16((size_t)T * (H + kRowPad)) +
         al16((size_t)T * (H / kGroup) * 4) + al16((size_t)T * E * 4) + kDecodeRows * 4 +
         (kMaxStages + 2) * 8 + al16(sizeof(Sched));
}

__device__ __forceinline__ Layout layout(uint8_t* smem, int T, int H, int E, int n_stages) {
  Layout L;
  L.n_stages = n_stages;
  L.stage_bytes = (int)stage_bytes_for(H);
  L.xq_stride = H + kRowPad;
  L.nbh = H / kGroup;
  L.stages = smem;
  uint8_t* p = smem + (size_t)n_stages * L.stage_bytes;
  L.red = reinterpret_cast<float*>(p);
  p += (size_t)kW * 2 * 4 * 32 * 4;
  L.xq = p;
  p += al16((size_t)T * L.xq_stride);
  L.sx = reinterpret_cast<float*>(p);
  p += al16((size_t)T * L.nbh * 4);
  L.lg = reinterpret_cast<float*>(p);
  p += al16((size_t)T * E * 4);
  L.gam = reinterpret_cast<float*>(p);
  p += kDecodeRows * 4;
  L.bar = reinterpret_cast<uint64_t*>(p);
  p += (kMaxStages + 2) * 8;
  L.sc = reinterpret_cast<Sched*>(p);
  return L;
}

// Phase C carve-up of the stage area: R down slots, the shared down slice,
// then the re-quantised rows and the partial outputs.
struct CLayout {
  size_t slot_bytes, ws2, hq, sh, hs, d, ds, end;
  int R, hq_stride, hs_stride;
};

__host__ __device__ __forceinline__ CLayout c_layout(int T, int k, int I, int Is, int U,
                                                     size_t area) {
  CLayout c;
  const int P = T * k;
  c.hq_stride = I + 16;
  c.hs_stride = 2 * Is + 16;
  c.slot_bytes = al16((size_t)16 * I + scale_slot(I / kGroup));
  const size_t tail = al16((size_t)16 * Is * 2) + al16((size_t)P * c.hq_stride) +
                      al16((size_t)P * (I / kGroup) * 4) + al16((size_t)T * c.hs_stride) +
                      al16((size_t)P * 16 * 4) + al16((size_t)2 * kDecodeRows * 16 * 4);
  int R = area > tail ? (int)((area - tail) / c.slot_bytes) : 0;
  if (R > U) R = U;
  c.R = R;
  c.ws2 = (size_t)R * c.slot_bytes;
  c.hq = c.ws2 + al16((size_t)16 * Is * 2);
  c.sh = c.hq + al16((size_t)P * c.hq_stride);
  c.hs = c.sh + al16((size_t)P * (I / kGroup) * 4);
  c.d = c.hs + al16((size_t)T * c.hs_stride);
  c.ds = c.d + al16((size_t)P * 16 * 4);
  c.end = c.ds + al16((size_t)2 * kDecodeRows * 16 * 4);
  return c;
}

// Block exclusive scan over kThreads values.
__device__ int exscan(int v, int* total, int* scratch) {
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

__device__ __forceinline__ void grid_arrive(int* counter) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(counter, 1);
  }
}

__device__ void grid_wait(int* counter, int target, int* status) {
  if (threadIdx.x == 0) {
    long long it = 0;
    while (ld_acquire(counter) < target) {
      if (++it > kSpinLimit) {
        atomicExch(status, 1);
        break;
      }
      if (it > 16) __nanosleep(32);
    }
    __threadfence();
  }
  __syncthreads();
}

__device__ __forceinline__ void stage_wait(uint64_t* bar, uint32_t parity, int* status) {
  long long it = 0;
  while (!mbar_test(bar, parity)) {
    if (++it > kSpinLimit) {
      atomicExch(status, 1);
      break;
    }
  }
}

// Every CTA quantises all T rows of x into its own shared memory (1 x 128
// groups, scale amax/448) and computes the shared-expert gates
// sigmoid(x . g): cheaper than waiting for another CTA's copy.  CTA 0 also
// writes them to the workspace for the checking entry points.
__device__ void quant_rows_local(const KArgs& a, const Layout& L, bool publish, uint4 gate8) {
  const int T = a.d.T, H = a.d.H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ngroups = H / kGroup;
  constexpr int kIlp = 4;
  for (int base = warp * kIlp; base < T * ngroups; base += kW * kIlp) {
    float v[kIlp][4];
#pragma unroll
    for (int u = 0; u < kIlp; ++u) {
      const int pg = base + u;
      uint2 raw = make_uint2(0u, 0u);
      if (pg < T * ngroups)
        raw = __ldcg(reinterpret_cast<const uint2*>(a.x + (size_t)(pg / ngroups) * H +
                                                    (pg % ngroups) * kGroup + 4 * lane));
      const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
      const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
      v[u][0] = __low2float(p0);
      v[u][1] = __high2float(p0);
      v[u][2] = __low2float(p1);
      v[u][3] = __high2float(p1);
    }
    float m[kIlp];
#pragma unroll
    for (int u = 0; u < kIlp; ++u)
      m[u] = fmaxf(fmaxf(fabsf(v[u][0]), fabsf(v[u][1])), fmaxf(fabsf(v[u][2]), fabsf(v[u][3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < kIlp; ++u) m[u] = fmaxf(m[u], __shfl_xor_sync(0xffffffffu, m[u], o));
#pragma unroll
    for (int u = 0; u < kIlp; ++u) {
      const int pg = base + u;
      if (pg >= T * ngroups) break;
      const int t = pg / ngroups, gi = pg % ngroups;
      const float s = group_scale(m[u]);
      const uint32_t packed = quant4(v[u][0], v[u][1], v[u][2], v[u][3], s);
      *reinterpret_cast<uint32_t*>(L.xq + (size_t)t * L.xq_stride + gi * kGroup + 4 * lane) = packed;
      if (lane == 0) L.sx[t * ngroups + gi] = s;
      if (publish) {
        *reinterpret_cast<uint32_t*>(a.w.xq + (size_t)t * H + gi * kGroup + 4 * lane) = packed;
        if (lane == 0) a.w.sx[(size_t)t * ngroups + gi] = s;
      }
    }
  }
  // gates: thread j holds gate elements [8j, 8j+8) (loaded before the wait;
  // H <= 2048); partial sums added lane-tree then in warp order
  float* gred = L.sc->gred;
  const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(&gate8);
  for (int t = 0; t < T; ++t) {
    float acc = 0.0f;
    if (8 * (int)threadIdx.x < H) {
      const uint4 xr = ld_cg16(a.x + (size_t)t * H + 8 * threadIdx.x);
      const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&xr);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        acc = fmaf(__low2float(xp[h]), __low2float(gp[h]), acc);
        acc = fmaf(__high2float(xp[h]), __high2float(gp[h]), acc);
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) gred[warp * kDecodeRows + t] = acc;
  }
  __syncthreads();
  if (threadIdx.x < T) {
    const int t = threadIdx.x;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kW; ++w) v += gred[w * kDecodeRows + t];
    const float gt = sigmoid_f32(v);
    L.gam[t] = gt;
    if (publish) a.w.gamma[t] = gt;
  }
}

// ---- shared expert gate/up: one [8 gate; 8 up] tile of bf16 rows, full K ----
// 64 KB at H = 2048: it spans stages 0 and 1.
__device__ void issue_shared_tile(const KArgs& a, int tile, uint8_t* stages, uint64_t* bar) {
  const int H = a.d.H, Is = a.d.Is;
  const uint32_t half = 8u * (uint32_t)H * 2u;
  mbar_expect(bar, 2u * half);
  bulk_copy(stages, a.L.ws13 + (size_t)(8 * tile) * H, half, bar);
  bulk_copy(stages + half, a.L.ws13 + (size_t)(Is + 8 * tile) * H, half, bar);
}

// Two warps (wsel 0 and 1) each take half of K; the second hands its partial
// tile to the first through shared memory (named barrier 1, 64 threads).
template <int NT>
__device__ void shared_tile(const KArgs& a, const Layout& L, int tile, const uint8_t* st, int wsel) {
  const int H = a.d.H, Is = a.d.Is, T = a.d.T;
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const size_t row = (size_t)2 * H;
  const bf16* xb[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) xb[nt] = a.x + (size_t)min(8 * nt + g, T - 1) * H;
  float acc[NT][4] = {};
  const int nb = H / 64;  // k32 blocks per warp
#pragma unroll 4
  for (int bi = 0; bi < nb; ++bi) {
    const int off = (wsel * nb + bi) * 32 + 8 * q;  // elements
    const uint4 ag = lds16(st + (size_t)g * row + 2 * off);
    const uint4 au = lds16(st + (size_t)(8 + g) * row + 2 * off);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_bf16_k32(acc[nt], ag, au, ld_cg16(xb[nt] + off));
  }
  float* red = L.red;
  if (wsel == 1)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) red[(nt * 4 + c) * 32 + lane] = acc[nt][c];
  asm volatile("bar.sync 1, 64;\n" ::: "memory");
  if (wsel == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float z[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) z[c] = acc[nt][c] + red[(nt * 4 + c) * 32 + lane];
      const int n = 8 * tile + g;
      const int tok = 8 * nt + 2 * q;
      const bf16 h0 = __float2bfloat16_rn(silu_f32(bf16_round(z[0])) * bf16_round(z[2]));
      const bf16 h1 = __float2bfloat16_rn(silu_f32(bf16_round(z[1])) * bf16_round(z[3]));
      if (tok < T) a.w.hs[(size_t)tok * Is + n] = h0;
      if (tok + 1 < T) a.w.hs[(size_t)(tok + 1) * Is + n] = h1;
    }
  }
}

// ---- routed gate/up tile: [8 gate; 8 up] rows of one expert, full K ---------
__device__ __forceinline__ void unit_coords(const KArgs& a, const Sched* sc, int r, int* e, int* n0,
                                            int* c) {
  const int per = a.d.I / 8;
  *c = r / per;
  *n0 = 8 * (r % per);
  *e = sc->chunk[*c].x;
}

// Four bulk copies: the 8 gate rows, the 8 up rows and their scale rows.
__device__ void issue_routed(const KArgs& a, const Layout& L, int r, int s) {
  const int H = a.d.H, I = a.d.I, nbh = L.nbh;
  int e, n0, c;
  unit_coords(a, L.sc, r, &e, &n0, &c);
  const uint8_t* W = a.L.w13 + (size_t)e * 2 * I * H;
  const float* S = a.L.s13 + (size_t)e * (2 * I / kGroup) * nbh;
  uint8_t* st = L.stages + (size_t)s * L.stage_bytes;
  const uint32_t half = 8u * (uint32_t)H;
  const float *lg, *lu;
  int dg, du;
  const uint32_t bg = scale_span(S + (size_t)(n0 / kGroup) * nbh, nbh, &lg, &dg);
  const uint32_t bu = scale_span(S + (size_t)((I + n0) / kGroup) * nbh, nbh, &lu, &du);
  uint8_t* sdst = st + (size_t)16 * H;
  mbar_expect(&L.bar[s], 2u * half + bg + bu);
  bulk_copy(st, W + (size_t)n0 * H, half, &L.bar[s]);
  bulk_copy(st + half, W + (size_t)(I + n0) * H, half, &L.bar[s]);
  bulk_copy(sdst, lg, bg, &L.bar[s]);
  bulk_copy(sdst + scale_slot(nbh), lu, bu, &L.bar[s]);
}

// One warp computes a whole tile over the full K, so tiles need no
// cross-warp reduction.  The inner loop is branch-free: invalid token columns
// read row 0 (their results are never stored).
template <int NT>
__device__ void routed_unit(const KArgs& a, const Layout& L, int r, int s) {
  const int H = a.d.H, I = a.d.I, k = a.d.k;
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const Sched* sc = L.sc;
  int e, n0, c;
  unit_coords(a, sc, r, &e, &n0, &c);
  const int s0 = sc->chunk[c].y, ntok = sc->chunk[c].z;
  const int nbh = L.nbh;
  const uint8_t* st = L.stages + (size_t)s * L.stage_bytes;
  const float* S = a.L.s13 + (size_t)e * (2 * I / kGroup) * nbh;
  const float* lo;
  int dg, du;
  scale_span(S + (size_t)(n0 / kGroup) * nbh, nbh, &lo, &dg);
  scale_span(S + (size_t)((I + n0) / kGroup) * nbh, nbh, &lo, &du);
  const float* Sg = reinterpret_cast<const float*>(st + (size_t)16 * H) + dg;
  const float* Su = reinterpret_cast<const float*>(st + (size_t)16 * H + scale_slot(nbh)) + du;
  const uint8_t* xb[NT];
  const float* sxc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tb = min(8 * nt + g, ntok - 1);
    xb[nt] = L.xq + (size_t)(sc->pair_of_slot[s0 + tb] / k) * L.xq_stride;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int tc = min(8 * nt + 2 * q + cc, ntok - 1);
      sxc[nt][cc] = L.sx + (size_t)(sc->pair_of_slot[s0 + tc] / k) * nbh;
    }
  }
  float acc[NT][4] = {};
#pragma unroll 4
  for (int b = 0; b < H / 64; ++b) {
    const int kb = b >> 1;  // 64-byte slices, two per 128 block
    const int off = b * 64 + 16 * q;
    const uint4 ag = lds16(st + (size_t)g * H + off);
    const uint4 au = lds16(st + (size_t)(8 + g) * H + off);
    const float sg = Sg[kb], su = Su[kb];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint4 bx = lds16(xb[nt] + off);
      const float s_a = sxc[nt][0][kb], s_b = sxc[nt][1][kb];
      float p[4] = {};
      mma_e4m3_k64(p, ag, au, bx);
      acc[nt][0] = fmaf(p[0], sg * s_a, acc[nt][0]);
      acc[nt][1] = fmaf(p[1], sg * s_b, acc[nt][1]);
      acc[nt][2] = fmaf(p[2], su * s_a, acc[nt][2]);
      acc[nt][3] = fmaf(p[3], su * s_b, acc[nt][3]);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tok = 8 * nt + 2 * q;
    const float h0 = silu_f32(bf16_round(acc[nt][0])) * bf16_round(acc[nt][2]);
    const float h1 = silu_f32(bf16_round(acc[nt][1])) * bf16_round(acc[nt][3]);
    if (tok < ntok) a.w.hbuf[(size_t)(s0 + tok) * I + n0 + g] = h0;
    if (tok + 1 < ntok) a.w.hbuf[(size_t)(s0 + tok + 1) * I + n0 + g] = h1;
  }
}

// ---- schedule (identical in every CTA) --------------------------------------
__device__ void build_schedule(const KArgs& a, const Layout& L, bool publish) {
  Sched* sc = L.sc;
  const int T = a.d.T, k = a.d.k, E = a.d.E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (T == 1 && E <= 32 * kW && k <= 32) {
    topk_one_row<kW>(L.lg, E, k, sc->cand_key, sc->cand_id, sc->idx, sc->w);
    // one row: its k experts are distinct, so slot = rank of the expert among them
    if (warp == 0) {
      __syncwarp();
      if (lane < k) {
        const int e = sc->idx[lane];
        int r = 0;
        for (int j = 0; j < k; ++j) r += sc->idx[j] < e;
        sc->chunk[r] = make_int4(e, r, 1, 0);
        sc->pair_of_slot[r] = lane;
        sc->slot_of_pair[lane] = r;
      }
      if (lane == 0) sc->n_used = k;
    }
    __syncthreads();
    if (publish) {
      if (threadIdx.x < k) {
        a.w.idx[threadIdx.x] = sc->idx[threadIdx.x];
        a.w.wts[threadIdx.x] = sc->w[threadIdx.x];
        a.w.slot_of_pair[threadIdx.x] = sc->slot_of_pair[threadIdx.x];
        a.w.pair_of_slot[threadIdx.x] = sc->pair_of_slot[threadIdx.x];
        a.w.chunks[threadIdx.x] = sc->chunk[threadIdx.x];
      }
      if (threadIdx.x == 0) *a.w.n_chunks = k;
    }
    return;
  }
  for (int t = warp; t < T; t += kW) topk_row(L.lg + (size_t)t * E, E, k, sc->idx + t * k, sc->w + t * k);
  for (int e = threadIdx.x; e < kMaxExperts; e += kThreads) sc->tok[e] = 0u;
  __syncthreads();
  for (int p = threadIdx.x; p < T * k; p += kThreads) atomicOr(&sc->tok[sc->idx[p]], 1u << (p / k));
  __syncthreads();
  const int e = threadIdx.x;
  const uint32_t mask = e < E ? sc->tok[e] : 0u;
  const int cnt = __popc(mask);
  int n_slots, n_used;
  const int slot0 = exscan(cnt, &n_slots, sc->scan);
  const int u = exscan(cnt > 0 ? 1 : 0, &n_used, sc->scan);
  if (cnt > 0) {
    sc->chunk[u] = make_int4(e, slot0, cnt, 0);
    uint32_t m = mask;
    for (int r = 0; m; ++r) {
      const int t = __ffs(m) - 1;
      m &= m - 1;
      int j = 0;
      while (sc->idx[t * k + j] != e) ++j;
      const int p = t * k + j, slot = slot0 + r;
      sc->pair_of_slot[slot] = p;
      sc->slot_of_pair[p] = slot;
    }
  }
  if (threadIdx.x == 0) sc->n_used = n_used;
  __syncthreads();
  if (publish) {
    for (int p = threadIdx.x; p < T * k; p += kThreads) {
      a.w.idx[p] = sc->idx[p];
      a.w.wts[p] = sc->w[p];
      a.w.slot_of_pair[p] = sc->slot_of_pair[p];
      a.w.pair_of_slot[p] = sc->pair_of_slot[p];
    }
    for (int c = threadIdx.x; c < n_used; c += kThreads) a.w.chunks[c] = sc->chunk[c];
    if (threadIdx.x == 0) *a.w.n_chunks = n_used;
  }
}

// ---- phase C pieces ---------------------------------------------------------
// Bulk copies of the down slices (16 rows x I and the scale row) of the
// schedule's experts [e0, e0 + n) into the slots, issued by one warp: every
// lane first announces its bytes, then one arrival closes the phase's count,
// then the lanes issue their copies in parallel.
__device__ void issue_down_round(const KArgs& a, const Sched* sc, const CLayout& cl, uint8_t* area,
                                 int m0, int e0, int n, uint64_t* bar) {
  const int H = a.d.H, I = a.d.I, nbi = I / kGroup;
  const int lane = threadIdx.x & 31;
  for (int i = lane; i < n; i += 32) {
    const float* lo;
    int d;
    const uint32_t bs =
        scale_span(a.L.s2 + ((size_t)sc->chunk[e0 + i].x * (H / kGroup) + m0 / kGroup) * nbi, nbi, &lo, &d);
    mbar_expect_only(bar, 16u * I + bs);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  for (int i = lane; i < n; i += 32) {
    const int e = sc->chunk[e0 + i].x;
    uint8_t* slot = area + (size_t)i * cl.slot_bytes;
    bulk_copy(slot, a.L.w2 + (size_t)e * H * I + (size_t)m0 * I, 16u * I, bar);
    const float* lo;
    int d;
    const uint32_t bs = scale_span(a.L.s2 + ((size_t)e * (H / kGroup) + m0 / kGroup) * nbi, nbi, &lo, &d);
    bulk_copy(slot + (size_t)16 * I, lo, bs, bar);
  }
}

__device__ void issue_shared_down(const KArgs& a, const CLayout& cl, uint8_t* area, int m0,
                                  uint64_t* bar) {
  const int Is = a.d.Is;
  mbar_expect(bar, 16u * Is * 2u);
  bulk_copy(area + cl.ws2, a.L.ws2 + (size_t)m0 * Is, 16u * Is * 2u, bar);
}

// One selected expert's 16 x I down slice (in slot slot_i) against its rows' codes.
template <int NT>
__device__ void down_item(const KArgs& a, const Sched* sc, const CLayout& cl, uint8_t* area, int m0,
                          int item, int slot_i) {
  const int H = a.d.H, I = a.d.I, nbi = I / kGroup;
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int4 ch = sc->chunk[item];
  const int s0 = ch.y, ntok = ch.z;
  const uint8_t* slot = area + (size_t)slot_i * cl.slot_bytes;
  const float* lo;
  int d;
  scale_span(a.L.s2 + ((size_t)ch.x * (H / kGroup) + m0 / kGroup) * nbi, nbi, &lo, &d);
  const float* S = reinterpret_cast<const float*>(slot + (size_t)16 * I) + d;
  const uint8_t* hq = area + cl.hq;
  const float* sh = reinterpret_cast<const float*>(area + cl.sh);
  float* s_d = reinterpret_cast<float*>(area + cl.d);
  const uint8_t* hb[NT];
  const float* shc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    hb[nt] = hq + (size_t)(s0 + min(8 * nt + g, ntok - 1)) * cl.hq_stride;
#pragma unroll
    for (int c = 0; c < 2; ++c) shc[nt][c] = sh + (size_t)(s0 + min(8 * nt + 2 * q + c, ntok - 1)) * nbi;
  }
  float acc[NT][4] = {};
#pragma unroll 4
  for (int bb = 0; bb < I / 64; ++bb) {
    const int kb = (bb * 64) / kGroup;
    const int off = bb * 64 + 16 * q;
    const uint4 a0 = lds16(slot + (size_t)g * I + off);
    const uint4 a1 = lds16(slot + (size_t)(8 + g) * I + off);
    const float sw = S[kb];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint4 bx = lds16(hb[nt] + off);
      const float s_a = shc[nt][0][kb], s_b = shc[nt][1][kb];
      float p[4] = {};
      mma_e4m3_k64(p, a0, a1, bx);
      acc[nt][0] = fmaf(p[0], sw * s_a, acc[nt][0]);
      acc[nt][1] = fmaf(p[1], sw * s_b, acc[nt][1]);
      acc[nt][2] = fmaf(p[2], sw * s_a, acc[nt][2]);
      acc[nt][3] = fmaf(p[3], sw * s_b, acc[nt][3]);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int tok = 8 * nt + 2 * q + (c & 1);
      if (tok < ntok) s_d[(s0 + tok) * 16 + g + 8 * (c >> 1)] = bf16_round(acc[nt][c]);
    }
}

// One K half of the shared expert's 16 x Is down slice; fp32 partial sums.
template <int NT>
__device__ void shared_down_item(const KArgs& a, const CLayout& cl, uint8_t* area, int half) {
  const int T = a.d.T, Is = a.d.Is;
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const uint8_t* ws = area + cl.ws2;
  const int kh = Is / 2;
  const uint8_t* hs = area + cl.hs;
  float* s_ds = reinterpret_cast<float*>(area + cl.ds);
  const uint8_t* hb[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) hb[nt] = hs + (size_t)min(8 * nt + g, T - 1) * cl.hs_stride;
  float acc[NT][4] = {};
#pragma unroll 4
  for (int bb = 0; bb < kh / 32; ++bb) {
    const int off = half * kh + bb * 32 + 8 * q;  // elements
    const uint4 a0 = lds16(ws + (size_t)g * Is * 2 + 2 * off);
    const uint4 a1 = lds16(ws + (size_t)(8 + g) * Is * 2 + 2 * off);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_bf16_k32(acc[nt], a0, a1, lds16(hb[nt] + 2 * off));
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int tok = 8 * nt + 2 * q + (c & 1);
      if (tok < T) s_ds[(half * kDecodeRows + tok) * 16 + g + 8 * (c >> 1)] = acc[nt][c];
    }
}

// Re-quantised SwiGLU rows (from hbuf) and the shared SwiGLU rows, the same
// in every CTA.
__device__ void phase_c_inputs(const KArgs& a, const CLayout& cl, uint8_t* area, bool publish) {
  const int T = a.d.T, k = a.d.k, I = a.d.I, Is = a.d.Is;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nbi = I / kGroup, P = T * k;
  uint8_t* hq = area + cl.hq;
  float* sh = reinterpret_cast<float*>(area + cl.sh);
  // the shared SwiGLU rows: issue their loads first (up to 4 per thread)
  uint8_t* hs = area + cl.hs;
  const int n_hs = T * (Is / 8);
  uint4 hsv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = threadIdx.x + u * kThreads;
    if (i < n_hs) hsv[u] = ld_cg16(a.w.hs + (size_t)(i / (Is / 8)) * Is + 8 * (i % (Is / 8)));
  }
  constexpr int kIlp = 4;  // (slot, group) pairs a warp works on together
  for (int base = warp * kIlp; base < P * nbi; base += kW * kIlp) {
    float4 v[kIlp];
#pragma unroll
    for (int u = 0; u < kIlp; ++u) {
      const int pg = base + u;
      v[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (pg < P * nbi)
        v[u] = __ldcg(reinterpret_cast<const float4*>(a.w.hbuf + (size_t)(pg / nbi) * I +
                                                      (pg % nbi) * kGroup + 4 * lane));
    }
    float m[kIlp];
#pragma unroll
    for (int u = 0; u < kIlp; ++u)
      m[u] = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < kIlp; ++u) m[u] = fmaxf(m[u], __shfl_xor_sync(0xffffffffu, m[u], o));
#pragma unroll
    for (int u = 0; u < kIlp; ++u) {
      const int pg = base + u;
      if (pg >= P * nbi) break;
      const int slot = pg / nbi, grp = pg % nbi;
      const float s = group_scale(m[u]);
      const uint32_t packed = quant4(v[u].x, v[u].y, v[u].z, v[u].w, s);
      *reinterpret_cast<uint32_t*>(hq + (size_t)slot * cl.hq_stride + grp * kGroup + 4 * lane) = packed;
      if (lane == 0) sh[(size_t)slot * nbi + grp] = s;
      if (publish) {
        *reinterpret_cast<uint32_t*>(a.w.hq + (size_t)slot * I + grp * kGroup + 4 * lane) = packed;
        if (lane == 0) a.w.sh[(size_t)slot * nbi + grp] = s;
      }
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = threadIdx.x + u * kThreads;
    if (i < n_hs)
      *reinterpret_cast<uint4*>(hs + (size_t)(i / (Is / 8)) * cl.hs_stride + 2 * 8 * (i % (Is / 8))) = hsv[u];
  }
  for (int i = threadIdx.x + 4 * kThreads; i < n_hs; i += kThreads) {
    const int t = i / (Is / 8), o = 8 * (i % (Is / 8));
    *reinterpret_cast<uint4*>(hs + (size_t)t * cl.hs_stride + 2 * o) = ld_cg16(a.w.hs + (size_t)t * Is + o);
  }
}

}  // namespace

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) k_decode_layer(KArgs a, int n_stages) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int G = gridDim.x, b = blockIdx.x;
  const int T = a.d.T, H = a.d.H, E = a.d.E, k = a.d.k, I = a.d.I, Is = a.d.Is;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const Layout L = layout(smem, T, H, E, n_stages);
  Sched* sc = L.sc;
  int* bar2 = a.w.done + 2;
  int* bar_exit = a.w.done + 3;
  int* epoch = a.w.done + 4;
  const int n_sh = Is / 8;  // shared gate/up tiles
  uint64_t* bar_c = &L.bar[kMaxStages];      // phase C down slices
  uint64_t* bar_s = &L.bar[kMaxStages + 1];  // phase C shared slice

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages + 2; ++s) mbar_init(&L.bar[s]);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  // ---- phase A: immutable weights first ------------------------------------
  const bool has_shared = b < n_sh;
  const int sh_stage = n_stages - 2;  // the shared tile spans the last two stages
  if (threadIdx.x == 0 && has_shared)
    issue_shared_tile(a, b, L.stages + (size_t)sh_stage * L.stage_bytes, &L.bar[sh_stage]);
  if (threadIdx.x == 32)
    for (int mt = b; mt < H / 16; mt += G) prefetch_l2(a.L.ws2 + (size_t)mt * 16 * Is, 16u * Is * 2);
  // router rows: experts b and b + G; each warp covers an eighth of K of both
  const int keighth = H / 8;
  const int k0 = warp * keighth;
  constexpr int kMaxV = 2;  // float4 per lane per expert: H up to 2048
  const int nv = (keighth + 127) / 128;
  float4 wv[2][kMaxV];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int er = b + G * h;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
      wv[h][i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (er < E && i < nv && 128 * i + 4 * lane < keighth)
        wv[h][i] = __ldg(reinterpret_cast<const float4*>(a.L.wr + (size_t)er * H + k0 + 128 * i +
                                                         4 * lane));
    }
  }
  const uint4 gate8 = 8 * (int)threadIdx.x < H
                          ? __ldg(reinterpret_cast<const uint4*>(a.L.gate + 8 * threadIdx.x))
                          : make_uint4(0u, 0u, 0u, 0u);
  // When every 128-group lies inside one warp's eighth of K (H >= 1024), the
  // router pass also quantises x and takes the gate dot product from the same
  // registers: the lane holds 4 consecutive inputs of a group per slice.
  const bool fuse_q = keighth % kGroup == 0;
  uint2 gw[kMaxV];
#pragma unroll
  for (int i = 0; i < kMaxV; ++i)
    gw[i] = (fuse_q && i < nv && 128 * i + 4 * lane < keighth)
                ? __ldg(reinterpret_cast<const uint2*>(a.L.gate + k0 + 128 * i + 4 * lane))
                : make_uint2(0u, 0u);
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) sc->tag = ld_acquire(epoch) + 1;
  __syncthreads();
  const unsigned long long tag = (unsigned long long)(unsigned)sc->tag << 32;
  float* red = L.red;  // [2][kW][kDecodeRows]
  for (int t0 = 0; t0 < T; t0 += 4) {  // rows in groups of four
    float acc[2][4], gacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int t = 0; t < 4; ++t) acc[h][t] = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
      if (i >= nv || 128 * i + 4 * lane >= keighth) continue;
      const int kk = k0 + 128 * i + 4 * lane;
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        const int t = t0 + tt;
        if (t >= T) break;
        const uint2 raw = __ldcg(reinterpret_cast<const uint2*>(a.x + (size_t)t * H + kk));
        const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
        const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
        const float x0 = __low2float(p0), x1 = __high2float(p0), x2 = __low2float(p1),
                    x3 = __high2float(p1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float s = acc[h][tt];
          s = fmaf(x0, wv[h][i].x, s);
          s = fmaf(x1, wv[h][i].y, s);
          s = fmaf(x2, wv[h][i].z, s);
          s = fmaf(x3, wv[h][i].w, s);
          acc[h][tt] = s;
        }
        if (fuse_q) {
          float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
          m = warp_max(m);
          const float sc_ = group_scale(m);
          const uint32_t packed = quant4(x0, x1, x2, x3, sc_);
          *reinterpret_cast<uint32_t*>(L.xq + (size_t)t * L.xq_stride + kk) = packed;
          if (lane == 0) L.sx[t * L.nbh + kk / kGroup] = sc_;
          if (b == 0) {
            *reinterpret_cast<uint32_t*>(a.w.xq + (size_t)t * H + kk) = packed;
            if (lane == 0) a.w.sx[(size_t)t * L.nbh + kk / kGroup] = sc_;
          }
          const __nv_bfloat162 g0 = *reinterpret_cast<const __nv_bfloat162*>(&gw[i].x);
          const __nv_bfloat162 g1 = *reinterpret_cast<const __nv_bfloat162*>(&gw[i].y);
          float gs = gacc[tt];
          gs = fmaf(x0, __low2float(g0), gs);
          gs = fmaf(x1, __high2float(g0), gs);
          gs = fmaf(x2, __low2float(g1), gs);
          gs = fmaf(x3, __high2float(g1), gs);
          gacc[tt] = gs;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        if (t0 + tt >= T) break;
        const float v = warp_sum(acc[h][tt]);
        if (lane == 0) red[(h * kW + warp) * kDecodeRows + t0 + tt] = v;
      }
    if (fuse_q)
#pragma unroll
      for (int tt = 0; tt < 4; ++tt) {
        if (t0 + tt >= T) break;
        const float v = warp_sum(gacc[tt]);
        if (lane == 0) sc->gred[warp * kDecodeRows + t0 + tt] = v;
      }
  }
  __syncthreads();
  if (threadIdx.x < 2 * T) {
    const int h = threadIdx.x / T, t = threadIdx.x % T;
    const int ee = b + G * h;
    if (ee < E) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kW; ++w) v += red[(h * kW + w) * kDecodeRows + t];
      st_relaxed64(a.w.tlog + (size_t)t * E + ee, tag | __float_as_uint(v));
    }
  }
  __syncthreads();

  // ---- phase B: quantise x, gather logits, schedule, routed gate/up ---------
  if (fuse_q) {
    if (threadIdx.x < T) {
      const int t = threadIdx.x;
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kW; ++w) v += sc->gred[w * kDecodeRows + t];
      const float gt = sigmoid_f32(v);
      L.gam[t] = gt;
      if (b == 0) a.w.gamma[t] = gt;
    }
  } else {
    quant_rows_local(a, L, b == 0, gate8);
  }
  for (int i = threadIdx.x; i < T * E; i += kThreads) {
    long long it = 0;
    unsigned long long v = ld_relaxed64(a.w.tlog + i);
    while ((v & 0xFFFFFFFF00000000ull) != tag) {
      if (++it > kSpinLimit) {
        atomicExch(a.w.status, 1);
        break;
      }
      if (it > 16) __nanosleep(32);
      v = ld_relaxed64(a.w.tlog + i);
    }
    L.lg[i] = __uint_as_float((uint32_t)v);
  }
  __syncthreads();
  build_schedule(a, L, b == 0);
  const int U = sc->n_used;
  const int n_routed = U * (I / 8);
  const int my_units = b < n_routed ? (n_routed - b + G - 1) / G : 0;
  // Unit i of this CTA is tile b + G*i.  Warp w < n_stages owns stage w and
  // takes units w, w + n_stages, ...; a shared tile first occupies the last
  // two stages and is computed by their two warps.
  const bool sh_warp = has_shared && warp >= sh_stage && warp < n_stages;
  if (lane == 0 && warp < n_stages && warp < my_units && !sh_warp)
    issue_routed(a, L, b + G * warp, warp);
  if (warp == kW - 1) {
    const size_t per = (size_t)H * I;
    if ((size_t)U * per <= kDownPrefetchBytes)
      for (int mt = b; mt < H / 16; mt += G)
        for (int c = lane; c < U; c += 32)
          prefetch_l2(a.L.w2 + (size_t)sc->chunk[c].x * per + (size_t)mt * 16 * I, 16u * I);
  }
  if (warp < n_stages) {
    uint32_t par = 0;  // parity of this warp's stage barrier
    if (sh_warp) {
      stage_wait(&L.bar[sh_stage], 0, a.w.status);
      if (warp == sh_stage) par ^= 1u;
      shared_tile<NT>(a, L, b, L.stages + (size_t)sh_stage * L.stage_bytes, warp - sh_stage);
      asm volatile("bar.sync 1, 64;\n" ::: "memory");  // both warps done with the tile
      if (lane == 0 && warp < my_units) issue_routed(a, L, b + G * warp, warp);
    }
    for (int i = warp; i < my_units; i += n_stages) {
      stage_wait(&L.bar[warp], par, a.w.status);
      par ^= 1u;
      routed_unit<NT>(a, L, b + G * i, warp);
      __syncwarp();
      if (lane == 0 && i + n_stages < my_units) issue_routed(a, L, b + G * (i + n_stages), warp);
    }
  }
  __syncthreads();
  // copy phase C's weights (warmed in L2) into the now idle stages
  uint8_t* area = L.stages;
  const CLayout cl = c_layout(T, k, I, Is, U, (size_t)n_stages * L.stage_bytes);
  const int mt0 = b;
  if (mt0 < H / 16) {
    if (threadIdx.x == 32) issue_shared_down(a, cl, area, 16 * mt0, bar_s);
    if (warp == 0 && U > 0) issue_down_round(a, sc, cl, area, 16 * mt0, 0, cl.R, bar_c);
  }
  grid_arrive(bar2);
  grid_wait(bar2, G, a.w.status);

  // ---- phase C: re-quantise, down projections, combine ----------------------
  uint32_t pc = 0, ps = 0;  // parities of the phase C barriers
  for (int mt = mt0; mt < H / 16; mt += G) {
    const int m0 = 16 * mt;
    if (mt != mt0) {
      if (threadIdx.x == 32) issue_shared_down(a, cl, area, m0, bar_s);
      if (warp == 0 && U > 0) issue_down_round(a, sc, cl, area, m0, 0, cl.R, bar_c);
    }
    phase_c_inputs(a, cl, area, b == 0 && mt == mt0);
    __syncthreads();
    stage_wait(bar_s, ps, a.w.status);
    ps ^= 1u;
    if (U == 0) {
      if (warp < 2) shared_down_item<NT>(a, cl, area, warp);
      __syncthreads();
    }
    for (int e0 = 0; e0 < U; e0 += cl.R) {
      const int n = U - e0 < cl.R ? U - e0 : cl.R;
      stage_wait(bar_c, pc, a.w.status);
      pc ^= 1u;
      // items: this round's experts, then (first round) the two shared halves
      const int n_items = n + (e0 == 0 ? 2 : 0);
      for (int it = warp; it < n_items; it += kW) {
        if (it < n)
          down_item<NT>(a, sc, cl, area, m0, e0 + it, it);
        else
          shared_down_item<NT>(a, cl, area, it - n);
      }
      __syncthreads();
      if (e0 + cl.R < U && warp == 0) {
        const int n2 = U - e0 - cl.R < cl.R ? U - e0 - cl.R : cl.R;
        issue_down_round(a, sc, cl, area, m0, e0 + cl.R, n2, bar_c);
      }
    }
    const float* s_d = reinterpret_cast<const float*>(area + cl.d);
    const float* s_ds = reinterpret_cast<const float*>(area + cl.ds);
    for (int i = threadIdx.x; i < T * 16; i += kThreads) {
      const int t = i >> 4, r = i & 15;
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) acc = fmaf(sc->w[t * k + j], s_d[sc->slot_of_pair[t * k + j] * 16 + r], acc);
      const float ds = bf16_round(s_ds[t * 16 + r] + s_ds[(kDecodeRows + t) * 16 + r]);
      a.y[(size_t)t * H + m0 + r] = __float2bfloat16_rn(fmaf(L.gam[t], ds, acc));
    }
    __syncthreads();
  }

  // ---- exit: the last CTA resets the barrier and advances the launch tag ----
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(bar_exit, 1);
    if (old == G - 1) {
      *bar2 = 0;
      *bar_exit = 0;
      *epoch = sc->tag;
      __threadfence();
    }
  }
}

size_t decode_layer_smem(int T, int H, int E, int n_stages) {
  return (size_t)n_stages * stage_bytes_for(H) + smem_after_stages(T, H, E);
}

// Stages that fit a shared-memory budget for T rows (0 if fewer than two).
int decode_layer_stages(int T, int H, int E, size_t budget) {
  const size_t fixed = smem_after_stages(T, H, E);
  if (budget <= fixed) return 0;
  int n = (int)((budget - fixed) / stage_bytes_for(H));
  if (n > kMaxStages) n = kMaxStages;
  return n >= 2 ? n : 0;
}

// Whether T rows fit: the shared tile (16 bf16 rows) in two stages, and
// phase C at least one down slot beside its inputs.
bool decode_layer_fits(int T, int H, int E, int k, int I, int Is, int n_stages) {
  if (n_stages < 2 || T * k > kDecodeRows * kMaxTopK || T > kDecodeRows) return false;
  if ((size_t)2 * stage_bytes_for(H) < (size_t)16 * H * 2) return false;
  const size_t area = (size_t)n_stages * stage_bytes_for(H);
  const int U = T * k < E ? T * k : E;
  const CLayout c = c_layout(T, k, I, Is, U, area);
  return c.R >= 1 && c.end <= area;
}

cudaError_t setup_decode_layer(size_t max_smem) {
  cudaError_t e = cudaFuncSetAttribute(k_decode_layer<1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_decode_layer<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)max_smem);
}

const void* decode_layer_kernel() { return reinterpret_cast<const void*>(k_decode_layer<2>); }

// One 8-column MMA tile covers up to 8 rows; two cover up to 16.
cudaError_t launch_decode_layer(const KArgs& a, int grid, int n_stages, size_t smem, bool pdl,
                                cudaStream_t s) {
  if (a.d.T <= 8)
    return launch_pdl(k_decode_layer<1>, dim3(grid), dim3(kThreads), smem, s, pdl, a, n_stages);
  return launch_pdl(k_decode_layer<2>, dim3(grid), dim3(kThreads), smem, s, pdl, a, n_stages);
}

}  // namespace moe

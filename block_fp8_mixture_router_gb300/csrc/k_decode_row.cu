// One-row decode layer (T = 1) as one kernel over every SM, split by role.
//
//   routed CTA (r, p), r < k, p < P = H/128: SwiGLU features [p*F, p*F + F)
//      of the rank-r expert (F = I/P; its 2F gate/up rows are four or fewer
//      16 KB bulk copies) and rows [128p, 128p + 128) of that expert's down
//      projection (one contiguous 128 x I copy);
//   shared gate/up CTA s < P: shared SwiGLU features [s*Fs, s*Fs + Fs);
//   shared down CTA (the rest): a block of the shared expert's output rows.
//
// Every CTA quantises x and takes the shared gate's dot product in one
// register pass; the routed CTAs also compute the router logits (experts 2b
// and 2b + 1) in it.  Results
// move between CTAs as 64-bit {launch tag, value} words in global memory,
// each written once per launch and polled until its tag is current:
//   logits            every CTA computes the same top-k;
//   routed SwiGLU h   the CTAs of one expert each read all I values and
//                     quantise them the same way (1 x 128 groups);
//   shared SwiGLU hs  the shared down CTAs read all Is values;
//   down outputs      routed CTA (r, p) combines 128/k of its block's rows:
//                     y = sum_j w_j d_j (rank order) + gamma * ds, bf16.
// There is no grid barrier.  Weights that do not depend on x (router rows,
// the shared expert) are requested before the kernel waits on its
// predecessor (programmatic dependent launch); a routed CTA issues all its
// copies as soon as the top-k is known.
//
// Router and top-k: PR #939 "Fish Audio Drama 3 text to speech on one CUDA
// GPU", sections "What it adds" and "Fidelity against the PyTorch oracle"
// (the lower index wins a tie).  Expert arithmetic: PR #939 section
// "Precision" (e4m3 inputs per row and per 128 inputs, amax/448).  SwiGLU
// storage: commit "one SwiGLU launch for the routed and shared experts".
// Combine order: commit "MoE combine on 8-wide vectors".  Launch chaining:
// PR #927, section "What this changes".
//
// Every wait is bounded: a poll or copy wait that does not complete within
// the spin limit sets the context's status flag and the kernel runs to its
// end without waiting further (its output is then undefined, and the host
// reports MOE_ERR_DEVICE_TIMEOUT).
#include <math.h>

#include "decode_common.cuh"

namespace moe {

namespace {

using namespace dec;

constexpr int kW = 16;  // warps per CTA: more warps hide more of each phase's latency
constexpr int kThreads = 32 * kW;
constexpr int kSguSlots = 3;      // ring slots of a shared gate/up CTA (one unit each)
constexpr int kSdnSlots = 6;      // ring slots of a shared down CTA
constexpr int kSdnUnit = 32;      // shared down rows per copy
constexpr int kMaxRowH = 2048;    // router rows live in registers: H <= 2048

// ---- roles ----------------------------------------------------------------
struct Roles {
  int P;    // 128-row output blocks
  int nR;   // routed CTAs (k * P)
  int nS1;  // shared gate/up CTAs (P)
  int nS2;  // shared down CTAs
  int F;    // routed SwiGLU features per CTA (I / P)
  int Fs;   // shared SwiGLU features per CTA (Is / P)
  int R2;   // shared down rows per CTA (multiple of kSdnUnit)
};

__host__ __device__ inline Roles make_roles(int G, int H, int k, int I, int Is) {
  Roles r;
  r.P = H / kGroup;
  r.nR = k * r.P;
  r.nS1 = r.P;
  r.nS2 = G - r.nR - r.nS1;
  r.F = I / r.P;
  r.Fs = Is / r.P;
  r.R2 = r.nS2 > 0 ? ((H + r.nS2 - 1) / r.nS2 + kSdnUnit - 1) / kSdnUnit * kSdnUnit : 0;
  return r;
}

// Routed weight rows sit in shared memory 16 bytes apart from a multiple of
// 128: the eight rows an MMA fragment reads at once then fall in different
// banks (a row per bulk copy).
constexpr int kRowPad = 16;

// Bytes of weights a role keeps in shared memory at once.
__host__ __device__ inline size_t data_bytes(const Roles& r, int H, int I, int Is) {
  const size_t routed = (size_t)2 * r.F * (H + kRowPad) + (size_t)kGroup * (I + kRowPad);
  const size_t sgu = (size_t)kSguSlots * 16 * H * 2;
  const size_t sdn = (size_t)kSdnSlots * kSdnUnit * Is * 2;
  size_t m = routed > sgu ? routed : sgu;
  return al16(m > sdn ? m : sdn);
}

// Shared memory after the weights.
struct Small {
  int idx[kMaxTopK];
  float w[kMaxTopK];
  int slot[kMaxTopK];
  uint32_t cand_key[2 * kW * kMaxTopK];
  uint32_t cand_id[2 * kW * kMaxTopK];
  float gred[kW];
  float gmax[kW];  // one scale per row: each warp's amax
  float gss[kW];   // add-norm: each warp's sum of squares
  float gamma;
  int tag;
  float comb[kMaxTopK + 1][16];  // down outputs gathered for the combine
};

struct Lay {
  uint8_t* data;
  uint8_t* xq;    // [H] e4m3 codes of x
  bf16* xs;       // [H] x
  float* sx;      // [H/128]
  float* wsc;     // routed: gate scale row, up scale row, down scales (widened)
  float* hall;    // [max(I, Is)] exchanged SwiGLU values
  uint8_t* hq;    // [I] their e4m3 codes (routed)
  float* sh;      // [I/128] their scales
  float* red;     // [kW][32][2] scratch
  float* lg;      // [E]
  uint64_t* bar;  // [8]
  Small* sm;
};

__host__ __device__ inline size_t small_bytes(int H, int E, int I, int Is) {
  const int nbh = H / kGroup;
  const int M = I > Is ? I : Is;
  return al16(H) + al16((size_t)H * 2) + al16((size_t)nbh * 4) + 3 * al16((size_t)(nbh + 8) * 4) +
         al16((size_t)M * 4) + al16(I) + al16((size_t)(I / kGroup) * 4) +
         (size_t)kW * 32 * 2 * 4 + al16((size_t)E * 4) + 8 * 8 + al16(sizeof(Small));
}

__device__ inline Lay make_lay(uint8_t* smem, const Roles& r, int H, int E, int I, int Is) {
  const int nbh = H / kGroup;
  const int M = I > Is ? I : Is;
  Lay L;
  uint8_t* p = smem;
  L.data = p;
  p += data_bytes(r, H, I, Is);
  L.xq = p;
  p += al16(H);
  L.xs = reinterpret_cast<bf16*>(p);
  p += al16((size_t)H * 2);
  L.sx = reinterpret_cast<float*>(p);
  p += al16((size_t)nbh * 4);
  L.wsc = reinterpret_cast<float*>(p);
  p += 3 * al16((size_t)(nbh + 8) * 4);
  L.hall = reinterpret_cast<float*>(p);
  p += al16((size_t)M * 4);
  L.hq = p;
  p += al16(I);
  L.sh = reinterpret_cast<float*>(p);
  p += al16((size_t)(I / kGroup) * 4);
  L.red = reinterpret_cast<float*>(p);
  p += (size_t)kW * 32 * 2 * 4;
  L.lg = reinterpret_cast<float*>(p);
  p += al16((size_t)E * 4);
  L.bar = reinterpret_cast<uint64_t*>(p);
  p += 8 * 8;
  L.sm = reinterpret_cast<Small*>(p);
  return L;
}

// Exchange words in the workspace (tagged 64-bit): [k][I] routed h, [k][H]
// routed down outputs, [Is] shared hs, [H] shared down outputs.
struct Xw {
  unsigned long long *h, *d, *hs, *ds;
};

__device__ inline Xw xw_of(unsigned long long* base, int k, int H, int I, int Is) {
  Xw x;
  x.h = base;
  x.d = x.h + (size_t)k * I;
  x.hs = x.d + (size_t)k * H;
  x.ds = x.hs + Is;
  return x;
}

// ---- routed gate/up: [8 gate; 8 up] rows of one expert, a part of K --------
// Lane (g, q) of the m16n8k32 MMAs: rows g (gate) and 8+g (up); the token
// operand is the single quantised row (all eight columns see it; column 0 is
// kept).  Partial products are scaled per 64-byte K slice by the weight
// block scale and the activation group scale.
__device__ __forceinline__ void routed_part(const uint8_t* rows, int ld, const float* sg,
                                            const float* su, const uint8_t* xq, const float* sx,
                                            int b0, int b1, float (&acc)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll 4
  for (int b = b0; b < b1; ++b) {  // 64-byte slices of K
    const int kb = b >> 1;
    const int off = b * 64 + 16 * q;
    const uint4 ag = lds16(rows + (size_t)g * ld + off);
    const uint4 au = lds16(rows + (size_t)(8 + g) * ld + off);
    const uint4 bx = lds16(xq + off);
    float p[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    mma_e4m3_k64(p, ag, au, bx);
    const float s = sx[kb];
    acc[0] = fmaf(p[0], sg[kb] * s, acc[0]);
    acc[2] = fmaf(p[2], su[kb] * s, acc[2]);
  }
}

// bf16 analogue over 32-element slices (shared expert; unscaled).
__device__ __forceinline__ void shared_part(const uint8_t* rows, int H, const bf16* xs, int b0,
                                            int b1, float (&acc)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const size_t row = (size_t)2 * H;
#pragma unroll 4
  for (int b = b0; b < b1; ++b) {
    const int off = b * 32 + 8 * q;  // elements
    const uint4 ag = lds16(rows + (size_t)g * row + 2 * off);
    const uint4 au = lds16(rows + (size_t)(8 + g) * row + 2 * off);
    const uint4 bx = lds16(xs + off);
    mma_bf16_k32(acc, ag, au, bx);
  }
}

// kChain = 0: one layer.  kChain = 1: the layers of a.chain in order, one row
// passed through them (layer l's x is layer l-1's y, read once a counter of
// the routed CTAs' finished combines says it is complete); every CTA keeps
// its role for every layer, and the shared CTAs start streaming layer l+1's
// weights as soon as they finish layer l.
// Order this thread's earlier shared-memory accesses before bulk copies
// that reuse the same bytes.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

template <int kChain>
__global__ void __launch_bounds__(kThreads, 1) k_decode_row(KArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int G = gridDim.x, b = blockIdx.x;
  const int H = a.d.H, E = a.d.E, k = a.d.k, I = a.d.I, Is = a.d.Is;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int nbh = H / kGroup, nbi = I / kGroup;
  const Roles R = make_roles(G, H, k, I, Is);
  const Lay L = make_lay(smem, R, H, E, I, Is);
  Small* sm = L.sm;
  const int* epoch = a.w.done + 4;
  int* status = a.w.status;
  int* ycount = a.w.done + 6;  // chain: routed combines done in this launch
  const Xw X = xw_of(a.w.xw, k, H, I, Is);
  const bool is_routed = b < R.nR;
  const bool is_sgu = !is_routed && b < R.nR + R.nS1;
  const bool is_sdn = !is_routed && !is_sgu;
  const int s1 = b - R.nR, s2 = b - R.nR - R.nS1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(&L.bar[i]);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  const uint32_t sgu_unit = 16u * (uint32_t)H * 2u;  // [8 gate; 8 up] bf16 rows
  const uint32_t sdn_unit = (uint32_t)kSdnUnit * (uint32_t)Is * 2u;
  const int sdn_m0 = is_sdn ? s2 * R.R2 : 0;
  const int sdn_rows = is_sdn ? max(0, min(R.R2, H - sdn_m0)) : 0;
  const int n_sdn_units = sdn_rows / kSdnUnit;
  const int n_sgu_units = R.Fs / 8;
  const int n_layers = kChain ? a.chain.n : 1;
  int base_tag = 0;     // thread 0: the first layer's launch tag
  int layer_tag = 0;    // every thread: the tag of the layer last computed
  for (int l = 0; l < n_layers; ++l) {
  // this layer's weights; the routed CTA's barriers complete once per layer
  const DevLayer LW = kChain ? a.chain.layers[l] : a.L;
  const uint32_t lp = (uint32_t)(l & 1);

  // ---- before the wait: the shared expert's weights and the router rows ----
  // (later layers: right after the previous layer, whose ring reads are done)
  if (threadIdx.x == 0) {
    if (l > 0) fence_proxy_async();
    if (is_sgu) {
      for (int u = 0; u < n_sgu_units && u < kSguSlots; ++u) {
        uint8_t* dst = L.data + (size_t)u * sgu_unit;
        const int n0 = s1 * R.Fs + 8 * u;
        mbar_expect(&L.bar[u], sgu_unit);
        bulk_copy(dst, LW.ws13 + (size_t)n0 * H, sgu_unit / 2, &L.bar[u]);
        bulk_copy(dst + sgu_unit / 2, LW.ws13 + (size_t)(Is + n0) * H, sgu_unit / 2, &L.bar[u]);
      }
    } else if (is_sdn) {
      for (int u = 0; u < n_sdn_units && u < kSdnSlots; ++u) {
        mbar_expect(&L.bar[u], sdn_unit);
        bulk_copy(L.data + (size_t)u * sdn_unit, LW.ws2 + (size_t)(sdn_m0 + kSdnUnit * u) * Is,
                  sdn_unit, &L.bar[u]);
      }
    }
  }
  // router rows: the routed CTAs compute every logit, experts 2b and 2b + 1
  // (the shared CTAs' own work would delay theirs); each warp covers a 1/kW
  // share of K of both
  const int keighth = H / kW;
  const int k0 = warp * keighth;
  constexpr int kMaxV = kMaxRowH / kW / 128 > 0 ? kMaxRowH / kW / 128 : 1;
  const int nv = keighth / 128;
  float4 wv[2][kMaxV];
  uint2 gw[kMaxV];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int er = is_routed ? 2 * b + h : E;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
      wv[h][i] = (er < E && i < nv)
                     ? __ldg(reinterpret_cast<const float4*>(LW.wr + (size_t)er * H + k0 +
                                                             128 * i + 4 * lane))
                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
#pragma unroll
  for (int i = 0; i < kMaxV; ++i)
    gw[i] = i < nv ? __ldg(reinterpret_cast<const uint2*>(LW.gate + k0 + 128 * i + 4 * lane))
                   : make_uint2(0u, 0u);
  // the add-norm's gamma (immutable) before the wait as well
  const bool addnorm = a.an.residual != nullptr;
  uint2 gn[kMaxV];
#pragma unroll
  for (int i = 0; i < kMaxV; ++i)
    gn[i] = (addnorm && i < nv)
                ? __ldg(reinterpret_cast<const uint2*>(a.an.gamma + k0 + 128 * i + 4 * lane))
                : make_uint2(0u, 0u);
  if (l == 0) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) base_tag = ld_acquire(epoch) + 1;
  }
  if (threadIdx.x == 0) sm->tag = base_tag + l;

  // ---- router logits, x quantisation (1 x 128 groups) and the shared gate ----
  float acc2[2] = {0.0f, 0.0f}, gacc = 0.0f, gmx = 0.0f;
  // both slices' x loads in flight together (the stores below could alias
  // x as far as the compiler knows, so it would not hoist the second)
  uint2 xr[kMaxV];
  if (kChain && l > 0) {
    // x = the previous layer's y: once every routed CTA has counted its
    // combine done (a release after its y stores), read it at L2
    if (threadIdx.x == 0) {
      const int want = R.nR * l;
      long long it = 0;
      while (ld_acquire(ycount) < want) {
        if (++it > kSpin) {
          atomicExch(status, 1);
          break;
        }
        if (it > 16) __nanosleep(32);
      }
    }
    __syncthreads();
    const bf16* yp = a.y + (size_t)(l - 1) * H;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
      xr[i] = i < nv ? __ldcg(reinterpret_cast<const uint2*>(yp + k0 + 128 * i + 4 * lane))
                     : make_uint2(0u, 0u);
  } else {
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
      xr[i] = i < nv ? __ldcg(reinterpret_cast<const uint2*>(a.x + k0 + 128 * i + 4 * lane))
                     : make_uint2(0u, 0u);
  }
  if (addnorm) {
    // residual add and RMS norm in this pass (every CTA the whole row): h =
    // bf16(residual + x), r = 1 / sqrt(sum(h^2) / H + eps) in fp32 over a
    // fixed order (lanes, then warps 0..kW-1), xn = bf16(h * r * gamma); xn
    // then stands for x below.  CTA 0 writes h (and xn if asked).
    uint2 rr[kMaxV];
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
      rr[i] = i < nv ? __ldcg(reinterpret_cast<const uint2*>(a.an.residual + k0 + 128 * i +
                                                             4 * lane))
                     : make_uint2(0u, 0u);
    float hv[kMaxV][4];
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
      if (i >= nv) continue;
      const __nv_bfloat162 r0 = *reinterpret_cast<const __nv_bfloat162*>(&rr[i].x);
      const __nv_bfloat162 r1 = *reinterpret_cast<const __nv_bfloat162*>(&rr[i].y);
      const __nv_bfloat162 x0 = *reinterpret_cast<const __nv_bfloat162*>(&xr[i].x);
      const __nv_bfloat162 x1 = *reinterpret_cast<const __nv_bfloat162*>(&xr[i].y);
      const __nv_bfloat162 h0 = __floats2bfloat162_rn(__low2float(r0) + __low2float(x0),
                                                      __high2float(r0) + __high2float(x0));
      const __nv_bfloat162 h1 = __floats2bfloat162_rn(__low2float(r1) + __low2float(x1),
                                                      __high2float(r1) + __high2float(x1));
      hv[i][0] = __low2float(h0);
      hv[i][1] = __high2float(h0);
      hv[i][2] = __low2float(h1);
      hv[i][3] = __high2float(h1);
#pragma unroll
      for (int c = 0; c < 4; ++c) ss = fmaf(hv[i][c], hv[i][c], ss);
      if (b == 0) {
        uint2 hp;
        hp.x = *reinterpret_cast<const uint32_t*>(&h0);
        hp.y = *reinterpret_cast<const uint32_t*>(&h1);
        *reinterpret_cast<uint2*>(a.an.h_out + k0 + 128 * i + 4 * lane) = hp;
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) sm->gss[warp] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kW; ++w) tot += sm->gss[w];
    const float rn = __frsqrt_rn(__fdiv_rn(tot, (float)H) + a.an.eps);
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
      if (i >= nv) continue;
      const __nv_bfloat162 g0 = *reinterpret_cast<const __nv_bfloat162*>(&gn[i].x);
      const __nv_bfloat162 g1 = *reinterpret_cast<const __nv_bfloat162*>(&gn[i].y);
      const __nv_bfloat162 n0 = __floats2bfloat162_rn(hv[i][0] * rn * __low2float(g0),
                                                      hv[i][1] * rn * __high2float(g0));
      const __nv_bfloat162 n1 = __floats2bfloat162_rn(hv[i][2] * rn * __low2float(g1),
                                                      hv[i][3] * rn * __high2float(g1));
      xr[i].x = *reinterpret_cast<const uint32_t*>(&n0);
      xr[i].y = *reinterpret_cast<const uint32_t*>(&n1);
      if (b == 0 && a.an.xn_out)
        *reinterpret_cast<uint2*>(a.an.xn_out + k0 + 128 * i + 4 * lane) = xr[i];
    }
  }
#pragma unroll
  for (int i = 0; i < kMaxV; ++i) {
    if (i >= nv) continue;
    const int kk = k0 + 128 * i + 4 * lane;
    const uint2 raw = xr[i];
    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
    const float x0 = __low2float(p0), x1 = __high2float(p0), x2 = __low2float(p1),
                x3 = __high2float(p1);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float s = acc2[h];
      s = fmaf(x0, wv[h][i].x, s);
      s = fmaf(x1, wv[h][i].y, s);
      s = fmaf(x2, wv[h][i].z, s);
      s = fmaf(x3, wv[h][i].w, s);
      acc2[h] = s;
    }
    float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
    m = warp_max(m);
    *reinterpret_cast<uint2*>(L.xs + kk) = raw;
    if (a.d.per_row) {
      gmx = fmaxf(gmx, m);  // quantised below, once the row's amax is known
    } else {
      const float sc = group_scale(m);
      const uint32_t packed = quant4(x0, x1, x2, x3, sc);
      *reinterpret_cast<uint32_t*>(L.xq + kk) = packed;
      if (lane == 0) L.sx[kk / kGroup] = sc;
      if (b == 0) {
        *reinterpret_cast<uint32_t*>(a.w.xq + kk) = packed;
        if (lane == 0) a.w.sx[kk / kGroup] = sc;
      }
    }
    const __nv_bfloat162 g0 = *reinterpret_cast<const __nv_bfloat162*>(&gw[i].x);
    const __nv_bfloat162 g1 = *reinterpret_cast<const __nv_bfloat162*>(&gw[i].y);
    gacc = fmaf(x0, __low2float(g0), gacc);
    gacc = fmaf(x1, __high2float(g0), gacc);
    gacc = fmaf(x2, __low2float(g1), gacc);
    gacc = fmaf(x3, __high2float(g1), gacc);
  }
  {
    const float v0 = warp_sum(acc2[0]), v1 = warp_sum(acc2[1]), vg = warp_sum(gacc);
    if (lane == 0) {
      L.red[warp] = v0;
      L.red[kW + warp] = v1;
      sm->gred[warp] = vg;
      sm->gmax[warp] = gmx;
    }
  }
  __syncthreads();
  if (a.d.per_row) {
    // one scale per row: every group takes the row's amax / 448
    float rm = 0.0f;
#pragma unroll
    for (int w = 0; w < kW; ++w) rm = fmaxf(rm, sm->gmax[w]);
    const float sc = group_scale(rm);
#pragma unroll
    for (int i = 0; i < kMaxV; ++i) {
      if (i >= nv) continue;
      const int kk = k0 + 128 * i + 4 * lane;
      const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&xr[i].x);
      const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&xr[i].y);
      const uint32_t packed =
          quant4(__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1), sc);
      *reinterpret_cast<uint32_t*>(L.xq + kk) = packed;
      if (lane == 0) L.sx[kk / kGroup] = sc;
      if (b == 0) {
        *reinterpret_cast<uint32_t*>(a.w.xq + kk) = packed;
        if (lane == 0) a.w.sx[kk / kGroup] = sc;
      }
    }
  }
  layer_tag = sm->tag;
  const unsigned long long tag = (unsigned long long)(unsigned)layer_tag << 32;
  if (threadIdx.x < 2 && is_routed) {
    const int ee = 2 * b + threadIdx.x;
    if (ee < E) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kW; ++w) v += L.red[threadIdx.x * kW + w];
      st_relaxed64(a.w.tlog + ee, tag | __float_as_uint(v));
    }
  }
  if (threadIdx.x == 32) {
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kW; ++w) v += sm->gred[w];
    sm->gamma = sigmoid_f32(v);
    if (b == 0) a.w.gamma[0] = sm->gamma;
  }
  __syncthreads();  // the router scratch is reused below

  if (is_routed) {
    // ---- routed: gather the logits, top-k, then this CTA's expert slice ----
    const int r = b / R.P, p = b % R.P;
    for (int e = threadIdx.x; e < E; e += kThreads)
      L.lg[e] = route_logit(poll_tagged(a.w.tlog + e, tag, status), a.d.rbf16);
    __syncthreads();
    // the top-k on the first 8 warps (the others wait at the barrier below)
    if (k <= 8 && E <= 256) {
      if (warp < 8) topk_one_row_fast<8>(L.lg, E, k, sm->cand_key, sm->cand_id, sm->idx, sm->w);
    } else {
      topk_one_row<kW>(L.lg, E, k, sm->cand_key, sm->cand_id, sm->idx, sm->w);
    }
    __syncthreads();
    const int e = sm->idx[r];
    const int n0 = p * R.F;       // first feature
    const int nu = R.F / 8;       // [8 gate; 8 up] units
    const uint32_t uhalf = 8u * (uint32_t)H;          // bytes of 8 rows (copied)
    const int ldu = H + kRowPad;                        // row stride in shared memory
    const size_t ubytes = (size_t)16 * ldu;             // one [8 gate; 8 up] unit
    const int ldd = I + kRowPad;
    const uint8_t* W13 = LW.w13 + (size_t)e * 2 * I * H;
    const float* S13 = LW.s13 + (size_t)e * (2 * I / kGroup) * nbh;
    uint8_t* w2s = L.data + (size_t)nu * ubytes;  // [128][ldd]
    const float *lg_, *lu_, *ld_;
    int dg, du, dd;
    const uint32_t bg = span16(S13 + (size_t)(n0 / kGroup) * nbh, nbh, &lg_, &dg);
    const uint32_t bu = span16(S13 + (size_t)((I + n0) / kGroup) * nbh, nbh, &lu_, &du);
    const uint32_t bd = span16(LW.s2 + ((size_t)e * nbh + p) * nbi, nbi, &ld_, &dd);
    const size_t wslot = al16((size_t)(nbh + 8) * 4);
    float* sgp = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(L.wsc)) + dg;
    float* sup = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(L.wsc) + wslot) + du;
    float* sdp = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(L.wsc) + 2 * wslot) + dd;
    // copies, one row each, issued in parallel: warp 0 the gate/up rows of
    // the units (bar u), warp 1 the down rows (bar 6), warp 2 the scales
    // (bar 7); each barrier's byte count is set before its copies
    // (a later layer's copies land where the previous layer's rows were read)
    if (kChain && l > 0 && warp < 3) fence_proxy_async();
    if (warp == 0) {
      if (lane < nu) mbar_expect(&L.bar[lane], 2 * uhalf);
      __syncwarp();
      for (int i = lane; i < 16 * nu; i += 32) {
        const int uu = i >> 4, j = i & 15;
        const int n = (j < 8 ? 0 : I) + n0 + 8 * uu + (j & 7);
        bulk_copy(L.data + (size_t)uu * ubytes + (size_t)j * ldu, W13 + (size_t)n * H,
                  (uint32_t)H, &L.bar[uu]);
      }
    } else if (warp == 1) {
      if (lane == 0) mbar_expect(&L.bar[6], (uint32_t)kGroup * I);
      __syncwarp();
      const uint8_t* W2 = LW.w2 + ((size_t)e * H + (size_t)kGroup * p) * I;
      for (int m = lane; m < kGroup; m += 32)
        bulk_copy(w2s + (size_t)m * ldd, W2 + (size_t)m * I, (uint32_t)I, &L.bar[6]);
    } else if (warp == 2 && lane == 0) {
      mbar_expect(&L.bar[7], bg + bu + bd);
      bulk_copy(L.wsc, lg_, bg, &L.bar[7]);
      bulk_copy(reinterpret_cast<uint8_t*>(L.wsc) + wslot, lu_, bu, &L.bar[7]);
      bulk_copy(reinterpret_cast<uint8_t*>(L.wsc) + 2 * wslot, ld_, bd, &L.bar[7]);
    }
    // the routing and the slot order (experts by id) for the checking entry points
    if (warp == 0 && lane < k) {
      const int me = sm->idx[lane];
      int s = 0;
      for (int j = 0; j < k; ++j) s += sm->idx[j] < me;
      sm->slot[lane] = s;
      if (b == 0) {
        a.w.idx[lane] = me;
        a.w.wts[lane] = sm->w[lane];
        a.w.slot_of_pair[lane] = s;
        a.w.pair_of_slot[s] = lane;
        a.w.chunks[s] = make_int4(me, s, 1, 0);
        if (lane == 0) *a.w.n_chunks = k;
      }
    }
    // gate/up: unit u by warps w with w % nu == u, each a part of K
    const int wpu = kW / nu;
    const int u = warp % nu, part = warp / nu;
    const int nsl = H / 64, per = nsl / wpu;
    copy_wait(&L.bar[7], lp, status);
    copy_wait(&L.bar[u], lp, status);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    routed_part(L.data + (size_t)u * ubytes, ldu, sgp, sup, L.xq, L.sx, part * per,
                part * per + per, acc);
    float* red = L.red;  // [kW][32][2]
    red[(warp * 32 + lane) * 2 + 0] = acc[0];
    red[(warp * 32 + lane) * 2 + 1] = acc[2];
    __syncthreads();
    if (warp < nu && q == 0) {
      float zg = 0.0f, zu = 0.0f;
      for (int pp = 0; pp < wpu; ++pp) {  // parts in K order
        const int w = pp * nu + warp;
        zg += red[(w * 32 + lane) * 2 + 0];
        zu += red[(w * 32 + lane) * 2 + 1];
      }
      const float h = silu_f32(bf16_round(zg)) * bf16_round(zu);
      publish(X.h + (size_t)r * I + n0 + 8 * warp + g, tag, h);
    }
    // all I SwiGLU values of expert r, quantised in 1 x 128 groups
    for (int i = threadIdx.x; i < I; i += kThreads)
      L.hall[i] = poll_tagged(X.h + (size_t)r * I + i, tag, status);
    __syncthreads();
    float hrs = 0.0f;  // one scale per row: the SwiGLU row's amax / 448
    if (a.d.per_row) {
      float m = 0.0f;
      for (int i = threadIdx.x; i < I / 4; i += kThreads) {
        const float4 v = *reinterpret_cast<const float4*>(L.hall + 4 * i);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
      m = warp_max(m);
      if (lane == 0) sm->gmax[warp] = m;
      __syncthreads();
#pragma unroll
      for (int w = 0; w < kW; ++w) hrs = fmaxf(hrs, sm->gmax[w]);
      hrs = group_scale(hrs);
    }
    for (int grp = warp; grp < nbi; grp += kW) {
      const float4 v = *reinterpret_cast<const float4*>(L.hall + grp * kGroup + 4 * lane);
      float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
      m = warp_max(m);
      const float s = a.d.per_row ? hrs : group_scale(m);
      const uint32_t packed = quant4(v.x, v.y, v.z, v.w, s);
      *reinterpret_cast<uint32_t*>(L.hq + grp * kGroup + 4 * lane) = packed;
      if (lane == 0) L.sh[grp] = s;
      if (p == 0) {
        const int slot = sm->slot[r];
        *reinterpret_cast<uint32_t*>(a.w.hq + (size_t)slot * I + grp * kGroup + 4 * lane) = packed;
        if (lane == 0) a.w.sh[(size_t)slot * nbi + grp] = s;
      }
    }
    __syncthreads();
    // down rows [128p + 16w, +16) of expert e over the full I
    copy_wait(&L.bar[6], lp, status);
    {
      // 128 rows = 8 m-tiles: warp w takes m-tile w % 8 over K half w / 8;
      // the second half's sums are added through shared memory
      constexpr int kMT = kGroup / 16;
      const int mt = warp % kMT, kh = warp / kMT, nkh = kW / kMT;
      const int per_h = (I / 64) / nkh;
      float dacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const uint8_t* rows = w2s + (size_t)(16 * mt) * ldd;
      for (int bsl = kh * per_h; bsl < kh * per_h + per_h; ++bsl) {
        const int grp = bsl >> 1;
        const int off = bsl * 64 + 16 * q;
        const uint4 a_lo = lds16(rows + (size_t)g * ldd + off);
        const uint4 a_hi = lds16(rows + (size_t)(8 + g) * ldd + off);
        const uint4 bx = lds16(L.hq + off);
        float pp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_e4m3_k64(pp, a_lo, a_hi, bx);
        const float s = sdp[grp] * L.sh[grp];
        dacc[0] = fmaf(pp[0], s, dacc[0]);
        dacc[2] = fmaf(pp[2], s, dacc[2]);
      }
      float* dred = L.red;  // [kW][32][2]
      dred[(warp * 32 + lane) * 2 + 0] = dacc[0];
      dred[(warp * 32 + lane) * 2 + 1] = dacc[2];
      __syncthreads();
      if (kh == 0 && q == 0) {
        float d0 = 0.0f, d1 = 0.0f;
        for (int hh = 0; hh < nkh; ++hh) {  // K halves in order
          const int w = hh * kMT + mt;
          d0 += dred[(w * 32 + lane) * 2 + 0];
          d1 += dred[(w * 32 + lane) * 2 + 1];
        }
        const int m = kGroup * p + 16 * mt + g;
        publish(X.d + (size_t)r * H + m, tag, bf16_round(d0));
        publish(X.d + (size_t)r * H + m + 8, tag, bf16_round(d1));
      }
    }
    // combine rows [128p + (128/k) r, +128/k): sum_j w_j d_j + gamma ds
    const int nrow = kGroup / k;
    const int m0 = kGroup * p + nrow * r;
    for (int i = threadIdx.x; i < (k + 1) * nrow; i += kThreads) {
      const int j = i / nrow, t = i % nrow;
      sm->comb[j][t] = j < k ? poll_tagged(X.d + (size_t)j * H + m0 + t, tag, status)
                             : poll_tagged(X.ds + m0 + t, tag, status);
    }
    __syncthreads();
    if (threadIdx.x < nrow) {
      float y = 0.0f;
      for (int j = 0; j < k; ++j) y = fmaf(sm->w[j], sm->comb[j][threadIdx.x], y);
      y = fmaf(sm->gamma, sm->comb[k][threadIdx.x], y);
      a.y[(kChain ? (size_t)l * H : 0) + m0 + threadIdx.x] = __float2bfloat16_rn(y);
    }
    if (kChain) {
      // the next layer reads this y once every routed CTA has counted itself
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ycount, 1);
      }
    }
  } else if (is_sgu) {
    // ---- shared gate/up: units of [8 gate; 8 up] rows, all warps split K ----
    const int nsl = H / 32, per = nsl / kW;
    for (int uu = 0; uu < n_sgu_units; ++uu) {
      const int slot = uu % kSguSlots;
      // the slot's completions so far: its uses in earlier layers, then here
      const int uses = (n_sgu_units - slot + kSguSlots - 1) / kSguSlots;
      copy_wait(&L.bar[slot], (uint32_t)((l * uses + uu / kSguSlots) & 1), status);
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      shared_part(L.data + (size_t)slot * sgu_unit, H, L.xs, warp * per, warp * per + per, acc);
      float* red = L.red;
      red[(warp * 32 + lane) * 2 + 0] = acc[0];
      red[(warp * 32 + lane) * 2 + 1] = acc[2];
      __syncthreads();
      if (threadIdx.x == 0 && uu + kSguSlots < n_sgu_units) {
        // the slot is free again: its next unit
        const int un = uu + kSguSlots;
        uint8_t* dst = L.data + (size_t)slot * sgu_unit;
        const int n0 = s1 * R.Fs + 8 * un;
        mbar_expect(&L.bar[slot], sgu_unit);
        bulk_copy(dst, LW.ws13 + (size_t)n0 * H, sgu_unit / 2, &L.bar[slot]);
        bulk_copy(dst + sgu_unit / 2, LW.ws13 + (size_t)(Is + n0) * H, sgu_unit / 2,
                  &L.bar[slot]);
      }
      if (warp == 0 && q == 0) {
        float zg = 0.0f, zu = 0.0f;
        for (int w = 0; w < kW; ++w) {  // parts in K order
          zg += red[(w * 32 + lane) * 2 + 0];
          zu += red[(w * 32 + lane) * 2 + 1];
        }
        const float hs = bf16_round(silu_f32(bf16_round(zg)) * bf16_round(zu));
        const int n = s1 * R.Fs + 8 * uu + g;
        publish(X.hs + n, tag, hs);
      }
      __syncthreads();
    }
  } else if (sdn_rows > 0) {
    // ---- shared down: rows [sdn_m0, +sdn_rows), 32 per unit, one warp each ----
    bf16* hsb = reinterpret_cast<bf16*>(L.hall);  // [Is] bf16
    for (int i = threadIdx.x; i < Is; i += kThreads)
      hsb[i] = __float2bfloat16_rn(poll_tagged(X.hs + i, tag, status));
    __syncthreads();
    for (int uu = warp; uu < n_sdn_units; uu += kW) {
      const int slot = uu % kSdnSlots;
      const int uses = (n_sdn_units - slot + kSdnSlots - 1) / kSdnSlots;
      copy_wait(&L.bar[slot], (uint32_t)((l * uses + uu / kSdnSlots) & 1), status);
      const uint8_t* rows = L.data + (size_t)slot * sdn_unit;
      for (int tile = 0; tile < kSdnUnit / 16; ++tile) {
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint8_t* tr = rows + (size_t)(16 * tile) * Is * 2;
#pragma unroll 4
        for (int bsl = 0; bsl < Is / 32; ++bsl) {
          const int off = bsl * 32 + 8 * q;
          const uint4 a_lo = lds16(tr + (size_t)g * Is * 2 + 2 * off);
          const uint4 a_hi = lds16(tr + (size_t)(8 + g) * Is * 2 + 2 * off);
          const uint4 bx = lds16(hsb + off);
          mma_bf16_k32(acc, a_lo, a_hi, bx);
        }
        if (q == 0) {
          const int m = sdn_m0 + kSdnUnit * uu + 16 * tile + g;
          publish(X.ds + m, tag, bf16_round(acc[0]));
          publish(X.ds + m + 8, tag, bf16_round(acc[2]));
        }
      }
      __syncwarp();
      // the slot is free again (only this warp read it): its next unit
      const int un = uu + kSdnSlots;
      if (lane == 0 && un < n_sdn_units) {
        mbar_expect(&L.bar[slot], sdn_unit);
        bulk_copy(L.data + (size_t)slot * sdn_unit,
                  LW.ws2 + (size_t)(sdn_m0 + kSdnUnit * un) * Is, sdn_unit, &L.bar[slot]);
      }
    }
  }

  // every thread is done with this layer's shared scratch (sm->tag, the
  // top-k, the exchange staging) before the next layer writes it
  __syncthreads();
  }  // layers

  // ---- exit: the last CTA advances the launch tag (or clears the words) ----
  launch_exit(a, sm->tag);
}

}  // namespace

size_t decode_row_smem(int G, int H, int E, int k, int I, int Is) {
  const Roles R = make_roles(G, H, k, I, Is);
  return data_bytes(R, H, I, Is) + small_bytes(H, E, I, Is);
}

// Whether the one-row kernel covers this shape on G CTAs within `budget`
// bytes of shared memory per CTA.
bool decode_row_fits(int G, int H, int E, int k, int I, int Is, size_t budget) {
  if (H % (kW * 128) != 0 || H > kMaxRowH) return false;
  if (E > 32 * kW || k > kMaxTopK || kGroup % k != 0 || kGroup / k > 16) return false;
  const Roles R = make_roles(G, H, k, I, Is);
  if (E > 2 * R.nR) return false;  // the routed CTAs compute two logits each
  if (R.nS2 < 1 || I % R.P != 0 || Is % R.P != 0) return false;
  if (R.F < 8 || R.F % 8 != 0 || kGroup % R.F != 0 || kW % (R.F / 8) != 0) return false;
  if (kW % (kGroup / 16) != 0 || (I / 64) % (kW / (kGroup / 16)) != 0) return false;
  if ((H / 64) % (kW / (R.F / 8)) != 0) return false;
  if (R.Fs < 8 || R.Fs % 8 != 0 || (H / 32) % kW != 0) return false;
  if (R.R2 % kSdnUnit != 0 || (size_t)R.R2 * R.nS2 < (size_t)H) return false;
  if (I % 64 != 0 || Is % 32 != 0 || I / kGroup > 8) return false;
  return decode_row_smem(G, H, E, k, I, Is) <= budget;
}

cudaError_t setup_decode_row(size_t max_smem) {
  const cudaError_t e = cudaFuncSetAttribute(
      k_decode_row<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_decode_row<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)max_smem);
}

cudaError_t launch_decode_row(const KArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s) {
  return launch_pdl(k_decode_row<0>, dim3(grid), dim3(kThreads), smem, s, pdl, a);
}

cudaError_t launch_decode_chain(const KArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s) {
  return launch_pdl(k_decode_row<1>, dim3(grid), dim3(kThreads), smem, s, pdl, a);
}

}  // namespace moe

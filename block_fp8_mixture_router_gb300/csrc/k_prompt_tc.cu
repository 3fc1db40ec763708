// Grouped path (five rows or more on the automatic path): the expert GEMMs on
// the fifth-generation tensor cores (tcgen05.mma with TMEM accumulators,
// operands staged by TMA).
//
// Expert arithmetic: PR #939 "Fish Audio Drama 3 text to speech on one CUDA
// GPU", section "Precision" (block-FP8 weights with one fp32 scale per
// 128x128 block, e4m3 inputs per row and per 128 inputs, amax/448); the
// commit "one SwiGLU launch for the routed and shared experts" (routed
// SwiGLU rows stored as their FP8 quantisation, shared rows as bf16).
//
// Operands are swapped relative to the usual token-by-weight product: a tile
// is 128 output features (M, the weight rows, always full) by up to 64
// (block-FP8) or 128 (bf16) tokens (N, rounded up to 16), so experts that see
// few rows waste no tensor work on padding rows, and one 128-feature tile is
// exactly one row of weight
// scale blocks.  For every 128-deep K block the MMAs write a fresh partial
// into one of up to four TMEM buffers (Cfg::kNumBuf); the epilogue warps read
// it back, multiply by (weight block scale x activation scale of each token)
// and accumulate in registers while the tensor cores fill the next buffers.
// The bf16 shared expert needs no per-block scaling and accumulates across K
// in TMEM.
//
// A gate tile and its up tile share the token operand and land in the same
// TMEM lanes, so the thread that owns feature j holds both halves of SwiGLU
// for it.  The tile's outputs are transposed through shared memory and
// stored token-major with coalesced rows.
//
// CTA roles (kTcThreads = 768 threads, 24 warps): warps 0 and 19 issue the
// TMA copies (0: the weight tiles and the item's scales, with the decoded
// item itself for the epilogue; 19: the token tiles), warp 1 owns TMEM and issues the MMAs of the first A tile, warp 18
// those of the second A tile of a pair, warps 2-17 are the epilogue (warp w
// reads TMEM lanes 32*(w%4).. and column quarter (w-2)/4 of the tile's
// tokens).  Issuing an async copy, an MMA, a commit or a barrier wait costs
// one thread tens to a couple of hundred cycles, so each K block's issue
// work is spread over two warps per side.  For the block-FP8 kinds the
// epilogue hands each finished item to warps 20-23 through shared memory
// (both tiles as bf16) and goes on to the next item's K blocks; those warps
// apply SwiGLU, quantise and store, so the stores no longer hold up the
// promotion, and through it the tensor cores.
// Every wait is bounded; a wait that gives up sets the status flag and all
// roles leave their loops.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_rowops.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

// Epilogue warps, 4 per TMEM lane quarter: the per-K-block promotion is a
// chain of dependent loads and FMAs, so four warps per SM sub-partition hide
// its latency (two left the epilogue issue-bound at 40 % of the issue slots).
// With two TMA, two MMA and four store warps that is 24 warps, 6 per
// sub-partition, so a thread may hold up to 80 registers; the block-FP8
// epilogue keeps 2 x 16 promoted accumulators and reads 8 columns of one
// tile from TMEM at a time.
constexpr int kEpiWarps = 16;
constexpr int kStoreWarps = 4;  // block-FP8 kinds: quantise and store finished items
constexpr int kTcThreads = 128 + 32 * (kEpiWarps + kStoreWarps);  // + two TMA, two MMA warps
constexpr int kWarpMma1 = 2 + kEpiWarps;          // MMAs of the pair's second tile
constexpr int kWarpTmaB = 3 + kEpiWarps;          // token-tile copies
constexpr int kWarpStore0 = 4 + kEpiWarps;        // first store warp
constexpr int kTile = 128;        // output features per tile (M)
constexpr int kKBytes = 128;      // bytes of K per stage (one 128B swizzle row)
constexpr int kATileBytes = kTile * kKBytes;
constexpr int kBBox = 16;         // token rows per TMA box
constexpr int kBBoxBytes = kBBox * kKBytes;
constexpr int kTmemCols = 512;

template <int kKind>
struct Cfg {
  static constexpr bool kF8 = kKind == kTcRoutedGateUp || kKind == kTcRoutedDown;
  // gate/up kinds: a gate tile and its up tile; routed down: two adjacent
  // output tiles.  Either way two A tiles share the token operand.
  static constexpr bool kSwiGLU = kKind == kTcRoutedGateUp || kKind == kTcSharedGateUp;
  static constexpr bool kPair = kSwiGLU || kKind == kTcRoutedDown;
  static constexpr bool kRouted = kF8;
  // Tokens per tile (N).  The block-FP8 kinds keep their promoted
  // accumulators in registers (gate and up: 2 x kCols per epilogue thread);
  // the bf16 kinds accumulate in TMEM.
  static constexpr int kN = kF8 ? 64 : 128;
  static constexpr int kCols = kN / (kEpiWarps / 4);  // token columns per epilogue thread
  // TMEM accumulator buffers (gate at +0, up at +kN) and their count
  static constexpr int kAccCols = (kPair ? 2 : 1) * kN;
  static constexpr int kNumBuf = (kTmemCols / kAccCols) < 4 ? (kTmemCols / kAccCols) : 4;
  static constexpr int kStages = kPair ? (kF8 ? 4 : 3) : (kF8 ? 6 : 4);
  static constexpr int kStageBytes = (kPair ? 2 : 1) * kATileBytes + kN * kKBytes;
};

struct Item {
  int e, f, row0, n;
  int kb0, kb1;  // K blocks of this item (a K split of the router, else all)
  int ks;        // its K split (router), else 0
};

// Named barrier of the epilogue warps only.
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kEpiWarps) : "memory");
}

// Work item w = (token tile * n_f + output tile) * ksplit + K split; token
// tiles of every expert in expert order (routed) or of all rows.
template <bool kRouted, int kN>
__device__ __forceinline__ Item decode_item(const TcGemm& g, const int* s_pre, const int* s_off,
                                            const int* s_cnt, int w) {
  Item it;
  // every role decodes every item, so this stays cheap: only the router
  // splits K (the routed kinds never do), and its split bounds fit 32-bit
  // products (K splits <= 16, K blocks well below 2^26)
  int wf = w;
  it.ks = 0;
  it.kb0 = 0;
  it.kb1 = g.n_k;
  if constexpr (!kRouted) {
    if (g.ksplit > 1) {
      wf = w / g.ksplit;
      it.ks = w - wf * g.ksplit;
      it.kb0 = it.ks * g.n_k / g.ksplit;
      it.kb1 = (it.ks + 1) * g.n_k / g.ksplit;
    }
  }
  const int tile = wf / g.n_f;
  it.f = wf - tile * g.n_f;
  if constexpr (kRouted) {
    int lo = 0, hi = g.E;  // largest e with s_pre[e] <= tile
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pre[mid] <= tile) lo = mid; else hi = mid;
    }
    const int j = tile - s_pre[lo];
    it.e = lo;
    it.row0 = s_off[lo] + kN * j;
    it.n = min(kN, s_cnt[lo] - kN * j);
  } else {
    it.e = 0;
    it.row0 = kN * tile;
    it.n = min(kN, g.T - it.row0);
  }
  return it;
}

// Byte range [b0, b1) of an array widened to 16-byte boundaries for one bulk
// copy: the copy starts at *off, is *bytes long, and byte b0 sits *lead bytes
// into it.
struct Span {
  uint64_t off;
  uint32_t bytes, lead;
};

__device__ __forceinline__ Span span16(uint64_t b0, uint64_t b1) {
  const uint64_t a0 = b0 & ~15ull, a1 = (b1 + 15) & ~15ull;
  return Span{a0, (uint32_t)(a1 - a0), (uint32_t)(b0 - a0)};
}

// The scales an item needs, as three spans copied into one scale slot:
// [0] the activation scales of its tokens (rows row0..row0+n-1 of sb
// [rows][n_k]), [1] and [2] the weight block scales of its two A tiles (n_k
// each).  Slot layout: span 0 at 0, span 1 at kSpanA, span 2 at kSpanA + kSpanW.
struct ItemScales {
  Span s[3];
};

__device__ __forceinline__ ItemScales item_scales(const TcGemm& g, const Item& it) {
  ItemScales r;
  r.s[0] = span16((uint64_t)it.row0 * g.n_k * 4, (uint64_t)(it.row0 + it.n) * g.n_k * 4);
  const uint64_t w0 = ((uint64_t)it.e * (g.a_rows_e / 128) + (uint64_t)it.f * (g.f_rows / 128)) * g.n_k * 4;
  const uint64_t w1 = w0 + (uint64_t)(g.up_rows / 128) * g.n_k * 4;
  r.s[1] = span16(w0, w0 + (uint64_t)g.n_k * 4);
  r.s[2] = span16(w1, w1 + (uint64_t)g.n_k * 4);
  return r;
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(tc::smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
      : "memory");
}

// Stores output tile columns c = w0, w0 + kW, ... of an item from tbuf ([token
// column][128 features], fp32), kW warps taking part, four columns per warp
// at a time so their reductions and divisions overlap: the routed gate/up
// quantises each column's 128 SwiGLU values as one group into hq and sh
// (per-row contexts store them as fp32 rows instead), the router stores fp32
// logits, the other kinds bf16 rows.
template <int kKind, int kW>
__device__ __forceinline__ void store_cols(const TcGemm& g, const Item& it, const float* tbuf,
                                           int fcol, int w0, int lane) {
  for (int c0s = w0; c0s < it.n; c0s += 4 * kW) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int col = c0s + kW * u;
      v[u] = col < it.n ? *reinterpret_cast<const float4*>(tbuf + col * kTile + 4 * lane)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if constexpr (kKind == kTcRoutedGateUp) {
      if (g.hf) {
        // one scale per row: the fp32 SwiGLU rows, quantised per row
        // once every feature tile of the row is done (k_quant_h_rows)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int col = c0s + kW * u;
          if (col < it.n)
            *reinterpret_cast<float4*>(g.hf + (size_t)(it.row0 + col) * g.ldo + fcol +
                                       4 * lane) = v[u];
        }
        continue;
      }
      float m[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        m[u] = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int u = 0; u < 4; ++u) m[u] = fmaxf(m[u], __shfl_xor_sync(0xffffffffu, m[u], o));
      // the four columns' scales and codes on their fast paths first,
      // the rare exact fallbacks after, so the four chains interleave
      float sq[4];
      uint32_t code[4];
      bool rare[4], und[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) sq[u] = group_scale_fast(m[u], rare[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (rare[u]) sq[u] = group_scale(m[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        code[u] = quant4_fast(v[u].x, v[u].y, v[u].z, v[u].w, sq[u], und[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (und[u]) code[u] = quant4_exact(v[u].x, v[u].y, v[u].z, v[u].w, sq[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int col = c0s + kW * u;
        if (col < it.n) {
          const size_t r = (size_t)(it.row0 + col);
          *reinterpret_cast<uint32_t*>(g.hq + r * g.ldo + fcol + 4 * lane) = code[u];
          if (lane == 0) g.sh[r * (g.ldo / kTile) + fcol / kTile] = sq[u];
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int col = c0s + kW * u;
        if (col >= it.n) continue;
        const size_t r = (size_t)(it.row0 + col);
        if constexpr (kKind == kTcRouter) {
          const int e = fcol + 4 * lane;  // logits [row][E], fp32
          float* o = g.outf + ((size_t)it.ks * g.T + r) * g.ldo + e;
          if (e + 3 < g.ldo) {
            *reinterpret_cast<float4*>(o) = v[u];
          } else {
            if (e < g.ldo) o[0] = v[u].x;
            if (e + 1 < g.ldo) o[1] = v[u].y;
            if (e + 2 < g.ldo) o[2] = v[u].z;
          }
        } else {
          __nv_bfloat162 p0 = __floats2bfloat162_rn(v[u].x, v[u].y);
          __nv_bfloat162 p1 = __floats2bfloat162_rn(v[u].z, v[u].w);
          uint2 o;
          o.x = *reinterpret_cast<uint32_t*>(&p0);
          o.y = *reinterpret_cast<uint32_t*>(&p1);
          *reinterpret_cast<uint2*>(g.out + r * g.ldo + fcol + 4 * lane) = o;
        }
      }
    }
  }
}

// Two bf16 values packed in a word (first in the low half) as floats.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// The routed gate/up's SwiGLU and store by the store warps, from the gate
// and up tiles in t16 ([tile][token column][128 features], bf16, tile 1 at
// column kN).  kW warps take four token columns each per pass, eight lanes
// per column and 16 of its 128 SwiGLU values per lane (4-value chunks k,
// k+8, k+16, k+24 of lane k of the eight, so that each load and store
// instruction covers whole rows).  A column's group amax is then three
// shuffles away, and each lane divides by its column's scale once for its
// 16 values.
template <int kW, int kN>
__device__ __forceinline__ void store_gateup_cols(const TcGemm& g, const Item& it,
                                                  const __nv_bfloat16* t16, int fcol, int w0,
                                                  int lane) {
  const int k = lane & 7;
  for (int cb = 4 * w0; cb < it.n; cb += 4 * kW) {
    const int col = cb + (lane >> 3);
    const bool ok = col < it.n;
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok) {
        const uint2 zg = *reinterpret_cast<const uint2*>(t16 + col * kTile + 4 * (k + 8 * i));
        const uint2 zu = *reinterpret_cast<const uint2*>(t16 + (kN + col) * kTile + 4 * (k + 8 * i));
        const float2 g01 = bf16x2_to_float2(zg.x), g23 = bf16x2_to_float2(zg.y);
        const float2 u01 = bf16x2_to_float2(zu.x), u23 = bf16x2_to_float2(zu.y);
        v[i] = make_float4(silu_f32(g01.x) * u01.x, silu_f32(g01.y) * u01.y,
                           silu_f32(g23.x) * u23.x, silu_f32(g23.y) * u23.y);
      }
    }
    const size_t r = (size_t)(it.row0 + (ok ? col : 0));
    if (g.hf) {
      // one scale per row: the fp32 SwiGLU rows, quantised per row once
      // every feature tile of the row is done (k_quant_h_rows)
      if (ok)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<float4*>(g.hf + r * g.ldo + fcol + 4 * (k + 8 * i)) = v[i];
      continue;
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    bool rare;
    float sq = group_scale_fast(m, rare);
    if (rare) sq = group_scale(m);
    uint32_t code[4];
    bool und[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) code[i] = quant4_fast(v[i].x, v[i].y, v[i].z, v[i].w, sq, und[i]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (und[i]) code[i] = quant4_exact(v[i].x, v[i].y, v[i].z, v[i].w, sq);
    if (ok) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint32_t*>(g.hq + r * g.ldo + fcol + 4 * (k + 8 * i)) = code[i];
      if (k == 0) g.sh[r * (g.ldo / kTile) + fcol / kTile] = sq;
    }
  }
}

// 24 warps: an SM sub-partition holds 6 of them, so a thread may use at most
// 80 registers (6 x 32 x 80 <= 16384 per sub-partition)
template <int kKind>
__global__ void __launch_bounds__(kTcThreads, 1) k_tc_gemm(const __grid_constant__ TcGemm g) {
  using C = Cfg<kKind>;
  constexpr bool kF8 = C::kF8, kPair = C::kPair, kRouted = C::kRouted;
  constexpr int S = C::kStages, kN = C::kN, kCols = C::kCols, NB = C::kNumBuf;
  constexpr int kAcc = C::kAccCols;
  extern __shared__ uint8_t smem_raw[];
  // block-FP8: the item whose scales scale slot s holds, decoded by the
  // weight-tile TMA warp and published with the slot's barrier, so that the
  // epilogue warps need not decode it again
  __shared__ Item s_item[2];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* stages = base;
  float* tbuf = reinterpret_cast<float*>(base + S * C::kStageBytes);  // [kN col][128 row]
  uint8_t* sbs = reinterpret_cast<uint8_t*>(tbuf + kN * kTile);       // 2 x scale spans
  const uint32_t span_a = (uint32_t)((kN * g.n_k * 4 + 32 + 15) & ~15);
  const uint32_t span_w = (uint32_t)((g.n_k * 4 + 32 + 15) & ~15);
  const uint32_t sbs_slot = kF8 ? span_a + 2 * span_w : 0u;
  // block-FP8: the current item's scale products [2 tiles][n_k][kN] (weight
  // block scale x token scale), formed once per item
  float* pbuf = reinterpret_cast<float*>(sbs + 2 * sbs_slot);
  uint64_t* bars = reinterpret_cast<uint64_t*>(pbuf + (kF8 ? 2 * g.n_k * kN : 0));
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = bars + 2 * S + NB;
  uint64_t* sfull = bars + 2 * S + 2 * NB;
  uint64_t* sempty = sfull + 2;
  // block-FP8: tbuf holds a finished item (dfull) / has been stored (dfree)
  uint64_t* dfull = sempty + 2;
  uint64_t* dfree = dfull + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(dfree + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_pre = reinterpret_cast<int*>(s_tmem + 2);  // [E+1]
  int* s_off = s_pre + kMaxExperts + 1;              // [E]
  int* s_cnt = s_off + kMaxExperts;                  // [E]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // full: both TMA warps arrive with their bytes; empty and tfull: one
    // commit from each MMA warp
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], 2);
      tc::mbar_init(&empty[i], kPair ? 2 : 1);
    }
    for (int i = 0; i < NB; ++i) {
      tc::mbar_init(&tfull[i], kPair ? 2 : 1);
      tc::mbar_init(&tempty[i], kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sfull[i], 1);
      tc::mbar_init(&sempty[i], kEpiWarps);
    }
    tc::mbar_init(dfull, kEpiWarps);
    tc::mbar_init(dfree, kStoreWarps);
    // an empty item in both slots: after a failed wait the epilogue may read
    // a slot that no item was published to, and must then find no K blocks
    for (int i = 0; i < 2; ++i) s_item[i] = Item{0, 0, 0, 0, 0, 0, 0};
    *s_abort = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_map(&g.a);
    tc::tma_prefetch_map(&g.b);
    tc::tma_prefetch_map(&g.bt);
  }
  if (warp == 1) {
    __syncwarp();
    tc::tmem_alloc(s_tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  // everything above touches no data of the previous kernel
  pdl_wait();
  pdl_trigger();
  int n_tiles;
  if constexpr (kRouted) {
    // token tiles per expert and their prefix (warp 0; E <= 256, 8 per lane)
    for (int e = threadIdx.x; e < g.E; e += kTcThreads) {
      s_cnt[e] = g.counts[e];
      s_off[e] = g.off[e];
    }
    __syncthreads();
    if (warp == 0) {
      int loc[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = 8 * lane + i;
        loc[i] = e < g.E ? (s_cnt[e] + kN - 1) / kN : 0;
        sum += loc[i];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - sum;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = 8 * lane + i;
        if (e < g.E) s_pre[e] = run;
        run += loc[i];
      }
      if (lane == 31) s_pre[g.E] = incl;
    }
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  if constexpr (kRouted) n_tiles = s_pre[g.E];
  else n_tiles = (g.T + kN - 1) / kN;
  const int n_items = n_tiles * g.n_f * g.ksplit;
  const int n_k = g.n_k;
  const int kx = kF8 ? kKBytes : kKBytes / 2;  // K elements per stage

  // The TMA and MMA warps walk their loops as whole warps: every lane polls
  // the barriers and computes the coordinates and descriptors, and lane 0
  // issues the copies, MMAs and commits.  A wait counts as
  // failed for the warp if it failed in any lane.
  if (warp == 0 || warp == kWarpTmaB) {
    // ---- TMA producers: warp 0 the weight tiles (and the item's scales),
    // warp kWarpTmaB the token tiles; each arrives on full with its bytes ----
    const bool wa = warp == 0;
    uint32_t st = 0, ph = 0;
    bool ok = true;
    int n_issued = 0;  // stages issued so far (the last S are drained on abort)
    for (int w = blockIdx.x, j = 0; w < n_items && ok; w += gridDim.x, ++j) {
      const Item it = decode_item<kRouted, kN>(g, s_pre, s_off, s_cnt, w);
      if (kF8 && wa) {
        // this item's activation scales into scale slot j % 2
        const int sl = j & 1;
        const bool r = tc::wait_bounded(&sempty[sl], ((j >> 1) & 1) ^ 1u, s_abort, g.status);
        if (__any_sync(0xffffffffu, !r)) {
          ok = false;
          break;
        }
        const ItemScales sc = item_scales(g, it);
        uint8_t* slot = sbs + sl * sbs_slot;
        if (lane == 0) {
          s_item[sl] = it;  // published by the arrival below (release)
          tc::mbar_arrive_expect_tx(&sfull[sl], sc.s[0].bytes + sc.s[1].bytes + sc.s[2].bytes);
          bulk_copy_g2s(slot, reinterpret_cast<const uint8_t*>(g.sb) + sc.s[0].off, sc.s[0].bytes,
                        &sfull[sl]);
          bulk_copy_g2s(slot + span_a, reinterpret_cast<const uint8_t*>(g.sa) + sc.s[1].off,
                        sc.s[1].bytes, &sfull[sl]);
          bulk_copy_g2s(slot + span_a + span_w, reinterpret_cast<const uint8_t*>(g.sa) + sc.s[2].off,
                        sc.s[2].bytes, &sfull[sl]);
        }
        __syncwarp();
      }
      const int arow = it.e * g.a_rows_e + it.f * g.f_rows;
      // a tile of more than half the token rows takes one box of kN rows
      // (rows past the tile belong to the next expert or lie beyond the
      // operand, which reads zeros; the MMA does not use them), a smaller
      // one its 16-row boxes: fewer copies for the issuing lane
      const bool whole = 2 * it.n > kN;
      const int nb = whole ? 1 : (it.n + kBBox - 1) / kBBox;
      const uint32_t bytes =
          wa ? (kPair ? 2 : 1) * kATileBytes : (whole ? kN * kKBytes : nb * kBBoxBytes);
      for (int kb = it.kb0; kb < it.kb1; ++kb) {
        const bool r = tc::wait_bounded(&empty[st], ph ^ 1u, s_abort, g.status);
        if (__any_sync(0xffffffffu, !r)) { ok = false; break; }
        uint8_t* sp = stages + st * C::kStageBytes;
        const int bx = (kb % g.b_kwrap) * kx;
        uint8_t* bp = sp + (kPair ? 2 : 1) * kATileBytes;
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(&full[st], bytes);
          if (wa) {
            tc::tma_load_2d(sp, &g.a, kb * kx, arow, &full[st]);
            if constexpr (kPair)
              tc::tma_load_2d(sp + kATileBytes, &g.a, kb * kx, arow + g.up_rows, &full[st]);
          } else if (whole) {
            tc::tma_load_2d(bp, &g.bt, bx, it.row0, &full[st]);
          } else {
            for (int i = 0; i < nb; ++i)
              tc::tma_load_2d(bp + i * kBBoxBytes, &g.b, bx, it.row0 + kBBox * i, &full[st]);
          }
        }
        __syncwarp();
        ++n_issued;
        if (++st == (uint32_t)S) { st = 0; ph ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      // let copies already in flight land before the CTA leaves (bounded:
      // a stage the other producer never armed gives up at the limit)
      const unsigned long long t0 = tc::global_ns();
      for (int i = 1; i <= S && i <= n_issued; ++i) {
        const int k = n_issued - i;  // stage k % S was filled in phase (k / S) & 1
        while (!tc::mbar_try_wait(&full[k % S], (uint32_t)((k / S) & 1)) &&
               tc::global_ns() - t0 < tc::kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1 || (kPair && warp == kWarpMma1)) {
    // ---- MMA issuers: warp 1 the first A tile, warp kWarpMma1 the second
    // (pairs); each commits once to empty and to tfull ----
    const int tile = warp == 1 ? 0 : 1;
    uint32_t st = 0, ph = 0, tb = 0, tph = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      const Item it = decode_item<kRouted, kN>(g, s_pre, s_off, s_cnt, w);
      const int n16 = (it.n + 15) & ~15;
      const uint32_t idesc = kF8 ? tc::idesc_f8(kTile, n16) : tc::idesc_bf16(kTile, n16);
      for (int kb = it.kb0; kb < it.kb1; ++kb) {
        if (kF8 || kb == it.kb0) {
          const bool r = tc::wait_bounded(&tempty[tb], tph ^ 1u, s_abort, g.status);
          if (__any_sync(0xffffffffu, !r)) { ok = false; break; }
          tc::fence_after_sync();
        }
        const bool r = tc::wait_bounded(&full[st], ph, s_abort, g.status);
        if (__any_sync(0xffffffffu, !r)) { ok = false; break; }
        tc::fence_after_sync();
        // descriptors of the stage's operands; each 32-byte K step adds 2 to
        // the start-address field (address >> 4)
        const uint32_t sa0 = tc::smem_u32(stages + st * C::kStageBytes);
        const uint64_t da = tc::sw128_desc(sa0 + tile * kATileBytes);
        const uint64_t db = tc::sw128_desc(sa0 + (kPair ? 2 : 1) * kATileBytes);
        const uint32_t d0 = tmem + tb * kAcc + tile * kN;
#pragma unroll
        for (int kk = 0; kk < kKBytes / 32; ++kk) {
          const uint32_t acc = (kk > 0 || (!kF8 && kb > it.kb0)) ? 1u : 0u;
          tc::mma_warp<kF8>(d0, da + 2 * kk, db + 2 * kk, idesc, acc);
        }
        tc::commit_warp(&empty[st]);
        if (++st == (uint32_t)S) { st = 0; ph ^= 1u; }
        if (kF8 || kb == it.kb1 - 1) {
          tc::commit_warp(&tfull[tb]);
          if (++tb == (uint32_t)NB) { tb = 0; tph ^= 1u; }
        }
      }
    }
  } else if (warp >= 2 && warp < 2 + kEpiWarps) {
    // ---- epilogue ----
    const int ew = warp - 2;
    const int q = warp & 3;
    const int c0 = kCols * (ew >> 2);  // this warp's first token column
    const int row = 32 * q + lane;
    const uint32_t tl = (uint32_t)(32 * q) << 16;
    uint32_t tb = 0, tph = 0;
    // After a failed wait the warps still walk every item (all later waits
    // give up at once), so each of them reaches every named barrier.
    for (int w = blockIdx.x, j = 0; w < n_items; w += gridDim.x, ++j) {
      // block-FP8: the item comes with its scale slot; the bf16 kinds decode it
      Item it;
      if constexpr (kF8) {
        tc::wait_bounded(&sfull[j & 1], (j >> 1) & 1, s_abort, g.status);
        it = s_item[j & 1];
      } else {
        it = decode_item<kRouted, kN>(g, s_pre, s_off, s_cnt, w);
      }
      const int n16 = (it.n + 15) & ~15;
      // this item's scales in the slot: [token][n_k], and n_k per A tile
      const float* sc_tok = nullptr;
      const float* s_wg = nullptr;
      const float* s_wu = nullptr;
      if constexpr (kF8) {
        const int sl = j & 1;
        const ItemScales sc = item_scales(g, it);
        const uint8_t* slot = sbs + sl * sbs_slot;
        epi_sync();  // every warp has left the previous item's K loop, pbuf's last reader
        sc_tok = reinterpret_cast<const float*>(slot + sc.s[0].lead);
        s_wg = reinterpret_cast<const float*>(slot + span_a + sc.s[1].lead);
        s_wu = reinterpret_cast<const float*>(slot + span_a + span_w + sc.s[2].lead);
        // (weight block scale x token scale) for every (tile, K block, token);
        // padding tokens get 0.  With n_k % 4 == 0 the token scales are read
        // as float4 rows (16-byte aligned then), four K blocks per thread,
        // consecutive lanes on consecutive vectors: no bank conflicts on
        // the reads, which a token-major walk (stride n_k) would have.
        if ((n_k & 3) == 0) {
          const int nq = n_k >> 2;
          for (int v = 32 * ew + lane; v < kN * nq; v += 32 * kEpiWarps) {
            const int t = v / nq, kq = v - t * nq;
            const float4 s4 = t < it.n ? reinterpret_cast<const float4*>(sc_tok + t * n_k)[kq]
                                       : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            const float st[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int kb = 4 * kq + r;
              pbuf[kb * kN + t] = s_wg[kb] * st[r];
              pbuf[(n_k + kb) * kN + t] = s_wu[kb] * st[r];
            }
          }
        } else {
          for (int i = 32 * ew + lane; i < n_k * kN; i += 32 * kEpiWarps) {
            const int kb = i / kN, t = i - kb * kN;
            const float st = t < it.n ? sc_tok[t * n_k + kb] : 0.0f;
            pbuf[i] = s_wg[kb] * st;
            pbuf[n_k * kN + i] = s_wu[kb] * st;
          }
        }
        epi_sync();
      }
      float acc0[kCols], acc1[kCols];
#pragma unroll
      for (int i = 0; i < kCols; ++i) { acc0[i] = 0.0f; acc1[i] = 0.0f; }
      for (int kb = (kF8 ? it.kb0 : it.kb1 - 1); kb < it.kb1; ++kb) {
        tc::wait_bounded(&tfull[tb], tph, s_abort, g.status);
        __syncwarp();  // lanes may leave the poll at different tries
        tc::fence_after_sync();
        const uint32_t ta0 = tmem + tl + tb * kAcc + c0;
        if constexpr (kF8) {
          // block-FP8: partial x (weight block scale x token scale), 8
          // columns of one tile under one TMEM wait at a time; the products
          // come from pbuf as broadcast vectors
          static_assert(kCols % 8 == 0, "x8 loads per tile");
#pragma unroll
          for (int c8 = 0; c8 < kCols / 8; ++c8) {
            if (c0 + 8 * c8 < n16) {
#pragma unroll
              for (int tile = 0; tile < 2; ++tile) {
                uint32_t va[8];
                tc::tmem_ld8(ta0 + tile * kN + 8 * c8, va);
                const float4* ps = reinterpret_cast<const float4*>(
                    pbuf + (tile * n_k + kb) * kN + c0 + 8 * c8);
                float* acc = tile == 0 ? acc0 : acc1;
#pragma unroll
                for (int q4 = 0; q4 < 2; ++q4) {
                  const float4 s4 = ps[q4];
                  const float ss[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const int c = 8 * c8 + 4 * q4 + i;
                    acc[c] = fmaf(__uint_as_float(va[4 * q4 + i]), ss[i], acc[c]);
                  }
                }
              }
            }
          }
        } else {
          // bf16: the whole K is in this accumulator
          epi_sync();  // every warp is done reading tbuf
#pragma unroll
          for (int c4 = 0; c4 < kCols / 16; ++c4) {
            if (c0 + 16 * c4 < n16) {
              uint32_t va[16], vb[16];
              if constexpr (kPair) tc::tmem_ld16x2(ta0 + 16 * c4, ta0 + kN + 16 * c4, va, vb);
              else tc::tmem_ld16(ta0 + 16 * c4, va);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float v = __uint_as_float(va[i]);
                if constexpr (kPair)
                  v = bf16_round(silu_f32(bf16_round(v)) * bf16_round(__uint_as_float(vb[i])));
                tbuf[(c0 + 16 * c4 + i) * kTile + row] = v;
              }
            }
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&tempty[tb]);
        if (++tb == (uint32_t)NB) { tb = 0; tph ^= 1u; }
      }
      if constexpr (kF8) {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sempty[j & 1]);  // scale slot free
        // hand the item to the store warps through tbuf, once they have
        // stored the previous one: both tiles as bf16, the precision SwiGLU
        // reads gate and up in and the down outputs are stored in
        if (j > 0) tc::wait_bounded(dfree, (uint32_t)((j - 1) & 1), s_abort, g.status);
        {
          __nv_bfloat16* t16 = reinterpret_cast<__nv_bfloat16*>(tbuf);
#pragma unroll
          for (int i = 0; i < kCols; ++i) {
            t16[(c0 + i) * kTile + row] = __float2bfloat16_rn(acc0[i]);
            t16[(kN + c0 + i) * kTile + row] = __float2bfloat16_rn(acc1[i]);
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(dfull);
        continue;
      }
      // bf16 kinds: the output tile, through tbuf
      epi_sync();
      store_cols<kKind, kEpiWarps>(g, it, tbuf, it.f * g.f_rows, ew, lane);
    }
  } else if (kF8 && warp >= kWarpStore0) {
    // ---- store warps (block-FP8): each item from tbuf to global memory ----
    const int sw = warp - kWarpStore0;
    for (int w = blockIdx.x, j = 0; w < n_items; w += gridDim.x, ++j) {
      const Item it = decode_item<kRouted, kN>(g, s_pre, s_off, s_cnt, w);
      tc::wait_bounded(dfull, (uint32_t)(j & 1), s_abort, g.status);
      const __nv_bfloat16* t16 = reinterpret_cast<const __nv_bfloat16*>(tbuf);
      if constexpr (C::kSwiGLU) {
        store_gateup_cols<kStoreWarps, kN>(g, it, t16, it.f * g.f_rows, sw, lane);
      } else {
        // the routed down pair: two output tiles of bf16 rows
        for (int ot = 0; ot < 2; ++ot) {
          const int fcol = it.f * g.f_rows + ot * kTile;
          for (int col = sw; col < it.n; col += kStoreWarps)
            *reinterpret_cast<uint2*>(g.out + (size_t)(it.row0 + col) * g.ldo + fcol + 4 * lane) =
                *reinterpret_cast<const uint2*>(t16 + (ot * kN + col) * kTile + 4 * lane);
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(dfree);
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int kKind>
size_t smem_bytes(int n_k) {
  using C = Cfg<kKind>;
  const size_t slot = C::kF8 ? (((size_t)C::kN * n_k * 4 + 32 + 15) & ~(size_t)15) +
                                   2 * (((size_t)n_k * 4 + 32 + 15) & ~(size_t)15)
                             : 0;
  const size_t prod = C::kF8 ? (size_t)2 * n_k * C::kN * 4 : 0;
  return 1024 + (size_t)C::kStages * C::kStageBytes + (size_t)C::kN * kTile * 4 + 2 * slot +
         prod + (2 * C::kStages + 2 * C::kNumBuf + 6) * 8 + 16 + (3 * kMaxExperts + 1) * 4;
}

const void* kernel_of(int kind) {
  switch (kind) {
    case kTcRoutedGateUp: return (const void*)k_tc_gemm<kTcRoutedGateUp>;
    case kTcRoutedDown: return (const void*)k_tc_gemm<kTcRoutedDown>;
    case kTcSharedGateUp: return (const void*)k_tc_gemm<kTcSharedGateUp>;
    case kTcSharedDown: return (const void*)k_tc_gemm<kTcSharedDown>;
    default: return (const void*)k_tc_gemm<kTcRouter>;
  }
}

}  // namespace

int tc_gemm_tile_rows(int kind) {
  switch (kind) {
    case kTcRoutedGateUp: return Cfg<kTcRoutedGateUp>::kN;
    case kTcRoutedDown: return Cfg<kTcRoutedDown>::kN;
    case kTcSharedGateUp: return Cfg<kTcSharedGateUp>::kN;
    case kTcSharedDown: return Cfg<kTcSharedDown>::kN;
    default: return Cfg<kTcRouter>::kN;
  }
}

size_t tc_gemm_smem(int kind, int n_k) {
  switch (kind) {
    case kTcRoutedGateUp: return smem_bytes<kTcRoutedGateUp>(n_k);
    case kTcRoutedDown: return smem_bytes<kTcRoutedDown>(n_k);
    case kTcSharedGateUp: return smem_bytes<kTcSharedGateUp>(n_k);
    case kTcSharedDown: return smem_bytes<kTcSharedDown>(n_k);
    default: return smem_bytes<kTcRouter>(n_k);
  }
}

cudaError_t setup_tc_gemm(int kind, size_t smem) {
  return cudaFuncSetAttribute(kernel_of(kind), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem);
}

cudaError_t launch_tc_gemm(int kind, const TcGemm& g, int grid, size_t smem, cudaStream_t s,
                           bool pdl) {
  if (grid < 1) return cudaSuccess;
  void* args[] = {const_cast<TcGemm*>(&g)};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelExC(&cfg, kernel_of(kind), args);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Tensor map of a row-major 2-D array [rows][cols] (element size `esize`),
// box = 128 bytes of columns x box_rows rows, 128-byte swizzle.
// The driver's encoder, looked up through the runtime so that the library
// loads on hosts without a driver (it then simply has no tensor-core path).
static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cudaGetLastError();
  }
  return fn;
}

bool make_tc_map(CUtensorMap* m, bool bf16_elems, const void* ptr, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = encoder();
  if (!encode) return false;
  const uint64_t esize = bf16_elems ? 2 : 1;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esize};
  cuuint32_t box[2] = {(cuuint32_t)(kKBytes / esize), box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = encode(
      m, bf16_elems ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
      const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace moe

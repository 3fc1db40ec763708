// Row kernels around the tcgen05 GEMMs (k_prompt_tc.cu): the activations
// quantised straight into the GEMMs' (expert, row) slot order with the shared
// gate, the SwiGLU rows' quantisation when a row takes one scale, and the
// router weights' exact three-way bf16 split.
//
// Activation quantisation: PR #939 "Fish Audio Drama 3 text to speech on one
// CUDA GPU", section "Precision" (e4m3 per row and per 128 inputs,
// amax / 448); the "Drama 3 text backbone" commit of PR #925 (dynamic 1 x 128
// FP8 activation quantization).  Router: PR #939 section "What it adds".
#include "moe_rowops.cuh"

namespace moe {

namespace {

// ---- activation quantisation straight into (expert, row) slot order --------
// Two rows per CTA of 256 threads, 128 threads per row, each 16 consecutive
// elements per pass (a 1 x 128 group is 8 threads): x[t] quantised in 1 x 128
// groups (as quant_row_and_gate), its codes (16 bytes per thread) and group
// scales written to each of the row's k slots, and gamma[t] from the same
// registers.  Every thread reads the slot numbers itself, so no barrier
// stands between the row's loads and its stores.
constexpr int kQsThreads = 256;
constexpr int kQsRowThreads = 128;           // threads per row
constexpr int kQsRows = kQsThreads / kQsRowThreads;
constexpr int kQsPass = 16 * kQsRowThreads;  // elements of a row per pass

__device__ __forceinline__ float amax8(const uint4 r) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    m = fmaxf(m, fmaxf(fabsf(__low2float(p)), fabsf(__high2float(p))));
  }
  return m;
}

__global__ void __launch_bounds__(kQsThreads, 4) k_quant_scatter(KArgs a, uint8_t* xg, float* sxg) {
  __shared__ float red[kQsThreads / 32];
  const int T = a.d.T, H = a.d.H, k = a.d.k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = threadIdx.x / kQsRowThreads;  // which of the CTA's rows
  const int t = blockIdx.x * kQsRows + half;
  const bool active = t < T;
  const int ngroups = H / kGroup;
  const bf16* xr = a.x + (size_t)t * H;
  const bool pre_q = a.an.pre_q != 0;  // the add-norm already wrote the row's codes
  // the shared gate's weights (immutable) before the wait
  const int base0 = 16 * (threadIdx.x % kQsRowThreads);
  uint4 g0 = make_uint4(0u, 0u, 0u, 0u), g1 = g0;
  if (base0 < H) {
    g0 = __ldg(reinterpret_cast<const uint4*>(a.L.gate + base0));
    g1 = __ldg(reinterpret_cast<const uint4*>(a.L.gate + base0 + 8));
  }
  pdl_wait();
  pdl_trigger();
  uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
  if (active && base0 < H) {
    x0 = *reinterpret_cast<const uint4*>(xr + base0);
    x1 = *reinterpret_cast<const uint4*>(xr + base0 + 8);
  }
  // one scale per row: the row's amax over its threads' warps
  float rs = 0.0f;
  if (a.d.per_row && !pre_q) {
    float m = 0.0f;
    if (active)
      for (int base = base0; base < H; base += kQsPass)
        m = fmaxf(m, fmaxf(amax8(*reinterpret_cast<const uint4*>(xr + base)),
                           amax8(*reinterpret_cast<const uint4*>(xr + base + 8))));
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    constexpr int kRowWarps = kQsRowThreads / 32;
    for (int w = 0; w < kRowWarps; ++w) rs = fmaxf(rs, red[half * kRowWarps + w]);
    rs = group_scale(rs);
    __syncthreads();  // red is free again
  }
  const int* slot_row = a.w.slot_of_pair + (size_t)t * k;
  float acc = 0.0f;  // the shared gate's dot product from the same registers
  if (active) {
    for (int base = base0; base < H; base += kQsPass) {
      if (base != base0) {
        x0 = *reinterpret_cast<const uint4*>(xr + base);
        x1 = *reinterpret_cast<const uint4*>(xr + base + 8);
        g0 = __ldg(reinterpret_cast<const uint4*>(a.L.gate + base));
        g1 = __ldg(reinterpret_cast<const uint4*>(a.L.gate + base + 8));
      }
      const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&xw[i]);
        const __nv_bfloat162 g = *reinterpret_cast<const __nv_bfloat162*>(&gw[i]);
        v[2 * i] = __low2float(p);
        v[2 * i + 1] = __high2float(p);
        acc = fmaf(v[2 * i], __low2float(g), acc);
        acc = fmaf(v[2 * i + 1], __high2float(g), acc);
      }
      const int gi = base / kGroup;
      uint4 packed;
      float sc;
      if (pre_q) {
        packed = *reinterpret_cast<const uint4*>(a.w.xq + (size_t)t * H + base);
        sc = a.w.sx[(size_t)t * ngroups + gi];
      } else {
        // a pass covers whole groups (H % 128 == 0), so the 8 threads of a
        // group take part in it together
        const unsigned grp = 0xFFu << (lane & 24);
        float m = fmaxf(amax8(x0), amax8(x1));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(grp, m, o));
        sc = a.d.per_row ? rs : group_scale(m);
        packed.x = quant4(v[0], v[1], v[2], v[3], sc);
        packed.y = quant4(v[4], v[5], v[6], v[7], sc);
        packed.z = quant4(v[8], v[9], v[10], v[11], sc);
        packed.w = quant4(v[12], v[13], v[14], v[15], sc);
      }
#pragma unroll 4
      for (int j = 0; j < k; ++j) {
        const size_t sl = (size_t)slot_row[j];
        *reinterpret_cast<uint4*>(xg + sl * H + base) = packed;
        if ((lane & 7) == 0) sxg[sl * ngroups + gi] = sc;
      }
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (threadIdx.x % kQsRowThreads == 0 && active) {
    constexpr int kRowWarps = kQsRowThreads / 32;
    float v = 0.0f;
    for (int w = 0; w < kRowWarps; ++w) v += red[half * kRowWarps + w];
    a.w.gamma[t] = sigmoid_f32(v);
  }
}

// ---- SwiGLU rows with one scale per row ---------------------------------------
// One warp per slot: the row's amax over its I fp32 values, one scale, and the
// e4m3 codes of every value (rows of hf [slots][I] -> hq [slots][I], and the
// row's scale in each of its I/128 entries of sh).
__global__ void __launch_bounds__(256) k_quant_h_rows(const float* __restrict__ hf,
                                                      uint8_t* __restrict__ hq,
                                                      float* __restrict__ sh, int n_rows, int I) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if (r >= n_rows) return;
  const float* row = hf + (size_t)r * I;
  float m = 0.0f;
  for (int c = 4 * lane; c < I; c += 128) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(row + c));
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  const float s = group_scale(warp_max(m));
  for (int c = 4 * lane; c < I; c += 128) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(row + c));
    *reinterpret_cast<uint32_t*>(hq + (size_t)r * I + c) = quant4(v.x, v.y, v.z, v.w, s);
  }
  for (int g = lane; g < I / kGroup; g += 32) sh[(size_t)r * (I / kGroup) + g] = s;
}

// Router weights as three bf16 parts, w = hi + mid + lo exactly (each part
// rounds the remainder of the previous ones; a float's 24 significant bits
// fit in three 8-bit ones).  With bf16 x every product x * part is exact in
// fp32, so the tensor-core GEMM over [hi | mid | lo] gives fp32 logits.
// out [Epad][3H]; rows E..Epad-1 are zero.
__global__ void k_split_router(const float* __restrict__ wr, bf16* __restrict__ out, int E,
                               int Epad, int H) {
  const size_t n = (size_t)Epad * H;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / H), c = (int)(i % H);
    const float w = e < E ? wr[(size_t)e * H + c] : 0.0f;
    const bf16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const bf16 mid = __float2bfloat16_rn(r1);
    const bf16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    bf16* row = out + (size_t)e * 3 * H;
    row[c] = hi;
    row[H + c] = mid;
    row[2 * H + c] = lo;
  }
}

}  // namespace

cudaError_t launch_split_router(const float* wr, bf16* out, int E, int Epad, int H,
                                cudaStream_t s) {
  k_split_router<<<1024, 256, 0, s>>>(wr, out, E, Epad, H);
  return cudaGetLastError();
}

cudaError_t launch_quant_h_rows(const float* hf, uint8_t* hq, float* sh, int n_rows, int I,
                                cudaStream_t s, bool pdl) {
  if (n_rows < 1) return cudaSuccess;
  return launch_pdl(k_quant_h_rows, dim3((n_rows + 7) / 8), dim3(256), 0, s, pdl, hf, hq, sh,
                    n_rows, I);
}

cudaError_t launch_quant_scatter(const KArgs& a, uint8_t* xg, float* sxg, cudaStream_t s,
                                 bool pdl) {
  return launch_pdl(k_quant_scatter, dim3((a.d.T + kQsRows - 1) / kQsRows), dim3(kQsThreads), 0,
                    s, pdl, a, xg, sxg);
}

}  // namespace moe

// Residual add + RMS norm in front of the layer, writing the normed rows and
// their FP8 groups in one pass.
//
// PR #925/#927 commit "add-norm fused with the routed experts' FP8 activation
// quantization": the residual add and RMS norm before the MoE also write the
// normed rows' FP8 groups, rounded exactly as the separate quantisation of the
// bf16 normed rows rounds them.  PR #939 section "Kernel contract": the RMS
// norm is the plain-gamma form; section "Precision": bf16 residual stream.
//
// One CTA per row, 256 threads; a thread owns NC 16-byte chunks of 8 values
// at chunk indices tid, tid + 256, ... (NC = 1 up to hidden 2048, 2 up to
// 4096, 4 up to 8192), so that the kernel keeps only the chunks it needs in
// registers and 8 CTAs fit on an SM: at 1024 rows every row's loads are in
// flight at once.  A 128-value group is 16 consecutive chunks, i.e. one
// half-warp, so a group's amax takes four shuffles.  The bytes are read once
// and written once: the kernel is bound by HBM bandwidth (and, for a handful
// of rows, by launch latency).
#include "addnorm.cuh"
#include "moe_device.cuh"

namespace moe {

namespace {

constexpr int kAnThreads = 256;

__device__ __forceinline__ void unpack8(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    v[2 * i] = __low2float(p);
    v[2 * i + 1] = __high2float(p);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&p);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// h_out may be the residual buffer and xn_out the x buffer (or the other way
// round): every thread reads its own chunks of both inputs before it writes
// the same chunks of the outputs, and no other thread touches them.
template <int NC>
__global__ void __launch_bounds__(kAnThreads, 8 / NC)
    k_add_rmsnorm_quant(const bf16* residual, const bf16* x, const bf16* __restrict__ gamma,
                        float eps, int H, bf16* h_out, bf16* xn_out,
                        uint8_t* __restrict__ codes, float* __restrict__ scales) {
  __shared__ float red[kAnThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nch = H >> 3;  // a multiple of 16
  const size_t row = (size_t)blockIdx.x * H;
  const uint4* rr = reinterpret_cast<const uint4*>(residual + row);
  const uint4* xr = reinterpret_cast<const uint4*>(x + row);

  // every chunk's loads first (once the previous kernel, which may have
  // written the inputs, has completed), then residual + x rounded to bf16
  // (the new residual stream), kept packed
  pdl_wait();
  uint4 ra[NC], xa[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int c = tid + j * kAnThreads;
    if (c < nch) {
      ra[j] = __ldcs(rr + c);
      xa[j] = __ldcs(xr + c);
    }
  }
  pdl_trigger();  // the next kernel's prologue may overlap the rest
  uint4 hp[NC];
  float ss = 0.0f;
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int c = tid + j * kAnThreads;
    if (c < nch) {
      float a[8], b[8];
      unpack8(ra[j], a);
      unpack8(xa[j], b);
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = a[i] + b[i];
      hp[j] = pack8(a);
      reinterpret_cast<uint4*>(h_out + row)[c] = hp[j];
      unpack8(hp[j], a);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(a[i], a[i], ss);
    }
  }

  // sum of squares over the row, in a fixed order (warps 0..7)
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kAnThreads / 32; ++w) tot += red[w];
  const float r = __frsqrt_rn(__fdiv_rn(tot, (float)H) + eps);

  // xn = h * r * gamma in bf16, then the group's scale and codes
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  const int ngroups = H >> 7;
#pragma unroll
  for (int j = 0; j < NC; ++j) {
    const int c = tid + j * kAnThreads;
    if (j * kAnThreads >= nch) break;  // the same for the whole block
    const bool on = c < nch;           // whole half-warps are on or off
    float v[8];
    if (on) {
      float g[8];
      unpack8(__ldg(gr + c), g);
      unpack8(hp[j], v);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = v[i] * r * g[i];
      const uint4 xp = pack8(v);
      reinterpret_cast<uint4*>(xn_out + row)[c] = xp;
      unpack8(xp, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (on) {
      const float s = group_scale(m);
      uint2 q;
      q.x = quant4(v[0], v[1], v[2], v[3], s);
      q.y = quant4(v[4], v[5], v[6], v[7], s);
      reinterpret_cast<uint2*>(codes + row)[c] = q;
      if ((lane & 15) == 0) scales[(size_t)blockIdx.x * ngroups + (c >> 4)] = s;
    }
  }
}

}  // namespace

cudaError_t launch_add_rmsnorm_quant(const bf16* residual, const bf16* x, const bf16* gamma,
                                     float eps, int rows, int H, bf16* h_out, bf16* xn_out,
                                     uint8_t* codes, float* scales, cudaStream_t s, bool pdl) {
  const int nch = H / 8;
  auto* kernel = nch <= kAnThreads       ? k_add_rmsnorm_quant<1>
                 : nch <= 2 * kAnThreads ? k_add_rmsnorm_quant<2>
                                         : k_add_rmsnorm_quant<4>;
  return launch_pdl(kernel, dim3(rows), dim3(kAnThreads), 0, s, pdl, residual, x, gamma, eps, H,
                    h_out, xn_out, codes, scales);
}

}  // namespace moe

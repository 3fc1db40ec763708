// moe_route_static: the router (logits, top-k, renormalised softmax) with its
// logits scratch in a fixed device array of this library instead of a
// context's workspace, so the call allocates nothing.
//
// Router: PR #939 "Fish Audio Drama 3 text to speech on one CUDA GPU",
// section "What it adds" (the router) and section "Fidelity against the
// PyTorch oracle" (near-tied 8th/9th experts).  The call is a library
// convenience; the pages define no such entry point.
#include <cudaTypedefs.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

// Router logits of one call, fp32 [rows][n_experts]; 1 MiB per device.
static __device__ __align__(256) float g_route_scratch[MOE_ROUTE_STATIC_MAX_LOGITS];

constexpr int kMaxDevices = 64;

// The scratch's device address per device ordinal, with the context it was
// looked up in: after a device reset the primary context is new, the library's
// device code is loaded again (possibly elsewhere), and the address is looked
// up again.
struct ScratchAddr {
  CUcontext ctx = nullptr;
  float* ptr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

PFN_cuCtxGetCurrent_v4000 ctx_getter() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    cudaGetLastError();
  });
  return fn;
}

// Address of this device's copy of the scratch, looked up once per device
// and context.  With no context current on the calling thread yet, the
// look-up itself makes the device's primary context current.
int scratch_for(int device, float** out) {
  if (device < 0 || device >= kMaxDevices) return MOE_ERR_UNSUPPORTED_SHAPE;
  const PFN_cuCtxGetCurrent_v4000 get_ctx = ctx_getter();
  CUcontext ctx = nullptr;
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr& e = g_scratch[device];
  if (!ctx || e.ctx != ctx || !e.ptr) {
    float* p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_route_scratch) != cudaSuccess ||
        !p) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    if (!ctx && (get_ctx(&ctx) != CUDA_SUCCESS || !ctx)) return MOE_ERR_CUDA;
    e.ctx = ctx;
    e.ptr = p;
  }
  *out = e.ptr;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_route_static(const void* x, const float* router, int rows, int hidden,
                                int n_experts, int top_k, int32_t* idx, float* w,
                                void* stream) {
  if (rows < 0) return MOE_ERR_INVALID_ARG;
  if (hidden <= 0 || hidden % kGroup != 0 || top_k < 1 || top_k > kMaxTopK ||
      n_experts < top_k || n_experts > kMaxExperts)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)rows * n_experts > MOE_ROUTE_STATIC_MAX_LOGITS) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!x || !router || !idx || !w) return MOE_ERR_INVALID_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  float* scratch = nullptr;
  const int rc = scratch_for(device, &scratch);
  if (rc != MOE_OK) return rc;

  KArgs a = {};
  a.d.T = rows;
  a.d.H = hidden;
  a.d.E = n_experts;
  a.d.k = top_k;
  a.L.wr = router;
  a.w.logits = scratch;
  a.w.idx = idx;
  a.w.wts = w;
  a.x = static_cast<const bf16*>(x);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_router(a, s) != cudaSuccess || launch_topk(a, s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

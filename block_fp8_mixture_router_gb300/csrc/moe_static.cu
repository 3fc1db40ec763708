// moe_route_static: the router (logits, top-k, renormalised softmax) with its
// logits scratch in a fixed device array of this library instead of a
// context's workspace, so the call allocates nothing.
//
// Router: PR #939 "Fish Audio Drama 3 text to speech on one CUDA GPU",
// section "What it adds" (the router) and section "Fidelity against the
// PyTorch oracle" (near-tied 8th/9th experts).  The call is a library
// convenience; the pages define no such entry point.
#include <atomic>

#include "moe_internal.cuh"

namespace moe {
namespace {

// Router logits of one call, fp32 [rows][n_experts]; 1 MiB per device.
static __device__ __align__(256) float g_route_scratch[MOE_ROUTE_STATIC_MAX_LOGITS];

constexpr int kMaxDevices = 64;
std::atomic<float*> g_scratch_addr[kMaxDevices];

// Address of this device's copy of the scratch, looked up once per device.
int scratch_for(int device, float** out) {
  if (device < 0 || device >= kMaxDevices) return MOE_ERR_UNSUPPORTED_SHAPE;
  float* p = g_scratch_addr[device].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_route_scratch) != cudaSuccess ||
        !p) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_addr[device].store(p, std::memory_order_release);
  }
  *out = p;
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

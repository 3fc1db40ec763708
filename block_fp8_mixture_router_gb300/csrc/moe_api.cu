// C ABI of the block-FP8 MoE layer: context, weight loading, forward.
//
// Interface style follows the pages: refuse unsupported shapes when the
// layer is opened (PR #939 section "What it adds": config.zig "checks every
// number the kernels assume and refuses any other checkpoint shape"),
// caller-owned buffers, an allocation cap that is checked before anything is
// allocated (PR #925, allocation-limit commit), and named error values instead
// of traps.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "addnorm.cuh"
#include "moe_internal.cuh"

using namespace moe;

struct moe_ctx {
  moe_config cfg;
  int device = 0;
  int sm_count = 0;
  bool loaded = false;
  int opt_path = 0;
  int opt_pdl = 1;
  int opt_poll_limit = 0;  // status[kPollLimitWord]; 0 = the kernels' default
  int opt_invariant = 0;   // batch-invariant rows: the grouped kernels for every T
  int opt_router_bf16 = 0; // route on logits rounded to bf16
  size_t row_smem = 0;     // one-row decode kernel: shared memory per CTA, 0 = unavailable
  size_t rows_smem = 0;    // 2..16-row decode kernel: shared memory per CTA, 0 = unavailable
  cudaStream_t last_stream = nullptr;
  std::vector<void*> allocs;
  // the value buffers of the workspace: every byte a forward reads from them
  // it wrote earlier in the same call (moe_debug_poison_workspace fills them)
  std::vector<std::pair<void*, size_t>> data_regions;
  DevLayer L{};
  DevWork w{};
  bf16* stage_x = nullptr;
  bf16* stage_y = nullptr;
  // prompt path on tcgen05: launch arguments with the fixed tensor maps
  bool tc_ok = false;
  TcGemm tc[5] = {};
  size_t tc_smem[5] = {};
  bf16* router3 = nullptr; // router as bf16 parts [Epad][3H] (hi | mid | lo)
  float* logits_part = nullptr;  // router K-split partial logits [splits][rows][E]
  int part_rows = 0;             // splits x rows the partial buffer holds
  uint8_t* xg = nullptr;   // e4m3 activations in slot order [max_rows*k][H]
  float* sxg = nullptr;    // their scales [max_rows*k][H/128]
  // prompt path: the shared expert runs on a second stream, forked from and
  // joined back into the caller's stream within each forward
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // the most recent forward, for moe_forward_codes: its rows (0 = none, or a
  // later call rewrote the workspace) and where its x codes live
  int fwd_rows = 0;
  bool fwd_slot_order = false;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

bool config_supported(const moe_config* c) {
  if (c->hidden <= 0 || c->hidden % kGroup) return false;
  if (c->inter <= 0 || c->inter % kGroup) return false;
  if (c->shared_inter <= 0 || c->shared_inter % kGroup) return false;
  if (c->top_k < 1 || c->top_k > kMaxTopK) return false;
  if (c->n_experts < c->top_k || c->n_experts > kMaxExperts) return false;
  if (c->act_group != kGroup && c->act_group != c->hidden) return false;
  if (c->max_rows < 1 || c->max_rows > 65536) return false;
  if (c->hidden > 65536 || c->inter > 65536 || c->shared_inter > 65536) return false;
  return true;
}

// One activation scale per row of x and of each SwiGLU row (act_group ==
// hidden) instead of one per 1 x 128 group.
bool per_row_scales(const moe_config& c) { return c.act_group == c.hidden && c.hidden > kGroup; }

// Byte layout of everything a context allocates, in allocation order.
struct Plan {
  size_t sizes[48];
  int n = 0;
  size_t total = 0;
  size_t add(size_t b) {
    b = (b + 255) & ~(size_t)255;
    sizes[n++] = b;
    total += b;
    return b;
  }
};

// K splits of the tensor-core router in batch-invariant mode, whatever the
// row count: a row's logits are then the same partial sums added in the same
// order at every T.
constexpr int kInvariantSplits = 4;

// Rows (splits x rows) of the router's partial-logit buffer: up to 16 splits
// while splits x rows stays within 16384, and always kInvariantSplits splits
// of max_rows.
size_t router_part_rows(const moe_config* c) {
  return std::max<size_t>(std::min<size_t>(16384, 16 * (size_t)c->max_rows),
                          (size_t)kInvariantSplits * c->max_rows);
}

// K splits of the tensor-core router for T rows: enough items to give every
// SM one, within the partial buffer.
int router_splits(int sm, int T, int n_f, int n_k, int part_rows) {
  const int base = (T + 127) / 128 * n_f;
  int ks = (sm + base - 1) / base;
  ks = std::min(ks, std::min(16, n_k));
  while (ks > 1 && (size_t)ks * T > (size_t)part_rows) --ks;
  return std::max(ks, 1);
}

Plan make_plan(const moe_config* c) {
  Plan p;
  const size_t H = c->hidden, E = c->n_experts, k = c->top_k, I = c->inter, Is = c->shared_inter;
  const size_t T = c->max_rows, G = kGroup, W = (T + 31) / 32;
  const size_t MC = (size_t)max_chunks((int)T, (int)k, (int)E);
  // weights
  p.add(E * 2 * I * H);                   // 0 w13
  p.add(E * (2 * I / G) * (H / G) * 4);   // 1 s13
  p.add(E * H * I);                       // 2 w2
  p.add(E * (H / G) * (I / G) * 4);       // 3 s2
  p.add(E * H * 4);                       // 4 router
  p.add(2 * Is * H * 2);                  // 5 ws13
  p.add(H * Is * 2);                      // 6 ws2
  p.add(H * 2);                           // 7 gate
  // workspace
  p.add(T * E * 4);                       // 8 logits
  p.add(T * k * 4);                       // 9 idx
  p.add(T * k * 4);                       // 10 wts
  p.add(T * H);                           // 11 xq
  p.add(T * (H / G) * 4);                 // 12 sx
  p.add(T * 4);                           // 13 gamma
  p.add(E * W * 4);                       // 14 bitmap
  p.add(E * W * 4);                       // 15 wprefix
  p.add(E * 4);                           // 16 counts
  p.add((E + 1) * 4);                     // 17 off
  p.add(T * k * 4);                       // 18 pair_of_slot
  p.add(T * k * 4);                       // 19 slot_of_pair
  p.add(MC * 16);                         // 20 chunks
  p.add(16);                              // 21 n_chunks
  p.add(T * k * I * 4);                   // 22 hbuf
  p.add(T * k * I);                       // 23 hq
  p.add(T * k * (I / G) * 4);             // 24 sh
  p.add(MC * (I / G) * 4);                // 25 gcount
  p.add(T * Is * 2);                      // 26 hs
  p.add(T * k * H * 2);                   // 27 dbuf
  p.add(T * H * 2);                       // 28 ds
  p.add(64);                              // 29 status and barrier counters
  p.add(T * H * 2);                       // 30 stage_x
  p.add(T * H * 2);                       // 31 stage_y
  p.add(kDecodeRows * E * 8);             // 32 tagged decode logits
  p.add(T * k * H);                       // 33 xg (slot order)
  p.add(T * k * (H / G) * 4);             // 34 sxg
  p.add(((E + 127) / 128) * 128 * 3 * H * 2);  // 35 router3
  p.add(router_part_rows(c) * E * 4);     // 36 router partial logits
  p.add(T * k * 4);                       // 37 schedule: rank in block
  p.add(((T + kSchedRows - 1) / kSchedRows) * E * 4);  // 38 schedule: rows per expert per block
  p.add(kDecodeRows * (k * I + k * H + Is + H) * 8);  // 39 decode exchange words
  return p;
}

void free_all(moe_ctx* c) {
  for (void* ptr : c->allocs) cudaFree(ptr);
  c->allocs.clear();
  if (c->ev_join) cudaEventDestroy(c->ev_join);
  if (c->ev_fork) cudaEventDestroy(c->ev_fork);
  if (c->side) cudaStreamDestroy(c->side);
  c->ev_join = c->ev_fork = nullptr;
  c->side = nullptr;
}

int check_launch(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

KArgs make_args(moe_ctx* c, const void* x, void* y, int T) {
  KArgs a = {};  // a.an zero: no add-norm in front of the layer
  a.d = Dims{T, c->cfg.hidden, c->cfg.n_experts, c->cfg.top_k, c->cfg.inter, c->cfg.shared_inter,
             c->opt_router_bf16, per_row_scales(c->cfg) ? 1 : 0};
  a.L = c->L;
  a.w = c->w;
  a.x = static_cast<const bf16*>(x);
  a.y = static_cast<bf16*>(y);
  return a;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

bool use_decode(const moe_ctx* c, int T);
bool use_row(const moe_ctx* c, int T);
bool use_rows(const moe_ctx* c, int T);
bool use_tc(const moe_ctx* c, int T);
bool router_args(const moe_ctx* c, const void* x, int T, TcGemm* rt, int* grid);
cudaError_t launch_topk_after_router(const KArgs& a, const moe_ctx* c, const TcGemm& rt,
                                     cudaStream_t s, bool pdl);

// Routing with the kernels the forward of T rows would use (the persistent
// decode kernel routes inside the layer: run the layer into the staging
// output and keep its published routing).
int run_router_and_quant(moe_ctx* c, const KArgs& a, cudaStream_t s) {
  if (use_decode(c, a.d.T) && use_row(c, a.d.T)) {
    KArgs b = a;
    b.y = c->stage_y;
    return launch_decode_row(b, c->sm_count, c->row_smem, c->opt_pdl != 0, s) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  }
  if (use_decode(c, a.d.T) && use_rows(c, a.d.T)) {
    KArgs b = a;
    b.y = c->stage_y;
    return launch_decode_rows(b, c->sm_count, c->rows_smem, c->opt_pdl != 0, s) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  }
  if (use_decode(c, a.d.T))
    return launch_route_decode(a, c->opt_pdl != 0, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  if (use_tc(c, a.d.T)) {
    TcGemm rt;
    int g_rt = 0;
    if (!router_args(c, a.x, a.d.T, &rt, &g_rt)) return MOE_ERR_CUDA;
    if (launch_tc_gemm(kTcRouter, rt, g_rt, c->tc_smem[kTcRouter], s) != cudaSuccess ||
        launch_topk_after_router(a, c, rt, s, false) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (launch_router(a, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_quant_gamma(a, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_topk(a, s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

// Records an event after each launch when profiling (names/events non-null).
struct StageRec {
  cudaEvent_t* ev = nullptr;
  const char** names = nullptr;
  int cap = 0;
  int n = 0;
  bool mark(const char* name, cudaStream_t s) {
    if (!ev) return true;
    if (n >= cap) return true;
    names[n] = name;
    return cudaEventRecord(ev[++n], s) == cudaSuccess;
  }
};

#define LAUNCH(expr, name)                                 \
  do {                                                     \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA;        \
    if (rec && !rec->mark(name, s)) return MOE_ERR_CUDA;   \
  } while (0)

// The decode kernels serve rows <= kDecodeRows for hidden sizes up to 4096.
// 2..kRowsAuto rows on the role-split multi-row kernel unless another kernel
// is asked for.  Above that the grouped tcgen05 kernels are faster on GB300
// than both it and the three chained decode kernels: per layer, 52.9 against
// 59.8 us at 5 rows, 53.7 against 54.7 us (chained) at 6, 57.0 against
// 68.5 us at 11 and 59.4 against 77.3 us at 16; at 4 rows they tie.
constexpr int kRowsAuto = 4;

bool use_decode(const moe_ctx* c, int T) {
  if (c->opt_path == 2 || c->opt_path == 4 || c->opt_invariant) return false;
  if (T > kDecodeRows || c->cfg.hidden > 4096) return false;
  // one scale per row: only the role-split decode kernels quantise whole rows
  if (per_row_scales(c->cfg)) return use_row(c, T) || use_rows(c, T);
  // automatic choice: the chained kernels only where the tcgen05 ones are
  // not available
  if ((c->opt_path == 0 || c->opt_path == 1) && T > kRowsAuto && c->tc_ok) return false;
  return true;
}

// One row on the role-split one-row kernel unless another decode kernel is
// asked for.
bool use_row(const moe_ctx* c, int T) {
  return T == 1 && c->row_smem > 0 && (c->opt_path == 0 || c->opt_path == 1);
}

bool use_rows(const moe_ctx* c, int T) {
  if (T < 2 || T > kDecodeRows || c->rows_smem <= 0) return false;
  return c->opt_path == 6 ||
         ((c->opt_path == 0 || c->opt_path == 1) && (T <= kRowsAuto || per_row_scales(c->cfg)));
}

// Tensor maps and launch arguments of the four tcgen05 GEMMs.  The weight
// and workspace addresses are fixed for the context's life; only the shared
// expert's input map (x) is encoded per forward.  Leaves tc_ok false (the
// grouped mma.sync kernels then serve every prompt) if any map or the shared
// memory a CTA needs is not available.
void setup_tc(moe_ctx* c) {
  const moe_config& f = c->cfg;
  const uint64_t H = f.hidden, E = f.n_experts, k = f.top_k, I = f.inter, Is = f.shared_inter;
  const uint64_t R = (uint64_t)f.max_rows * k;
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device) !=
      cudaSuccess) {
    cudaGetLastError();
    return;
  }
  if (H / kGroup > 32 || I / kGroup > 32) return;  // activation scales staged per tile
  if (H % (2 * kGroup)) return;                     // down items: two output tiles
  TcGemm* g = c->tc;
  const uint64_t Epad = (E + 127) / 128 * 128;
  for (int i = 0; i < 5; ++i) {
    g[i].E = (int)E;
    g[i].status = c->w.status;
    g[i].counts = c->w.counts;
    g[i].off = c->w.off;
  }
  bool ok = true;
  // routed gate/up: W13 [E*2I][H] x xg [slots][H]
  ok &= make_tc_map(&g[kTcRoutedGateUp].a, false, c->L.w13, E * 2 * I, H, 128);
  ok &= make_tc_map(&g[kTcRoutedGateUp].b, false, c->xg, R, H, 16);
  ok &= make_tc_map(&g[kTcRoutedGateUp].bt, false, c->xg, R, H,
                    (uint32_t)tc_gemm_tile_rows(kTcRoutedGateUp));
  g[kTcRoutedGateUp].n_k = (int)(H / kGroup);
  g[kTcRoutedGateUp].n_f = (int)(I / kGroup);
  g[kTcRoutedGateUp].a_rows_e = (int)(2 * I);
  g[kTcRoutedGateUp].up_rows = (int)I;
  g[kTcRoutedGateUp].ldo = (int)I;
  g[kTcRoutedGateUp].sa = c->L.s13;
  g[kTcRoutedGateUp].sb = c->sxg;
  g[kTcRoutedGateUp].hq = c->w.hq;
  g[kTcRoutedGateUp].sh = c->w.sh;
  g[kTcRoutedGateUp].hf = per_row_scales(f) ? c->w.hbuf : nullptr;
  // routed down: W2 [E*H][I] x hq [slots][I]
  ok &= make_tc_map(&g[kTcRoutedDown].a, false, c->L.w2, E * H, I, 128);
  ok &= make_tc_map(&g[kTcRoutedDown].b, false, c->w.hq, R, I, 16);
  ok &= make_tc_map(&g[kTcRoutedDown].bt, false, c->w.hq, R, I,
                    (uint32_t)tc_gemm_tile_rows(kTcRoutedDown));
  g[kTcRoutedDown].n_k = (int)(I / kGroup);
  g[kTcRoutedDown].n_f = (int)(H / (2 * kGroup));  // two adjacent output tiles per item
  g[kTcRoutedDown].f_rows = 2 * kGroup;
  g[kTcRoutedDown].up_rows = kGroup;
  g[kTcRoutedDown].a_rows_e = (int)H;
  g[kTcRoutedDown].ldo = (int)H;
  g[kTcRoutedDown].sa = c->L.s2;
  g[kTcRoutedDown].sb = c->w.sh;
  g[kTcRoutedDown].out = c->w.dbuf;
  // shared gate/up: Ws13 [2Is][H] x x [rows][H] (x's map is set per forward)
  ok &= make_tc_map(&g[kTcSharedGateUp].a, true, c->L.ws13, 2 * Is, H, 128);
  g[kTcSharedGateUp].n_k = (int)(H / 64);
  g[kTcSharedGateUp].n_f = (int)(Is / kGroup);
  g[kTcSharedGateUp].up_rows = (int)Is;
  g[kTcSharedGateUp].ldo = (int)Is;
  g[kTcSharedGateUp].out = c->w.hs;
  // shared down: Ws2 [H][Is] x hs [rows][Is]
  ok &= make_tc_map(&g[kTcSharedDown].a, true, c->L.ws2, H, Is, 128);
  ok &= make_tc_map(&g[kTcSharedDown].b, true, c->w.hs, (uint64_t)f.max_rows, Is, 16);
  ok &= make_tc_map(&g[kTcSharedDown].bt, true, c->w.hs, (uint64_t)f.max_rows, Is,
                    (uint32_t)tc_gemm_tile_rows(kTcSharedDown));
  g[kTcSharedDown].n_k = (int)(Is / 64);
  g[kTcSharedDown].n_f = (int)(H / kGroup);
  g[kTcSharedDown].ldo = (int)H;
  g[kTcSharedDown].out = c->w.ds;
  // router: [hi | mid | lo] [Epad][3H] x x [rows][H] (x's map per forward)
  ok &= make_tc_map(&g[kTcRouter].a, true, c->router3, Epad, 3 * H, 128);
  g[kTcRouter].n_k = (int)(3 * H / 64);
  g[kTcRouter].n_f = (int)(Epad / kGroup);
  g[kTcRouter].ldo = (int)E;
  g[kTcRouter].outf = c->w.logits;
  for (int i = 0; i < 5; ++i) {
    g[i].b_kwrap = g[i].n_k;
    g[i].ksplit = 1;
    if (i != kTcRoutedDown) g[i].f_rows = kGroup;
  }
  g[kTcRouter].b_kwrap = (int)(H / 64);
  for (int i = 0; i < 5 && ok; ++i) {
    c->tc_smem[i] = tc_gemm_smem(i, g[i].n_k);
    ok &= c->tc_smem[i] <= (size_t)optin && setup_tc_gemm(i, c->tc_smem[i]) == cudaSuccess;
  }
  cudaGetLastError();
  c->tc_ok = ok;
}

// Rows above the decode range run on the tcgen05 kernels unless the
// warp-MMA kernels are asked for or the shape has no tcgen05 set-up.
bool use_tc(const moe_ctx* c, int T) {
  return !use_decode(c, T) && c->tc_ok && c->opt_path != 4;
}

// Router launch arguments for T rows of x: the input's tensor map and the K
// splits.  Returns false if the map cannot be encoded.
bool router_args(const moe_ctx* c, const void* x, int T, TcGemm* rt, int* grid) {
  *rt = c->tc[kTcRouter];
  if (!make_tc_map(&rt->b, true, x, (uint64_t)T, (uint64_t)c->cfg.hidden, 16) ||
      !make_tc_map(&rt->bt, true, x, (uint64_t)T, (uint64_t)c->cfg.hidden,
                   (uint32_t)tc_gemm_tile_rows(kTcRouter)))
    return false;
  rt->T = T;
  rt->ksplit = c->opt_invariant ? std::min(kInvariantSplits, rt->n_k)
                                : router_splits(c->sm_count, T, rt->n_f, rt->n_k, c->part_rows);
  rt->outf = rt->ksplit > 1 ? c->logits_part : c->w.logits;
  *grid = std::min(c->sm_count, (T + 127) / 128 * rt->n_f * rt->ksplit);
  return true;
}

cudaError_t launch_topk_after_router(const KArgs& a, const moe_ctx* c, const TcGemm& rt,
                                     cudaStream_t s, bool pdl) {
  return rt.ksplit > 1 ? launch_topk_splits(a, c->logits_part, rt.ksplit, s, pdl)
                       : launch_topk(a, s, pdl);
}

// pre_q: w.xq / w.sx already hold x's codes (written by the add-norm kernel
// of moe_forward_addnorm); the grouped path then scatters them as they are.
int run_forward(moe_ctx* c, const void* x, void* y, int T, cudaStream_t s,
                StageRec* rec = nullptr, bool pre_q = false) {
  KArgs a = make_args(c, x, y, T);
  a.an.pre_q = pre_q ? 1 : 0;
  c->fwd_rows = T;
  c->fwd_slot_order = use_tc(c, T);
  const int grid = 2 * c->sm_count;
  if (use_decode(c, T) && use_row(c, T)) {
    LAUNCH(launch_decode_row(a, c->sm_count, c->row_smem, c->opt_pdl != 0, s), "decode_row");
    return MOE_OK;
  }
  if (use_decode(c, T) && use_rows(c, T)) {
    LAUNCH(launch_decode_rows(a, c->sm_count, c->rows_smem, c->opt_pdl != 0, s), "decode_rows");
    return MOE_OK;
  }
  if (use_decode(c, T)) {
    const bool pdl = c->opt_pdl != 0;
    LAUNCH(launch_route_decode(a, pdl, s), "route_decode");
    LAUNCH(launch_gateup_decode(a, grid, pdl, s), "gateup_decode");
    LAUNCH(launch_down_combine_decode(a, pdl, s), "down_combine_decode");
    return MOE_OK;
  }
  if (use_tc(c, T)) {
    TcGemm rt;
    int g_rt = 0;
    if (!router_args(c, x, T, &rt, &g_rt)) return MOE_ERR_CUDA;
    TcGemm sgu = c->tc[kTcSharedGateUp];
    sgu.b = rt.b;
    sgu.bt = rt.bt;  // the router's and the shared gate/up's tiles have the same rows
    TcGemm sdn = c->tc[kTcSharedDown];
    sgu.T = sdn.T = T;
    const int tiles = (T + 127) / 128;
    const int g_sgu = std::min(c->sm_count, tiles * sgu.n_f);
    const int g_sdn = std::min(c->sm_count, tiles * sdn.n_f);
    // The shared expert needs only x: it runs on the side stream alongside
    // the routing kernels and the routed GEMMs, and the combine waits for
    // it.  A profiled forward keeps every kernel on the caller's stream so
    // that each stage is timed alone.
    const bool fork = rec == nullptr && c->side != nullptr;
    if (fork) {
      if (cudaEventRecord(c->ev_fork, s) != cudaSuccess ||
          cudaStreamWaitEvent(c->side, c->ev_fork, 0) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (launch_tc_gemm(kTcSharedGateUp, sgu, g_sgu, c->tc_smem[kTcSharedGateUp], c->side) !=
              cudaSuccess ||
          launch_tc_gemm(kTcSharedDown, sdn, g_sdn, c->tc_smem[kTcSharedDown], c->side) !=
              cudaSuccess ||
          cudaEventRecord(c->ev_join, c->side) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else {
      LAUNCH(launch_tc_gemm(kTcSharedGateUp, sgu, g_sgu, c->tc_smem[kTcSharedGateUp], s),
             "shared_gateup_tc");
      LAUNCH(launch_tc_gemm(kTcSharedDown, sdn, g_sdn, c->tc_smem[kTcSharedDown], s),
             "shared_down_tc");
    }
    // the main stream's kernels are chained by programmatic dependent launch:
    // each waits for its predecessor before touching its data, and its
    // prologue (barriers, tensor memory, descriptor prefetch) overlaps the
    // predecessor's tail
    const bool pdl = c->opt_pdl != 0;
    LAUNCH(launch_tc_gemm(kTcRouter, rt, g_rt, c->tc_smem[kTcRouter], s, pdl), "router_tc");
    LAUNCH(launch_topk_after_router(a, c, rt, s, pdl), "topk");
    LAUNCH(launch_schedule(a, s, pdl), "schedule");
    LAUNCH(launch_quant_scatter(a, c->xg, c->sxg, s, pdl), "quant_scatter");
    LAUNCH(launch_tc_gemm(kTcRoutedGateUp, c->tc[kTcRoutedGateUp], c->sm_count,
                          c->tc_smem[kTcRoutedGateUp], s, pdl),
           "gateup_tc");
    if (per_row_scales(c->cfg))
      LAUNCH(launch_quant_h_rows(c->w.hbuf, c->w.hq, c->w.sh, T * c->cfg.top_k, c->cfg.inter, s,
                                 pdl),
             "quant_h_rows");
    LAUNCH(launch_tc_gemm(kTcRoutedDown, c->tc[kTcRoutedDown], c->sm_count,
                          c->tc_smem[kTcRoutedDown], s, pdl),
           "down_tc");
    if (fork && cudaStreamWaitEvent(s, c->ev_join, 0) != cudaSuccess) return MOE_ERR_CUDA;
    // after the join the combine waits on the side stream as well: plain launch
    LAUNCH(launch_combine(a, s, pdl && !fork), "combine");
    return MOE_OK;
  }
  LAUNCH(launch_router(a, s), "router");
  LAUNCH(launch_quant_gamma(a, s), "quant_gamma");
  LAUNCH(launch_topk(a, s), "topk");
  LAUNCH(launch_schedule(a, s), "schedule");
  LAUNCH(launch_gateup(a, grid, s), "gateup");
  LAUNCH(launch_down(a, grid, s), "down");
  LAUNCH(launch_combine(a, s), "combine");
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_NOT_LOADED: return "weights not loaded";
    case MOE_ERR_ALLOC_LIMIT: return "allocation would exceed the workspace cap";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int moe_required_bytes(const moe_config* cfg, size_t* bytes) {
  if (!cfg || !bytes) return MOE_ERR_INVALID_ARG;
  if (!config_supported(cfg)) return MOE_ERR_UNSUPPORTED_SHAPE;
  *bytes = make_plan(cfg).total;
  return MOE_OK;
}

int moe_create(const moe_config* cfg, int device, moe_ctx** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || device < 0) return MOE_ERR_INVALID_ARG;
  if (!config_supported(cfg)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const Plan plan = make_plan(cfg);
  if (cfg->workspace_cap_bytes && plan.total > cfg->workspace_cap_bytes) return MOE_ERR_ALLOC_LIMIT;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  DeviceGuard guard(device);
  if (!guard.ok) return MOE_ERR_CUDA;
  moe_ctx* c = new (std::nothrow) moe_ctx();
  if (!c) return MOE_ERR_CUDA;
  c->cfg = *cfg;
  c->device = device;
  if (cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    delete c;
    return MOE_ERR_CUDA;
  }
  void* ptrs[48];
  for (int i = 0; i < plan.n; ++i) {
    if (cudaMalloc(&ptrs[i], plan.sizes[i]) != cudaSuccess) {
      cudaGetLastError();
      free_all(c);
      delete c;
      return MOE_ERR_CUDA;
    }
    c->allocs.push_back(ptrs[i]);
  }
  // (values only: logits, weights, codes, scales, activations, outputs.  The
  // index arrays are left out: a wrong value there is a wrong address.)
  for (int i : {8, 10, 11, 12, 13, 22, 23, 24, 26, 27, 28, 30, 31, 33, 34, 36})
    c->data_regions.emplace_back(ptrs[i], plan.sizes[i]);
  c->L.w13 = (const uint8_t*)ptrs[0];
  c->L.s13 = (const float*)ptrs[1];
  c->L.w2 = (const uint8_t*)ptrs[2];
  c->L.s2 = (const float*)ptrs[3];
  c->L.wr = (const float*)ptrs[4];
  c->L.ws13 = (const bf16*)ptrs[5];
  c->L.ws2 = (const bf16*)ptrs[6];
  c->L.gate = (const bf16*)ptrs[7];
  DevWork& w = c->w;
  w.logits = (float*)ptrs[8];
  w.idx = (int*)ptrs[9];
  w.wts = (float*)ptrs[10];
  w.xq = (uint8_t*)ptrs[11];
  w.sx = (float*)ptrs[12];
  w.gamma = (float*)ptrs[13];
  w.bitmap = (uint32_t*)ptrs[14];
  w.wprefix = (int*)ptrs[15];
  w.counts = (int*)ptrs[16];
  w.off = (int*)ptrs[17];
  w.pair_of_slot = (int*)ptrs[18];
  w.slot_of_pair = (int*)ptrs[19];
  w.chunks = (int4*)ptrs[20];
  w.n_chunks = (int*)ptrs[21];
  w.hbuf = (float*)ptrs[22];
  w.hq = (uint8_t*)ptrs[23];
  w.sh = (float*)ptrs[24];
  w.gcount = (int*)ptrs[25];
  w.hs = (bf16*)ptrs[26];
  w.dbuf = (bf16*)ptrs[27];
  w.ds = (bf16*)ptrs[28];
  w.status = (int*)ptrs[29];
  w.done = w.status + 1;
  w.tlog = (unsigned long long*)ptrs[32];
  c->stage_x = (bf16*)ptrs[30];
  c->stage_y = (bf16*)ptrs[31];
  c->xg = (uint8_t*)ptrs[33];
  c->sxg = (float*)ptrs[34];
  c->router3 = (bf16*)ptrs[35];
  c->logits_part = (float*)ptrs[36];
  w.sched_rank = (int*)ptrs[37];
  w.sched_blk = (int*)ptrs[38];
  w.xw = (unsigned long long*)ptrs[39];
  c->part_rows = (int)router_part_rows(cfg);
  if (cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return MOE_ERR_CUDA;
  }
  // counters start at zero and are reset by the kernels that use them
  if (cudaMemset(w.gcount, 0, plan.sizes[25]) != cudaSuccess ||
      cudaMemset(w.status, 0, plan.sizes[29]) != cudaSuccess ||
      cudaMemset(w.n_chunks, 0, plan.sizes[21]) != cudaSuccess ||
      cudaMemset(w.tlog, 0, plan.sizes[32]) != cudaSuccess ||
      cudaMemset(w.xw, 0, plan.sizes[39]) != cudaSuccess) {
    free_all(c);
    delete c;
    return MOE_ERR_CUDA;
  }
  // role-split decode kernels: one CTA per SM, roles fixed by the shape
  {
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) ==
        cudaSuccess) {
      const int E = cfg->n_experts;
      // one-row kernel: every SM one CTA, roles fixed by the shape
      const size_t rs = decode_row_smem(c->sm_count, cfg->hidden, E, cfg->top_k, cfg->inter,
                                        cfg->shared_inter);
      if (decode_row_fits(c->sm_count, cfg->hidden, E, cfg->top_k, cfg->inter, cfg->shared_inter,
                          (size_t)optin) &&
          setup_decode_row(rs) == cudaSuccess)
        c->row_smem = rs;
      const size_t rr = decode_rows_smem(cfg->hidden);
      if (decode_rows_fits(c->sm_count, cfg->hidden, E, cfg->top_k, cfg->inter, cfg->shared_inter,
                           (size_t)optin) &&
          setup_decode_rows(rr) == cudaSuccess)
        c->rows_smem = rr;
    }
    cudaGetLastError();
  }
  if (setup_schedule() != cudaSuccess) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return MOE_ERR_CUDA;
  }
  setup_tc(c);
  // one scale per row needs the tcgen05 kernels above 16 rows (the warp-MMA
  // and chained decode kernels quantise 1 x 128 groups only)
  if (per_row_scales(*cfg) && !c->tc_ok) {
    free_all(c);
    delete c;
    return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  *out = c;
  return MOE_OK;
}

int moe_load_weights(moe_ctx* c, const moe_weights* wt, int pointers_on_device, void* stream) {
  if (!c || !wt) return MOE_ERR_INVALID_ARG;
  if (!wt->w13 || !wt->s13 || !wt->w2 || !wt->s2 || !wt->router || !wt->ws13 || !wt->ws2 ||
      !wt->shared_gate)
    return MOE_ERR_INVALID_ARG;
  if (pointers_on_device != 0 && pointers_on_device != 1) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  const Plan plan = make_plan(&c->cfg);
  const size_t H = c->cfg.hidden, E = c->cfg.n_experts, I = c->cfg.inter,
               Is = c->cfg.shared_inter, G = kGroup;
  const size_t n13 = E * (2 * I / G) * (H / G), n2 = E * (H / G) * (I / G);
  // scales must be finite and positive: check them on the host first
  std::vector<float> s13(n13), s2(n2);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(s13.data(), wt->s13, n13 * 4, cudaMemcpyDefault, s) != cudaSuccess ||
      cudaMemcpyAsync(s2.data(), wt->s2, n2 * 4, cudaMemcpyDefault, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  for (float v : s13)
    if (!(v > 0.0f) || !isfinite(v)) return MOE_ERR_INVALID_ARG;
  for (float v : s2)
    if (!(v > 0.0f) || !isfinite(v)) return MOE_ERR_INVALID_ARG;
  (void)plan;
  struct Cp { void* dst; const void* src; size_t n; } cps[] = {
      {(void*)c->L.w13, wt->w13, E * 2 * I * H},
      {(void*)c->L.s13, wt->s13, n13 * 4},
      {(void*)c->L.w2, wt->w2, E * H * I},
      {(void*)c->L.s2, wt->s2, n2 * 4},
      {(void*)c->L.wr, wt->router, E * H * 4},
      {(void*)c->L.ws13, wt->ws13, 2 * Is * H * 2},
      {(void*)c->L.ws2, wt->ws2, H * Is * 2},
      {(void*)c->L.gate, wt->shared_gate, H * 2},
  };
  for (const Cp& cp : cps)
    if (cudaMemcpyAsync(cp.dst, cp.src, cp.n, cudaMemcpyDefault, s) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  // the router as exact bf16 parts for the tensor-core router
  const int Epad = (int)((E + 127) / 128 * 128);
  if (launch_split_router(c->L.wr, c->router3, (int)E, Epad, (int)H, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  c->loaded = true;
  return MOE_OK;
}

int moe_forward(moe_ctx* c, const void* x, void* y, int rows, void* stream) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (rows < 0) return MOE_ERR_INVALID_ARG;
  if (rows > c->cfg.max_rows) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!c->loaded) return MOE_ERR_NOT_LOADED;
  if (rows == 0) return MOE_OK;
  if (!x || !y) return MOE_ERR_INVALID_ARG;
  const size_t nb = (size_t)rows * c->cfg.hidden * 2;
  if (overlaps(x, nb, y, nb)) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)x | (uintptr_t)y) & 15) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->last_stream = s;
  return run_forward(c, x, y, rows, s);
}

int moe_forward_host(moe_ctx* c, const void* x_host, void* y_host, int rows, void* stream) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (rows < 0) return MOE_ERR_INVALID_ARG;
  if (rows > c->cfg.max_rows) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!c->loaded) return MOE_ERR_NOT_LOADED;
  if (rows == 0) return MOE_OK;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->last_stream = s;
  const size_t nb = (size_t)rows * c->cfg.hidden * 2;
  if (cudaMemcpyAsync(c->stage_x, x_host, nb, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  int rc = run_forward(c, c->stage_x, c->stage_y, rows, s);
  if (rc) return rc;
  if (cudaMemcpyAsync(y_host, c->stage_y, nb, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_route(moe_ctx* c, const void* x, int rows, int32_t* idx, float* w, void* stream) {
  if (!c || rows < 0) return MOE_ERR_INVALID_ARG;
  if (rows > c->cfg.max_rows) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!c->loaded) return MOE_ERR_NOT_LOADED;
  if (rows == 0) return MOE_OK;
  if (!x || !idx || !w) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->last_stream = s;
  KArgs a = make_args(c, x, nullptr, rows);
  c->fwd_rows = 0;  // the routing kernels rewrite the workspace's codes
  int rc = run_router_and_quant(c, a, s);
  if (rc) return rc;
  const size_t n = (size_t)rows * c->cfg.top_k;
  if (cudaMemcpyAsync(idx, c->w.idx, n * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(w, c->w.wts, n * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_quantize(moe_ctx* c, const void* x, int rows, uint8_t* codes, float* scales, void* stream) {
  if (!c || rows < 0) return MOE_ERR_INVALID_ARG;
  if (rows > c->cfg.max_rows) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!c->loaded) return MOE_ERR_NOT_LOADED;
  if (rows == 0) return MOE_OK;
  if (!x || !codes || !scales) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->last_stream = s;
  KArgs a = make_args(c, x, nullptr, rows);
  c->fwd_rows = 0;  // rewrites the workspace's codes
  if (launch_quant_gamma(a, s) != cudaSuccess) return MOE_ERR_CUDA;
  const size_t H = c->cfg.hidden;
  if (cudaMemcpyAsync(codes, c->w.xq, rows * H, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(scales, c->w.sx, rows * (H / kGroup) * 4, cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int moe_add_rmsnorm_quantize(moe_ctx* c, const void* residual, const void* x, const void* gamma,
                             float eps, int rows, void* h_out, void* xn_out, uint8_t* codes,
                             float* scales, void* stream) {
  if (!c || rows < 0) return MOE_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || !isfinite(eps)) return MOE_ERR_INVALID_ARG;
  const int H = c->cfg.hidden;
  if (H > kAddNormMaxHidden || per_row_scales(c->cfg)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!residual || !x || !gamma || !h_out || !xn_out || !codes || !scales)
    return MOE_ERR_INVALID_ARG;
  if ((((uintptr_t)residual | (uintptr_t)x | (uintptr_t)gamma | (uintptr_t)h_out |
        (uintptr_t)xn_out) & 15) || ((uintptr_t)codes & 7) || ((uintptr_t)scales & 3))
    return MOE_ERR_INVALID_ARG;
  const size_t nb = (size_t)rows * H * 2, nc = (size_t)rows * H,
               ns = (size_t)rows * (H / kGroup) * 4, ng = (size_t)H * 2;
  // each output is either exactly one of the row inputs (in place) or apart
  // from it; outputs never overlap each other or gamma
  auto in_place_or_apart = [&](const void* out) {
    return (out == residual || !overlaps(out, nb, residual, nb)) &&
           (out == x || !overlaps(out, nb, x, nb));
  };
  if (!in_place_or_apart(h_out) || !in_place_or_apart(xn_out) ||
      overlaps(h_out, nb, xn_out, nb) || overlaps(h_out, nb, gamma, ng) ||
      overlaps(xn_out, nb, gamma, ng))
    return MOE_ERR_INVALID_ARG;
  const void* others[] = {residual, x, h_out, xn_out};
  for (const void* p : others)
    if (overlaps(codes, nc, p, nb) || overlaps(scales, ns, p, nb)) return MOE_ERR_INVALID_ARG;
  if (overlaps(codes, nc, scales, ns) || overlaps(codes, nc, gamma, ng) ||
      overlaps(scales, ns, gamma, ng))
    return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->last_stream = s;
  if (launch_add_rmsnorm_quant(static_cast<const bf16*>(residual), static_cast<const bf16*>(x),
                               static_cast<const bf16*>(gamma), eps, rows, H,
                               static_cast<bf16*>(h_out), static_cast<bf16*>(xn_out), codes,
                               scales, s, c->opt_pdl != 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_forward_addnorm(moe_ctx* c, const void* residual, const void* x, const void* gamma,
                        float eps, int rows, void* h_out, void* xn_out, void* y, void* stream) {
  if (!c || rows < 0) return MOE_ERR_INVALID_ARG;
  if (rows > c->cfg.max_rows) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!c->loaded) return MOE_ERR_NOT_LOADED;
  if (!(eps >= 0.0f) || !isfinite(eps)) return MOE_ERR_INVALID_ARG;
  const int H = c->cfg.hidden;
  if (H > kAddNormMaxHidden || per_row_scales(c->cfg)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!residual || !x || !gamma || !h_out || !y) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)residual | (uintptr_t)x | (uintptr_t)gamma | (uintptr_t)h_out |
       (uintptr_t)xn_out | (uintptr_t)y) & 15)
    return MOE_ERR_INVALID_ARG;
  // outputs apart from every input and from each other (the one-row kernel
  // reads the inputs in every CTA while one of them writes the outputs)
  const size_t nb = (size_t)rows * H * 2, ng = (size_t)H * 2;
  const void* outs[] = {h_out, xn_out, y};
  for (int i = 0; i < 3; ++i) {
    if (!outs[i]) continue;
    if (overlaps(outs[i], nb, residual, nb) || overlaps(outs[i], nb, x, nb) ||
        overlaps(outs[i], nb, gamma, ng))
      return MOE_ERR_INVALID_ARG;
    for (int j = i + 1; j < 3; ++j)
      if (outs[j] && overlaps(outs[i], nb, outs[j], nb)) return MOE_ERR_INVALID_ARG;
  }
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->last_stream = s;
  if (use_decode(c, rows) && use_row(c, rows)) {
    // one row: the add-norm runs inside the layer's one kernel
    KArgs a = make_args(c, x, y, rows);
    a.an = AddNorm{static_cast<const bf16*>(residual), static_cast<const bf16*>(gamma),
                   static_cast<bf16*>(h_out), static_cast<bf16*>(xn_out), eps, 0};
    c->fwd_rows = rows;
    c->fwd_slot_order = false;
    return check_launch(launch_decode_row(a, c->sm_count, c->row_smem, c->opt_pdl != 0, s));
  }
  // more rows: the add-norm kernel writes h, the normed rows and their codes,
  // and the grouped path scatters those codes without quantising again
  bf16* xn = xn_out ? static_cast<bf16*>(xn_out) : c->stage_x;
  if (launch_add_rmsnorm_quant(static_cast<const bf16*>(residual), static_cast<const bf16*>(x),
                               static_cast<const bf16*>(gamma), eps, rows, H,
                               static_cast<bf16*>(h_out), xn, c->w.xq, c->w.sx, s,
                               c->opt_pdl != 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  return run_forward(c, xn, y, rows, s, nullptr, true);
}

int moe_expert_activations(moe_ctx* c, int rows, uint8_t* hq, float* sh, void* stream) {
  if (!c || rows < 0) return MOE_ERR_INVALID_ARG;
  if (rows > c->cfg.max_rows) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!c->loaded) return MOE_ERR_NOT_LOADED;
  if (rows == 0) return MOE_OK;
  if (!hq || !sh) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  KArgs a = make_args(c, nullptr, nullptr, rows);
  return check_launch(launch_gather_hq(a, hq, sh, static_cast<cudaStream_t>(stream)));
}

int moe_forward_codes(moe_ctx* c, int rows, uint8_t* codes, float* scales, void* stream) {
  if (!c || rows < 0) return MOE_ERR_INVALID_ARG;
  if (rows > c->cfg.max_rows) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!c->loaded) return MOE_ERR_NOT_LOADED;
  if (rows == 0) return MOE_OK;
  if (!codes || !scales || rows != c->fwd_rows) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  KArgs a = make_args(c, nullptr, nullptr, rows);
  return check_launch(launch_gather_codes(a, c->xg, c->sxg, c->fwd_slot_order, codes, scales,
                                          static_cast<cudaStream_t>(stream)));
}

int moe_profile_forward(moe_ctx* c, const void* x, void* y, int rows, float* stage_ms,
                        const char** stage_names, int capacity, int* n_stages, void* stream) {
  if (!c || !stage_ms || !stage_names || !n_stages || capacity < 1) return MOE_ERR_INVALID_ARG;
  *n_stages = 0;
  if (rows < 0) return MOE_ERR_INVALID_ARG;
  if (rows > c->cfg.max_rows) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!c->loaded) return MOE_ERR_NOT_LOADED;
  if (rows == 0) return MOE_OK;
  if (!x || !y) return MOE_ERR_INVALID_ARG;
  const size_t nb = (size_t)rows * c->cfg.hidden * 2;
  if (overlaps(x, nb, y, nb)) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->last_stream = s;
  const int kMaxStages = 16;
  cudaEvent_t ev[kMaxStages + 1];
  int made = 0;
  int rc = MOE_OK;
  for (; made <= kMaxStages; ++made)
    if (cudaEventCreate(&ev[made]) != cudaSuccess) {
      rc = MOE_ERR_CUDA;
      break;
    }
  StageRec rec;
  if (rc == MOE_OK) {
    rec.ev = ev;
    rec.names = stage_names;
    rec.cap = capacity < kMaxStages ? capacity : kMaxStages;
    if (cudaEventRecord(ev[0], s) != cudaSuccess) rc = MOE_ERR_CUDA;
  }
  if (rc == MOE_OK) rc = run_forward(c, x, y, rows, s, &rec);
  if (rc == MOE_OK && cudaEventSynchronize(ev[rec.n]) != cudaSuccess) rc = MOE_ERR_CUDA;
  if (rc == MOE_OK) {
    for (int i = 0; i < rec.n; ++i)
      if (cudaEventElapsedTime(&stage_ms[i], ev[i], ev[i + 1]) != cudaSuccess) rc = MOE_ERR_CUDA;
    *n_stages = rec.n;
  }
  for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
  if (rc != MOE_OK) cudaGetLastError();
  return rc;
}

int moe_set_option(moe_ctx* c, int option, int value) {
  if (!c) return MOE_ERR_INVALID_ARG;
  switch (option) {
    case MOE_OPT_PATH:
      // 5 named a persistent multi-row decode kernel that no longer exists
      if (value < 0 || value > 6 || value == 5) return MOE_ERR_INVALID_ARG;
      if (per_row_scales(c->cfg) && (value == 3 || value == 4)) return MOE_ERR_UNSUPPORTED_SHAPE;
      c->opt_path = value;
      return MOE_OK;
    case MOE_OPT_PDL:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      c->opt_pdl = value;
      return MOE_OK;
    case MOE_OPT_ROUTER_BF16:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      c->opt_router_bf16 = value;
      return MOE_OK;
    case MOE_OPT_BATCH_INVARIANT:
      if (value != 0 && value != 1) return MOE_ERR_INVALID_ARG;
      c->opt_invariant = value;
      return MOE_OK;
    case MOE_OPT_POLL_LIMIT:
    case MOE_OPT_LAUNCH_EPOCH: {
      if (value < 0 || (option == MOE_OPT_LAUNCH_EPOCH && value >= kTagClear))
        return MOE_ERR_INVALID_ARG;
      DeviceGuard guard(c->device);
      if (!guard.ok) return MOE_ERR_CUDA;
      // the word is read by launches on the context's stream: none may be in flight
      int* word = option == MOE_OPT_POLL_LIMIT ? c->w.status + kPollLimitWord : c->w.done + 4;
      if (cudaStreamSynchronize(c->last_stream) != cudaSuccess ||
          cudaMemcpy(word, &value, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      if (option == MOE_OPT_POLL_LIMIT) c->opt_poll_limit = value;
      return MOE_OK;
    }
    default:
      return MOE_ERR_INVALID_ARG;
  }
}

int moe_last_device_status(moe_ctx* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  int flag = 0;
  if (cudaStreamSynchronize(c->last_stream) != cudaSuccess ||
      cudaMemcpy(&flag, c->w.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(c->w.status, 0, 4) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (flag) {
    // a bounded wait gave up: counters may be mid-count, start them afresh
    const Plan plan = make_plan(&c->cfg);
    if (cudaMemset(c->w.status, 0, plan.sizes[29]) != cudaSuccess ||
        cudaMemset(c->w.gcount, 0, plan.sizes[25]) != cudaSuccess ||
        cudaMemset(c->w.tlog, 0, plan.sizes[32]) != cudaSuccess ||
        cudaMemset(c->w.xw, 0, plan.sizes[39]) != cudaSuccess ||
        (c->opt_poll_limit &&
         cudaMemcpy(c->w.status + kPollLimitWord, &c->opt_poll_limit, sizeof(int),
                    cudaMemcpyHostToDevice) != cudaSuccess)) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  return flag ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

// ---- layers in sequence ------------------------------------------------------

struct moe_chain {
  int n = 0;
  std::vector<moe_ctx*> ctx;
  DevLayer* table = nullptr;          // [n] on the device
};

int moe_chain_create(moe_ctx* const* layers, int n_layers, moe_chain** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!layers || n_layers < 1) return MOE_ERR_INVALID_ARG;
  if (n_layers > kMaxChain) return MOE_ERR_UNSUPPORTED_SHAPE;
  const moe_ctx* c0 = layers[0];
  if (!c0) return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const moe_ctx* c = layers[l];
    if (!c) return MOE_ERR_INVALID_ARG;
    if (!c->loaded) return MOE_ERR_NOT_LOADED;
    if (c->device != c0->device || c->cfg.hidden != c0->cfg.hidden ||
        c->cfg.n_experts != c0->cfg.n_experts || c->cfg.top_k != c0->cfg.top_k ||
        c->cfg.inter != c0->cfg.inter || c->cfg.shared_inter != c0->cfg.shared_inter ||
        c->cfg.act_group != c0->cfg.act_group)
      return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  DeviceGuard guard(c0->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  moe_chain* ch = new (std::nothrow) moe_chain();
  if (!ch) return MOE_ERR_CUDA;
  ch->n = n_layers;
  ch->ctx.assign(layers, layers + n_layers);
  std::vector<DevLayer> host(n_layers);
  for (int l = 0; l < n_layers; ++l) host[l] = layers[l]->L;
  const size_t nt = sizeof(DevLayer) * n_layers;
  if (cudaMalloc(&ch->table, nt) != cudaSuccess ||
      cudaMemcpy(ch->table, host.data(), nt, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaGetLastError();
    if (ch->table) cudaFree(ch->table);
    delete ch;
    return MOE_ERR_CUDA;
  }
  *out = ch;
  return MOE_OK;
}

int moe_chain_forward(moe_chain* ch, const void* x, void* y_all, int rows, void* stream) {
  if (!ch || rows < 0) return MOE_ERR_INVALID_ARG;
  moe_ctx* c0 = ch->ctx[0];
  for (moe_ctx* c : ch->ctx)
    if (rows > c->cfg.max_rows) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MOE_OK;
  if (!x || !y_all) return MOE_ERR_INVALID_ARG;
  const size_t H = c0->cfg.hidden, nb = (size_t)rows * H * 2;
  if (overlaps(x, nb, y_all, nb * ch->n)) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)x | (uintptr_t)y_all) & 15) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c0->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rows == 1 && use_decode(c0, 1) && use_row(c0, 1)) {
    // one launch over every layer; the first context's workspace and launch
    // tags serve the whole chain
    c0->last_stream = s;
    c0->fwd_rows = 0;  // its checking buffers now hold the last layer's values
    KArgs a = make_args(c0, x, y_all, 1);
    a.chain = Chain{ch->table, ch->n};
    return check_launch(launch_decode_chain(a, c0->sm_count, c0->row_smem, c0->opt_pdl != 0, s));
  }
  // otherwise each layer's forward, y of layer l the input of layer l + 1
  const char* src = static_cast<const char*>(x);
  char* dst = static_cast<char*>(y_all);
  for (int l = 0; l < ch->n; ++l) {
    moe_ctx* c = ch->ctx[l];
    c->last_stream = s;
    const int rc = run_forward(c, src, dst, rows, s);
    if (rc != MOE_OK) return rc;
    src = dst;
    dst += nb;
  }
  return MOE_OK;
}

void moe_chain_destroy(moe_chain* ch) {
  if (!ch) return;
  {
    DeviceGuard guard(ch->ctx[0]->device);
    cudaDeviceSynchronize();
    cudaFree(ch->table);
  }
  delete ch;
}

int moe_debug_poison_workspace(moe_ctx* c, int byte, void* stream) {
  if (!c || byte < 0 || byte > 255) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(c->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  c->last_stream = s;
  for (const auto& r : c->data_regions)
    if (cudaMemsetAsync(r.first, byte, r.second, s) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  c->fwd_rows = 0;  // the workspace no longer holds a forward's codes
  return MOE_OK;
}

void moe_destroy(moe_ctx* c) {
  if (!c) return;
  {
    DeviceGuard guard(c->device);
    cudaDeviceSynchronize();
    free_all(c);
  }
  delete c;
}

}  // extern "C"

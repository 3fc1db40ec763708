// Internal declarations shared by the kernels and the C-ABI host code.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

typedef __nv_bfloat16 bf16;

constexpr int kGroup = 128;       // activation group = weight block edge
constexpr int kChunk = 16;        // tokens per expert chunk (two n8 MMA tiles)
constexpr int kSchedRows = 128;   // rows per block of the prompt schedule (4 bitmap words)
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 16;
constexpr int kDecodeRows = 16;   // rows at or below which the decode kernels run

// Context status block (int words): [0] the device status flag, [1..12] the
// kernels' barrier counters (DevWork::done; done[6] counts the one-row chain
// kernel's finished combines), [13..14] unused,
// [kPollLimitWord] tries before a poll of another CTA's exchange word gives
// up (0 = the kernels' default; a checking option).
constexpr int kPollLimitWord = 15;
// The role-split decode kernels' launch tags stay below kTagWrap: the launch
// whose last tag reaches kTagClear clears the exchange words and restarts the
// epoch, and one launch uses at most kMaxChain tags (one per layer).
constexpr int kTagWrap = 0x7FFFFFFF;
constexpr int kMaxChain = 4096;
constexpr int kTagClear = kTagWrap - kMaxChain;

struct Dims {
  int T, H, E, k, I, Is;
  int rbf16;    // 1: route on logits rounded to bf16 (selection and softmax)
  int per_row;  // 1: one activation scale per row of x and of each SwiGLU row
};

// Device copies of the weights (context-owned).
struct DevLayer {
  const uint8_t* w13;  // e4m3 [E][2I][H]
  const float* s13;    // [E][2I/128][H/128]
  const uint8_t* w2;   // e4m3 [E][H][I]
  const float* s2;     // [E][H/128][I/128]
  const float* wr;     // fp32 [E][H]
  const bf16* ws13;    // [2Is][H]
  const bf16* ws2;     // [H][Is]
  const bf16* gate;    // [H]
};

// Workspace (context-owned, sized for max_rows).
struct DevWork {
  float* logits;        // [T][E]
  int* idx;             // [T][k]
  float* wts;           // [T][k]
  uint8_t* xq;          // [T][H]
  float* sx;            // [T][H/128]
  float* gamma;         // [T]
  uint32_t* bitmap;     // [E][ceil(T/32)]
  int* wprefix;         // [E][ceil(T/32)]
  int* counts;          // [E]
  int* off;             // [E+1]
  int* pair_of_slot;    // [T*k]  slot order = (expert, row)
  int* slot_of_pair;    // [T*k]
  int4* chunks;         // [max_chunks] {expert, first slot, tokens, 0}
  int* n_chunks;        // [1]
  float* hbuf;          // [T*k][I]  SwiGLU rows before re-quantisation
  uint8_t* hq;          // [T*k][I]  by slot
  float* sh;            // [T*k][I/128]
  int* gcount;          // [max_chunks][I/128] arrival counters (self-resetting)
  bf16* hs;             // [T][Is]
  bf16* dbuf;           // [T*k][H] by slot
  bf16* ds;             // [T][H]
  int* status;          // [1] device status flag
  int* done;            // [12] barrier counters (self-resetting) and the decode launch tag
  unsigned long long* tlog;  // [kDecodeRows][E] decode logits as {launch tag, value} words
  unsigned long long* xw;  // decode exchange words: [16k][I] h, [16k][H] d, [16][Is] hs, [16][H] ds
  int* sched_rank;      // [T*k] rank of each pair among its expert's rows in its 128-row block
  int* sched_blk;       // [ceil(T/128)][E] rows per expert in each 128-row block
};

// The residual add + RMS norm in front of the layer, when a forward takes
// (residual, x) instead of x (moe_forward_addnorm); residual == nullptr for
// a plain forward.
struct AddNorm {
  const bf16* residual;  // [T][H]
  const bf16* gamma;     // [H]
  bf16* h_out;           // [T][H] the new residual stream, bf16(residual + x)
  bf16* xn_out;          // [T][H] the normed rows, or nullptr
  float eps;
  int pre_q;             // 1: w.xq / w.sx already hold the normed rows' codes
};

// Layers passed through in one launch (the one-row chain kernel): n layers'
// weights (layer l's y, in the output, is layer l+1's x).
struct Chain {
  const DevLayer* layers;      // [n] device array
  int n;
};

struct KArgs {
  Dims d;
  DevLayer L;
  DevWork w;
  const bf16* x;  // the layer's input; with an add-norm, the block output added to residual
  bf16* y;        // the layer's output; in a chain, [n][H] (every layer's y)
  AddNorm an;
  Chain chain;    // n == 0: one layer
};

// Upper bound of sum_e ceil(count_e / kChunk) over experts with sum_e count_e = T*k.
inline int max_chunks(int T, int k, int E) { return (T * k + kChunk - 1) / kChunk + E; }

// Launchers (return cudaGetLastError()).
cudaError_t launch_router(const KArgs& a, cudaStream_t s);
cudaError_t launch_quant_gamma(const KArgs& a, cudaStream_t s);
cudaError_t launch_topk(const KArgs& a, cudaStream_t s, bool pdl = false);
// top-k of logits given as `ks` partial sums part[ks][T][E], summed in split
// order into the workspace logits first
cudaError_t launch_topk_splits(const KArgs& a, const float* part, int ks, cudaStream_t s,
                               bool pdl = false);
cudaError_t launch_schedule(const KArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t setup_schedule();
cudaError_t launch_gateup(const KArgs& a, int grid, cudaStream_t s);
cudaError_t launch_down(const KArgs& a, int grid, cudaStream_t s);
cudaError_t launch_combine(const KArgs& a, cudaStream_t s, bool pdl = false);

// ---- one-row decode kernel (k_decode_row.cu) ---------------------------------
size_t decode_row_smem(int G, int H, int E, int k, int I, int Is);
bool decode_row_fits(int G, int H, int E, int k, int I, int Is, size_t budget);
cudaError_t setup_decode_row(size_t max_smem);
cudaError_t launch_decode_row(const KArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s);
// The one-row kernel over the layers of a.chain in one launch.
cudaError_t launch_decode_chain(const KArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s);

// ---- 2..16-row decode kernel (k_decode_rows.cu) ---------------------------------
size_t decode_rows_smem(int H);
bool decode_rows_fits(int G, int H, int E, int k, int I, int Is, size_t budget);
cudaError_t setup_decode_rows(size_t max_smem);
cudaError_t launch_decode_rows(const KArgs& a, int grid, size_t smem, bool pdl, cudaStream_t s);

// ---- prompt path on tcgen05 tensor cores (k_prompt_tc.cu) -------------------
enum { kTcRoutedGateUp = 0, kTcRoutedDown = 1, kTcSharedGateUp = 2, kTcSharedDown = 3,
       kTcRouter = 4 };

// One grouped GEMM launch: out-features x tokens tiles of 128 x (<=128).
struct TcGemm {
  CUtensorMap a;       // weights [rows][K], 128-byte boxes of 128 rows
  CUtensorMap b;       // tokens or slots [rows][K], 128-byte boxes of 16 rows
  CUtensorMap bt;      // the same operand in boxes of a whole token tile (64 or
                       // 128 rows): one copy per K block for a full tile
  int n_k;             // K blocks of 128 bytes
  int b_kwrap;         // K blocks after which the B operand's K coordinate wraps
  int ksplit;          // K splits per output tile (router; partial sums), else 1
  int n_f;             // 128-row output tiles per token tile
  int a_rows_e;        // weight rows per expert (routed)
  int up_rows;         // rows from an item's first A tile to its second
  int f_rows;          // A rows (output features) per item
  int E;               // experts (routed)
  int T;               // rows (shared)
  int ldo;             // row length of the output
  const int* counts;   // [E] rows per expert (routed)
  const int* off;      // [E] first slot per expert (routed)
  const float* sa;     // weight block scales (routed)
  const float* sb;     // activation scales [slot][n_k] (routed)
  uint8_t* hq;         // routed gate/up: e4m3 SwiGLU rows [slot][ldo]
  float* hf;           // routed gate/up with one scale per row: fp32 SwiGLU rows
                       // [slot][ldo] instead of hq (quantised by k_quant_h_rows)
  float* sh;           // routed gate/up: their scales [slot][ldo/128]
  bf16* out;           // expert kinds: bf16 [row][ldo]
  float* outf;         // router: fp32 logits [ksplit][row][ldo] (partials when ksplit > 1)
  int* status;         // device status flag (set when a wait gives up)
};

size_t tc_gemm_smem(int kind, int n_k);
// Token rows per tile (N) of each GEMM kind: the box rows of TcGemm::bt.
int tc_gemm_tile_rows(int kind);
cudaError_t setup_tc_gemm(int kind, size_t smem);
cudaError_t launch_tc_gemm(int kind, const TcGemm& g, int grid, size_t smem, cudaStream_t s,
                           bool pdl = false);
cudaError_t launch_quant_scatter(const KArgs& a, uint8_t* xg, float* sxg, cudaStream_t s,
                                 bool pdl = false);
cudaError_t launch_quant_h_rows(const float* hf, uint8_t* hq, float* sh, int n_rows, int I,
                                cudaStream_t s, bool pdl = false);
cudaError_t launch_split_router(const float* wr, bf16* out, int E, int Epad, int H, cudaStream_t s);
bool make_tc_map(CUtensorMap* m, bool bf16_elems, const void* ptr, uint64_t rows, uint64_t cols,
                 uint32_t box_rows);
cudaError_t launch_gather_hq(const KArgs& a, uint8_t* hq, float* sh, cudaStream_t s);
cudaError_t launch_gather_codes(const KArgs& a, const uint8_t* xg, const float* sxg,
                                bool slot_order, uint8_t* codes, float* scales, cudaStream_t s);

// Decode path (rows <= kDecodeRows): three kernels chained with programmatic
// dependent launch when `pdl` is set.
cudaError_t launch_route_decode(const KArgs& a, bool pdl, cudaStream_t s);
cudaError_t launch_gateup_decode(const KArgs& a, int grid, bool pdl, cudaStream_t s);
cudaError_t launch_down_combine_decode(const KArgs& a, bool pdl, cudaStream_t s);

// Launch `kernel` on `s`, allowing it to start before the previous kernel in
// the stream completes when `pdl` is set (it must call griddepcontrol.wait
// before reading that kernel's results).
template <typename... KArgsT, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgsT...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe

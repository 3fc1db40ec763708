/*
 * block_fp8_moe: the block-FP8 mixture-of-experts layer of the Drama 3 backbone
 * on one GB300 (sm_103a), as a C ABI.
 *
 * The layer (PR #925/#920/#927, commit "the Drama 3 text backbone"; PR #939
 * "Fish Audio Drama 3 text to speech on one CUDA GPU", section "Precision"):
 *
 *   y[t] = sum_{j<k} w[t,j] * E_{idx[t,j]}(x[t]) + sigmoid(x[t] . g) * S(x[t])
 *
 *   - router: logits = x . Wr^T in fp32; the k largest (ties to the lower
 *     expert index, as the tie seen in section "Fidelity against the PyTorch
 *     oracle" of PR #939 requires a rule); w = softmax over the k selected
 *     logits (= fp32 softmax renormalised over the selection);
 *   - E_e: a SwiGLU expert with e4m3 weights and one fp32 scale per 128x128
 *     block.  Its inputs are quantised dynamically per row and per 128 inputs
 *     (scale = amax / 448, round to nearest even, saturating), its gate/up
 *     outputs are rounded to bf16, SwiGLU is taken in fp32 and re-quantised
 *     the same way for the down projection (commit "one SwiGLU launch for the
 *     routed and shared experts": routed rows are stored as their FP8
 *     quantisation), and its output is rounded to bf16;
 *   - S: the shared SwiGLU expert with bf16 weights, outputs rounded to bf16;
 *   - combine in fp32, routed terms in rank order then the shared term, one
 *     rounding to bf16 (commit "MoE combine on 8-wide vectors": every sum
 *     keeps its order).
 *
 * Conventions for every call:
 *   - Return value: MOE_OK (0) or one of the negative MOE_ERR_* codes below;
 *     no call aborts, traps or prints.
 *   - Tensors are dense row-major with the innermost dimension last.  bf16
 *     values are passed as their 16-bit patterns (uint16_t), e4m3 values as
 *     their 8-bit codes (OCP E4M3).
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream.  Calls marked "asynchronous" only enqueue work on it.
 *   - A context is used by one stream at a time; contexts are independent.
 */
#ifndef BLOCK_FP8_MOE_H
#define BLOCK_FP8_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,       /* null pointer, negative size, aliasing, bad option */
  MOE_ERR_UNSUPPORTED_SHAPE = -2, /* a config the kernels do not assume, or rows > max_rows */
  MOE_ERR_NOT_LOADED = -3,        /* forward/route before moe_load_weights succeeded */
  MOE_ERR_ALLOC_LIMIT = -4,       /* weights + workspace would exceed workspace_cap_bytes */
  MOE_ERR_CUDA = -5,              /* a CUDA runtime call failed (no device, OOM, launch) */
  MOE_ERR_DEVICE_TIMEOUT = -6     /* a bounded device-side wait gave up (see moe_last_device_status) */
};

typedef struct moe_ctx moe_ctx; /* opaque: owns the device weights and workspace */

/* Layer shape.  Supported: hidden % 128 == 0, inter % 128 == 0,
 * shared_inter % 128 == 0, 1 <= top_k <= 16, top_k <= n_experts <= 256,
 * act_group == 128 or act_group == hidden, 1 <= max_rows <= 65536.  The
 * Drama 3 layer is hidden 2048, 256 experts, top-8, inter 512,
 * shared_inter 512.
 * act_group: 128 quantises the experts' inputs per row and per 128 values
 * (PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA GPU",
 * section "Precision"); hidden gives each row of x, and each routed SwiGLU
 * row, one scale (row amax / 448), the other reading of "dynamic per-row"
 * activations.  Weight scales stay per 128 x 128 block either way.  With one
 * scale per row, 16 rows or fewer run on the role-split decode kernels and
 * more on the tcgen05 kernels (MOE_OPT_PATH 3 and 4, and
 * moe_add_rmsnorm_quantize, return MOE_ERR_UNSUPPORTED_SHAPE), and a device
 * without the tcgen05 kernels for the shape refuses the context. */
typedef struct {
  int hidden;          /* H */
  int n_experts;       /* E */
  int top_k;           /* k */
  int inter;           /* I: routed SwiGLU width */
  int shared_inter;    /* Is: shared SwiGLU width */
  int act_group;       /* activation quantisation group: 128, or hidden (one scale per row) */
  int max_rows;        /* largest T one forward accepts; sizes the workspace */
  size_t workspace_cap_bytes; /* 0 = no cap; else weights + workspace must fit */
} moe_config;

/* Weights of one layer, as a block-FP8 checkpoint stores them ("weights load
 * as stored; nothing is requantized").  All pointers are read only during
 * moe_load_weights and stay owned by the caller.
 *   w13    e4m3 [E][2I][H]  rows 0..I-1 are the gate projection, I..2I-1 up
 *   s13    fp32 [E][2I/128][H/128]  one scale per 128x128 block of w13
 *   w2     e4m3 [E][H][I]   down projection
 *   s2     fp32 [E][H/128][I/128]
 *   router fp32 [E][H]
 *   ws13   bf16 [2Is][H]    shared expert gate (rows 0..Is-1) and up
 *   ws2    bf16 [H][Is]     shared expert down
 *   shared_gate bf16 [H]    gate vector g of the shared expert */
typedef struct {
  const uint8_t* w13;
  const float* s13;
  const uint8_t* w2;
  const float* s2;
  const float* router;
  const uint16_t* ws13;
  const uint16_t* ws2;
  const uint16_t* shared_gate;
} moe_weights;

/* Validate `cfg`, select `device`, allocate the weight buffers and the
 * workspace for cfg->max_rows rows.  Refuses unsupported shapes
 * (MOE_ERR_UNSUPPORTED_SHAPE) and sizes above the cap (MOE_ERR_ALLOC_LIMIT)
 * before allocating anything.  On success *out owns everything; on failure
 * *out is NULL and nothing is left allocated.  Synchronous.
 * Defined by: PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
 * GPU", section "What it adds" (config.zig checks every number the kernels
 * assume and refuses any other checkpoint shape); PR #925 "drama: load the
 * checkpoint with direct I/O in file order and build the codec on its own
 * thread", conversation, the allocation-cap commit (setAllocationLimit: a
 * refused allocation leaves usage unchanged). */
int moe_create(const moe_config* cfg, int device, moe_ctx** out);

/* Copy one layer's weights into the context (layout described in
 * moe_weights).  pointers_on_device = 1: device pointers; 0: host pointers
 * (pageable or pinned).  Checks the block scales are finite and positive;
 * returns after the copies have completed (synchronous on `stream`).
 * Defined by: PR #925 "drama: load the checkpoint with direct I/O in file
 * order and build the codec on its own thread", conversation, commit "the
 * Drama 3 text backbone on CUDA" (weights load as stored; nothing is
 * requantized). */
int moe_load_weights(moe_ctx* ctx, const moe_weights* w, int pointers_on_device, void* stream);

/* y = MoE(x).  x: bf16 [rows][H] on the device; y: bf16 [rows][H] on the
 * device; x and y must not overlap and must be 16-byte aligned
 * (MOE_ERR_INVALID_ARG otherwise).  0 <= rows <= max_rows; rows == 0 does
 * nothing.  Asynchronous on `stream`: no allocation, no host synchronisation,
 * expert counts stay on the device.  Results are bitwise identical from run
 * to run for the same inputs.  Device-side faults of earlier work surface as
 * MOE_ERR_CUDA on a later call.
 * Defined by: PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
 * GPU", sections "Precision" (per-row, per-128 e4m3 inputs, amax / 448) and
 * "What it adds" (the prompt pass and the frame step); the commits "the Drama
 * 3 text backbone on CUDA" (256-expert top-8 block-FP8 MoE with a gated shared
 * expert), "one SwiGLU launch for the routed and shared experts" and "MoE
 * combine on 8-wide vectors". */
int moe_forward(moe_ctx* ctx, const void* x, void* y, int rows, void* stream);

/* The same layer with x and y in host memory: copies x to the device, runs
 * moe_forward, copies y back and synchronises `stream` before returning.
 * Pinned host buffers give the fastest copies.
 * Defined by: the layer of moe_forward (PR #939 "drama3: Fish Audio Drama 3
 * text to speech on one CUDA GPU", section "Precision"). */
int moe_forward_host(moe_ctx* ctx, const void* x_host, void* y_host, int rows, void* stream);

/* Router only (same kernels as moe_forward): idx int32 [rows][k] in rank
 * order and w fp32 [rows][k], both device pointers.  Asynchronous.
 * Defined by: PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
 * GPU", section "What it adds" (the router) and section "Fidelity against the
 * PyTorch oracle" (8th and 9th experts 6e-5 apart or exactly tied: a tie rule
 * is needed; here the lower expert wins). */
int moe_route(moe_ctx* ctx, const void* x, int rows, int32_t* idx, float* w, void* stream);

/* Router without a context, for callers that must not allocate device
 * memory: a runtime that has already handed all of the device's memory to
 * its own pool, or a latency-critical loop that cannot afford cudaMalloc's
 * implicit synchronisation.  This call is a library convenience; the pages
 * that define the layer have no counterpart to it.
 *
 * Computes what moe_route computes, with the CUDA-core router kernels that
 * moe_route runs when MOE_OPT_PATH is 4 (fp32 logits x . router^T, the top_k
 * largest with ties to the lower expert, softmax over the selection): x bf16
 * [rows][hidden], router fp32 [n_experts][hidden],
 * idx int32 [rows][top_k] in rank order, w fp32 [rows][top_k]; all device
 * pointers on the current device, owned by the caller.  Asynchronous on
 * `stream`.
 *
 * The logits live in one scratch array per device inside this library
 * (MOE_ROUTE_STATIC_MAX_LOGITS fp32 values, 1 MiB): rows * n_experts above
 * that limit returns MOE_ERR_UNSUPPORTED_SHAPE (256 experts: up to 1024 rows
 * per call) before anything is launched.  Nothing in the scratch has to start
 * at zero: every logit a call reads was written by the same call.
 *   - The call makes no cudaMalloc or cudaFree call and calls no allocating
 *     library routine.
 *   - The first call on each device looks up the scratch's address
 *     (cudaGetSymbolAddress).  Under CUDA's lazy module loading (the default
 *     since CUDA 12.2) that look-up, or the first launch, can make the driver
 *     load this library's device code and the scratch array, which takes
 *     device memory once.  Make that first call during set-up, before any
 *     stream capture starts and before the caller's memory pool claims the
 *     device; later calls allocate nothing.
 *   - The address is cached per device and per CUDA context: after a device
 *     reset the next call looks it up again.
 *   - All calls on one device share the scratch: two calls whose work can
 *     overlap on the device (other streams, other host threads) race and give
 *     wrong results.  Order them on one stream, or with events.
 * Supported: hidden % 128 == 0, 1 <= top_k <= 16, top_k <= n_experts <= 256,
 * device ordinals 0..63; rows == 0 does nothing. */
#define MOE_ROUTE_STATIC_MAX_LOGITS 262144
int moe_route_static(const void* x, const float* router, int rows, int hidden, int n_experts,
                     int top_k, int32_t* idx, float* w, void* stream);

/* Fills the value buffers of the context's workspace with `byte` (0..255):
 * every buffer of values that a forward reads only after writing them in the
 * same call (logits, routing weights, activation and SwiGLU codes and their
 * scales, expert outputs, staging rows).  Index arrays (routing, schedule),
 * weights, counters, launch tags and the status word are left alone.  A forward after it gives the same bits as before it: a check that
 * no kernel depends on what an earlier call left behind (0xFF makes every
 * bf16, fp32 and e4m3 value there a NaN).  Asynchronous on `stream`.
 * A test entry point; the pages that define the layer have no counterpart
 * to it. */
int moe_debug_poison_workspace(moe_ctx* ctx, int byte, void* stream);

/* Activation quantisation only: codes e4m3 [rows][H] and scales fp32
 * [rows][H/128], both device pointers.  Asynchronous.  This launches the
 * row quantisation kernel of the warp-MMA prompt path; every forward kernel
 * quantises with the same device routines (group scale, then codes), but the
 * codes a forward actually fed its experts are read back with
 * moe_forward_codes.
 * Defined by: PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
 * GPU", section "Precision" (e4m3 per row and per 128 inputs, amax / 448);
 * commit "the Drama 3 text backbone on CUDA" (dynamic 1 x 128 FP8 activation
 * quantization). */
int moe_quantize(moe_ctx* ctx, const void* x, int rows, uint8_t* codes, float* scales,
                 void* stream);

/* Residual add + RMS norm in front of the layer, with the normed rows' FP8
 * groups, in one launch (PR #925/#927 commit "add-norm fused with the routed
 * experts' FP8 activation quantization"; PR #939 section "Kernel contract":
 * plain-gamma RMS norm).  Per row t of H = the context's hidden size:
 *   h_out[t]  = bf16(residual[t] + x[t])                       (new residual)
 *   xn_out[t] = bf16(h * (1 / sqrt(sum(h^2) / H + eps)) * gamma) (fp32 math)
 *   codes[t], scales[t] = the 1 x 128 e4m3 groups of the bf16 row xn_out[t],
 *     bit for bit what moe_quantize returns for it.
 * residual, x, h_out, xn_out bf16 [rows][H]; gamma bf16 [H]; codes e4m3
 * [rows][H]; scales fp32 [rows][H/128]; all device pointers owned by the
 * caller, the bf16 ones 16-byte aligned, codes 8-byte and scales 4-byte
 * aligned.  h_out and xn_out may each be exactly `residual` or `x` (in place);
 * no other overlap is allowed (MOE_ERR_INVALID_ARG).  eps must be finite and
 * >= 0; a zero row with eps = 0 divides by zero (the output is NaN, as the
 * formula says).  Needs no loaded weights and no workspace, so rows is not
 * bounded by max_rows; hidden above 8192 returns MOE_ERR_UNSUPPORTED_SHAPE;
 * rows == 0 does nothing.  Asynchronous on `stream`.
 * Defined by: PR #925/#927 commit "add-norm fused with the routed experts'
 * FP8 activation quantization"; PR #939 "drama3: Fish Audio Drama 3 text to
 * speech on one CUDA GPU", section "Kernel contract" (plain-gamma RMS norm). */
int moe_add_rmsnorm_quantize(moe_ctx* ctx, const void* residual, const void* x,
                             const void* gamma, float eps, int rows, void* h_out, void* xn_out,
                             uint8_t* codes, float* scales, void* stream);

/* The residual add + RMS norm and the layer in one call: the layer's input
 * is the normed sum, and the add-norm feeds the experts the FP8 groups it
 * quantises itself (PR #925/#927 commit "add-norm fused with the routed
 * experts' FP8 activation quantization").  Per row t of H values:
 *   h_out[t] = bf16(residual[t] + x[t])                          (new residual)
 *   xn[t]    = bf16(h * (1 / sqrt(sum(h^2) / H + eps)) * gamma)   (fp32 math)
 *   y[t]     = the layer of moe_forward on xn[t]
 * One row runs as one kernel: every CTA of the one-row kernel takes the
 * add-norm of the row in its first pass.  More rows run the add-norm kernel
 * of moe_add_rmsnorm_quantize, whose codes and scales the grouped path
 * scatters to the experts as they are.  The sum of squares is reduced in a
 * different order in the two cases, so a normed value within about 1e-6
 * relative of a bf16 rounding midpoint may round the other way between them.
 * residual, x, h_out, xn_out, y bf16 [rows][H]; gamma bf16 [H]; device
 * pointers, 16-byte aligned.  xn_out may be NULL (the normed rows are then
 * not kept); h_out, xn_out and y must not overlap any input or each other
 * (MOE_ERR_INVALID_ARG).  eps finite and >= 0.  Contexts with one scale per
 * row, or hidden above 8192, return MOE_ERR_UNSUPPORTED_SHAPE.
 * Asynchronous on `stream`; moe_forward_codes afterwards returns the codes
 * the experts read.
 * Defined by: PR #925/#927 commit "add-norm fused with the routed experts'
 * FP8 activation quantization"; PR #939 "drama3: Fish Audio Drama 3 text to
 * speech on one CUDA GPU", section "Kernel contract" (plain-gamma RMS norm)
 * and section "Precision" (bf16 residual stream). */
int moe_forward_addnorm(moe_ctx* ctx, const void* residual, const void* x, const void* gamma,
                        float eps, int rows, void* h_out, void* xn_out, void* y, void* stream);

/* Expert-side intermediates of the most recent moe_forward, for checking:
 * hq e4m3 [rows][k][I] and sh fp32 [rows][k][I/128] (the re-quantised SwiGLU
 * rows fed to each selected expert's down projection, in rank order), device
 * pointers.  Asynchronous; call on the stream of that forward.
 * Defined by: commit "one SwiGLU launch for the routed and shared experts"
 * (routed rows stored as their FP8 quantization); PR #939 "drama3: Fish Audio
 * Drama 3 text to speech on one CUDA GPU", section "Precision". */
int moe_expert_activations(moe_ctx* ctx, int rows, uint8_t* hq, float* sh, void* stream);

/* The FP8 codes and group scales of x that the experts of the most recent
 * moe_forward (or moe_forward_host) read: codes e4m3 [rows][k][H] and scales
 * fp32 [rows][k][H/128], one copy per (row, rank) pair in rank order, device
 * pointers.  The decode kernels quantise a row once for all its experts; the
 * tcgen05 prompt kernels give each pair its own slot-ordered copy, and this
 * call gathers every copy.  rows must equal that forward's rows, and no
 * moe_route or moe_quantize may have run on the context since
 * (MOE_ERR_INVALID_ARG otherwise).  Asynchronous; call on the stream of that
 * forward.
 * Defined by: PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
 * GPU", section "Precision" (e4m3 per row and per 128 inputs, amax / 448);
 * commit "the Drama 3 text backbone on CUDA" (dynamic 1 x 128 FP8 activation
 * quantization). */
int moe_forward_codes(moe_ctx* ctx, int rows, uint8_t* codes, float* scales, void* stream);

/* Options.  MOE_OPT_PATH: 0 = automatic (the role-split one-row kernel for
 * 1 row, the role-split multi-row kernel for 2..4 rows, the grouped prompt
 * kernels on the tcgen05 tensor cores for more; the three chained decode
 * kernels take 5..16 rows where the tcgen05 kernels are not available), 1 =
 * the same as 0, 2 = always the grouped prompt kernels, 3 = rows <= 16 on the three
 * chained decode kernels, 4 = always the grouped prompt kernels with
 * warp-level MMAs instead of tcgen05 (the path every forward takes when a
 * context's shape leaves no room for the tcgen05 kernels: hidden or inter
 * above 4096), 6 = 2..16 rows on the role-split multi-row kernel (5 is not
 * a path and returns MOE_ERR_INVALID_ARG).  A
 * role-split kernel needs the device to have enough SMs for its roles;
 * without them 0, 1 and 6 take the chained kernels.
 * MOE_OPT_PDL: 1 = launch with programmatic dependent launch so a layer's
 * immutable weight reads overlap the previous kernel's tail (default), 0 =
 * plain launches.
 * MOE_OPT_BATCH_INVARIANT: 1 = a row's y is bit-identical whatever rows
 * share its forward (any row count, any position): every row count runs on
 * the grouped kernels (the decode kernels sum in other orders), and the
 * router's K split is fixed (its partial sums are added in one order at
 * every row count).  Costs the decode kernels' speed at 16 rows or fewer.
 * 0 = off (default); MOE_OPT_PATH then chooses.
 * MOE_OPT_ROUTER_BF16: 1 = route on the fp32 logits rounded to bf16
 * (nearest, ties to even): the top-k, its tie rule (lower expert first) and
 * the softmax over the selection all take the rounded values, as a router
 * with bf16 logits does; exact ties between experts become common.  0 = fp32
 * logits (default).  moe_route reports the routing of the variant in force.
 * Checking options (they make the failure and wrap-around paths run; both
 * wait for the context's last stream and write one device word):
 * MOE_OPT_POLL_LIMIT: tries before a role-split decode kernel's poll of
 * another CTA's result gives up and sets the status flag (0 = the built-in
 * limit).  A small value makes a normal one-row forward give up: its output
 * is then undefined, moe_last_device_status returns MOE_ERR_DEVICE_TIMEOUT
 * and restarts the counters, and the next forward is exact again.  Waits for
 * the kernel's own copies keep the built-in limit.
 * MOE_OPT_LAUNCH_EPOCH: the launch epoch of the role-split decode kernels
 * (0 <= value < 2^31 - 1 - 4096).  Their exchange words carry the launch's
 * tag, epoch + 1 (a chain launch uses one tag per layer); the launch whose
 * last tag reaches 2^31 - 1 - 4096 clears every word and restarts the epoch
 * at 0, so a tag never comes back over a stale word.
 * Defined by: PR #920 "drama: Drama 3 (fishaudio/drama-3) text-to-speech on
 * CUDA", section "Receipt" (backbone outputs at chunk sizes 1, 7 and 128 are
 * hash-identical) against PR #939, section "Determinism and request state"
 * (prompt chunk seams fail) for MOE_OPT_BATCH_INVARIANT; PR #939, section
 * "Fidelity against the PyTorch oracle" (the 8th and 9th experts tie exactly
 * on bf16 logits) for MOE_OPT_ROUTER_BF16;
 * PR #927 "drama: the backbone chain launches with programmatic
 * dependent launch", section "What this changes" (the one-row GEMV prefetches
 * immutable weights before its wait); PR #939 "drama3: Fish Audio Drama 3 text
 * to speech on one CUDA GPU", section "What it adds" (the prompt pass and the
 * frame step: every path computes the same layer). */
enum {
  MOE_OPT_PATH = 1,
  MOE_OPT_PDL = 2,
  MOE_OPT_POLL_LIMIT = 3,
  MOE_OPT_LAUNCH_EPOCH = 4,
  MOE_OPT_BATCH_INVARIANT = 5,
  MOE_OPT_ROUTER_BF16 = 6
};
int moe_set_option(moe_ctx* ctx, int option, int value);

/* One forward like moe_forward, timed per kernel: a CUDA event is recorded
 * after every launch on `stream` and the call waits for them.  On return
 * stage_ms[i] is the device time of the i-th launch and stage_names[i] a
 * static name, for i < *n_stages (at most `capacity`).  Synchronous; for
 * measurement only (the events add small gaps between launches).
 * Defined by: PR #920 "drama: Drama 3 (fishaudio/drama-3) text-to-speech on
 * CUDA", section "Receipt" (per-stage timings of the decode step,
 * speed-stages.json). */
int moe_profile_forward(moe_ctx* ctx, const void* x, void* y, int rows, float* stage_ms,
                        const char** stage_names, int capacity, int* n_stages, void* stream);

/* Bytes moe_create would allocate for `cfg` (weights + workspace + staging).
 * Defined by: PR #925 "drama: load the checkpoint with direct I/O in file
 * order and build the codec on its own thread", conversation, the
 * allocation-cap commit (setAllocationLimit: an engine admits a model against
 * a memory budget). */
int moe_required_bytes(const moe_config* cfg, size_t* bytes);

/* Device-side status of the context: MOE_OK, or MOE_ERR_DEVICE_TIMEOUT if a
 * bounded wait in an earlier forward gave up.  Synchronises the context's
 * last stream.  Reading clears the flag.
 * Defined by: PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
 * GPU", conversation, the follow-up fixes (a bad value is refused by name with
 * an error, not trapped on). */
int moe_last_device_status(moe_ctx* ctx);

/* Layers in sequence: the backbone's MoE layers, the output of layer l the
 * input of layer l + 1 (nothing in between), as one object over contexts that
 * stay owned by the caller and must outlive it.  All contexts loaded, on one
 * device, with one shape; at most 4096 layers (MOE_ERR_UNSUPPORTED_SHAPE
 * otherwise).  Allocates a small device table; synchronous.
 * Defined by: PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
 * GPU", section "What it adds" (the frame step runs the next backbone row as
 * one CUDA graph); PR #927 "drama: the backbone chain launches with
 * programmatic dependent launch", section "What this changes". */
typedef struct moe_chain moe_chain;
int moe_chain_create(moe_ctx* const* layers, int n_layers, moe_chain** out);

/* x bf16 [rows][H] through every layer: y_all bf16 [n_layers][rows][H] holds
 * each layer's output (device pointers, 16-byte aligned, x apart from
 * y_all).  One row on a shape the one-row kernel serves runs as ONE launch
 * over all layers: every CTA keeps its role from layer to layer, a layer's
 * input is read from the words the previous layer's combine publishes, and
 * the CTAs that finish a layer early start streaming the next layer's shared
 * expert at once.  That launch uses the first context's workspace and launch
 * tags (a forward on that context in between is fine when stream-ordered);
 * moe_forward_codes on it is refused afterwards.  More rows run each layer's
 * moe_forward in order.  rows <= every context's max_rows.  Asynchronous on
 * `stream`.
 * Defined by: PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
 * GPU", section "What it adds" (the frame step runs the next backbone row as
 * one CUDA graph) and section "Precision" (the layer of moe_forward). */
int moe_chain_forward(moe_chain* chain, const void* x, void* y_all, int rows, void* stream);

/* Release the chain's table.  NULL is accepted; the contexts stay.
 * Defined by: PR #925 "drama: load the checkpoint with direct I/O in file
 * order and build the codec on its own thread", conversation (the worker
 * thread that owns the modules releases them). */
void moe_chain_destroy(moe_chain* chain);

/* Release everything the context owns.  NULL is accepted.
 * Defined by: PR #925 "drama: load the checkpoint with direct I/O in file
 * order and build the codec on its own thread", conversation (one worker
 * thread owns the context, stream and modules and releases them). */
void moe_destroy(moe_ctx* ctx);

/* Static text for a status code.
 * Defined by: PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
 * GPU", conversation, the follow-up fixes (errors refused by name). */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* BLOCK_FP8_MOE_H */

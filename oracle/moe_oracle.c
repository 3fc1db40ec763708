/*
 * CPU oracle for the block-FP8 mixture-of-experts layer of the Drama 3 backbone.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain definition that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or constant with the CUDA library.
 *
 * Single-threaded, double accumulation, e4m3 decoded through a 256-entry table,
 * block-FP8 inner sums taken exactly in int64.  Every step follows the order
 * in which the pages describe the layer:
 *
 *   [A] PR #925/#920/#927, commit "the Drama 3 text backbone": every backbone
 *       layer has "a 256-expert top-8 block-FP8 MoE and a gated shared
 *       expert", FP8 activations are quantized dynamically in 1 x 128 groups,
 *       and the expert weights are used as stored (no requantisation).
 *   [B] PR #939 "Fish Audio Drama 3 text to speech on one CUDA GPU", section
 *       "Precision": bf16 activations; the FP8 experts round their inputs to
 *       e4m3 per row and per 128 inputs with scale amax / 448; fp32 wherever
 *       the reference is fp32; skipping the quantisation moves each MoE
 *       block's output by about 1e-2 relative.
 *   [C] PR #925/#927 commit "one SwiGLU launch for the routed and shared
 *       experts": routed SwiGLU rows are stored as their FP8 quantisation,
 *       the shared expert's rows as bf16.
 *   [D] PR #925/#927 commit "MoE combine on 8-wide vectors": the combine keeps
 *       the order of every sum.
 *   [E] PR #939, section "Fidelity against the PyTorch oracle", prompt pass:
 *       the router's 8th and 9th experts can be 6e-5 apart or exactly tied,
 *       so the top-k tie rule matters; ties go to the lower expert index.
 *   [F] PR #925/#927 commit "add-norm fused with the routed experts' FP8
 *       activation quantization": the residual add and RMS norm before the
 *       MoE also write the normed rows' FP8 groups, rounded exactly as the
 *       separate quantisation of those (bf16) rows would round them.
 *   [G] PR #939, section "Kernel contract": the backbone's RMS norm is the
 *       plain-gamma form (x / rms(x) * gamma, no 1 + gamma offset); section
 *       "Precision": bf16 residual stream.
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 * router logits fp32-rounded for selection, softmax over the selected logits
 * (equal to softmax-then-renormalise), scale 1 for an all-zero group, routed
 * gate/up outputs rounded to bf16 before SwiGLU, SwiGLU in full precision then
 * rounded to fp32 before its re-quantisation, expert outputs rounded to bf16,
 * routing weights applied in the combine, shared expert gated by
 * sigmoid(x . g), shared term added last.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- planted mistakes (tests only) -------------------------------------- */
/* 0 = none.  Each value plants one plausible error so that the pin tests can
 * show that they turn red. */
enum {
  MUT_NONE = 0,
  MUT_TIE_HIGH = 1,        /* top-k ties go to the higher index */
  MUT_SCALE_447 = 2,       /* activation scale amax / 447 */
  MUT_ENC_TRUNC = 3,       /* e4m3 encode truncates instead of RNE */
  MUT_DROP_EXPERT = 4,     /* last selected expert left out of the combine */
  MUT_SWAP_GATE_UP = 5,    /* gate and up halves exchanged */
  MUT_SCALE_TRANSPOSE = 6, /* weight block scale indexed [kb][nb] */
  MUT_GATE_SIGN = 7,       /* shared gate sigmoid(-x.g) */
  MUT_NO_RENORM = 8,       /* routing weights = full softmax, not renormalised */
  MUT_ENC_TIE_UP = 9,      /* e4m3 encode ties away from zero instead of to even */
  MUT_NORM_EPS_OUTSIDE = 10,   /* 1 / (sqrt(ms) + eps) instead of 1 / sqrt(ms + eps) */
  MUT_NORM_NO_RESIDUAL = 11,   /* residual left out of the add */
  MUT_NORM_GAMMA_PLUS_ONE = 12,/* (1 + gamma) offset form instead of plain gamma */
  MUT_NORM_QUANT_UNROUNDED = 13,/* FP8 groups from the normed value before its bf16 rounding */
  MUT_ROUTER_BF16_IGNORED = 14, /* the bf16-logit router variant leaves the logits in fp32 */
  MUT_PER_ROW_IGNORED = 15,     /* the one-scale-per-row variant keeps 1 x 128 groups */
};
static int g_mut = 0;
void orc_set_mutation(int m) { g_mut = m; }
int orc_get_mutation(void) { return g_mut; }

/* ---- e4m3 (OCP 8-bit floating point, E4M3 variant) ---------------------- */
/* Bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite
 * 448, smallest subnormal 2^-9.  The table is built from that closed form. */
static double g_e4m3[256];
static int g_e4m3_ready = 0;

static void e4m3_init(void) {
  if (g_e4m3_ready) return;
  for (int c = 0; c < 256; ++c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7)
      v = NAN;
    else if (e == 0)
      v = ldexp((double)m, -9); /* m/8 * 2^-6 */
    else
      v = ldexp(8.0 + m, e - 10); /* (1 + m/8) * 2^(e-7) */
    g_e4m3[c] = s ? -v : v;
  }
  g_e4m3_ready = 1;
}

double orc_e4m3_decode(uint8_t c) {
  e4m3_init();
  return g_e4m3[c];
}

void orc_e4m3_table(double* out) {
  e4m3_init();
  memcpy(out, g_e4m3, sizeof(g_e4m3));
}

/* Round to the nearest e4m3 value, ties to the even code, saturating to
 * +-448 (infinities too), NaN to 0x7F.  The sign of zero is kept.  The
 * search runs over the 127 non-negative finite codes, which the table lists
 * in increasing order. */
uint8_t orc_e4m3_encode(float v) {
  e4m3_init();
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  /* largest code lo with value(lo) <= a; codes 0x00..0x7E are increasing */
  int lo = 0, hi = 0x7E;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (g_e4m3[mid] <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  int code = lo;
  if (g_e4m3[lo] != a) {
    int up = lo + 1; /* exists because a < 448 */
    double dlo = a - g_e4m3[lo], dup = g_e4m3[up] - a;
    if (g_mut == MUT_ENC_TRUNC)
      code = lo;
    else if (dup < dlo)
      code = up;
    else if (dup == dlo)
      code = (g_mut == MUT_ENC_TIE_UP) ? up : ((lo & 1) ? up : lo);
  }
  return sign | (uint8_t)code;
}

void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

/* ---- bf16 and fp32 rounding --------------------------------------------- */
double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to bf16 once, to nearest, ties to even. */
uint16_t orc_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int ex;
  (void)frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
  int qexp = ex - 8;   /* 8 significant bits */
  if (qexp < -133) qexp = -133; /* subnormal spacing 2^-133 */
  double q = nearbyint(ldexp(a, -qexp)); /* default mode: nearest, ties even */
  double r = ldexp(q, qexp);
  if (r > 3.3895313892515355e38) return sign | 0x7F80;
  float f = (float)r; /* exact: r is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

void orc_bf16_from_double_array(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_double(v[i]);
}

static double bf16r(double v) { return orc_bf16_to_double(orc_bf16_from_double(v)); }

/* ---- dynamic activation quantisation ([A], [B]) ------------------------- */
/* Per group of `group` values: amax over |v|, scale = fp32(amax / 448),
 * codes = e4m3(fp32(v / scale)).  Both divisions are correctly rounded fp32
 * divisions of fp32 operands (double quotient, rounded once to fp32, is
 * exact for that).  An all-zero group takes scale 1. */
void orc_quant_row(const float* v, int n, int group, uint8_t* codes, float* scales) {
  for (int g0 = 0, gi = 0; g0 < n; g0 += group, ++gi) {
    double amax = 0.0;
    for (int i = 0; i < group; ++i) {
      double a = fabs((double)v[g0 + i]);
      if (a > amax) amax = a;
    }
    float s;
    if (amax == 0.0)
      s = 1.0f;
    else
      s = (float)(amax / (g_mut == MUT_SCALE_447 ? 447.0 : 448.0));
    scales[gi] = s;
    for (int i = 0; i < group; ++i) {
      float q = (float)((double)v[g0 + i] / (double)s);
      codes[g0 + i] = orc_e4m3_encode(q);
    }
  }
}

/* ---- residual add + RMS norm + activation quantisation ([F], [G]) -------- */
/* Per row t of H values:
 *   h_i  = bf16(residual_i + x_i)                  (the new residual stream)
 *   r    = 1 / sqrt(sum_i h_i^2 / H + eps)          (double)
 *   xn_i = bf16(h_i * r * gamma_i)                   (the normed row)
 * and the FP8 groups of xn exactly as orc_quant_row gives them for the bf16
 * row.  A zero row with eps = 0 divides by zero (NaN), as the formula does. */
void orc_add_rmsnorm(const uint16_t* residual, const uint16_t* x, const uint16_t* gamma,
                     int T, int H, int group, double eps, uint16_t* h_out, uint16_t* xn_out,
                     uint8_t* codes, float* scales) {
  double* h = (double*)malloc(sizeof(double) * (size_t)H);
  float* xf = (float*)malloc(sizeof(float) * (size_t)H);
  if (!h || !xf) {
    free(h);
    free(xf);
    return;
  }
  for (int t = 0; t < T; ++t) {
    const uint16_t* rr = residual + (size_t)t * H;
    const uint16_t* xr = x + (size_t)t * H;
    double ss = 0.0;
    for (int i = 0; i < H; ++i) {
      const double sum = g_mut == MUT_NORM_NO_RESIDUAL
                             ? orc_bf16_to_double(xr[i])
                             : orc_bf16_to_double(rr[i]) + orc_bf16_to_double(xr[i]);
      h_out[(size_t)t * H + i] = orc_bf16_from_double(sum);
      h[i] = bf16r(sum);
      ss += h[i] * h[i];
    }
    const double ms = ss / H;
    const double r = g_mut == MUT_NORM_EPS_OUTSIDE ? 1.0 / (sqrt(ms) + eps)
                                                   : 1.0 / sqrt(ms + eps);
    for (int i = 0; i < H; ++i) {
      double g = orc_bf16_to_double(gamma[i]);
      if (g_mut == MUT_NORM_GAMMA_PLUS_ONE) g += 1.0;
      const double v = h[i] * r * g;
      xn_out[(size_t)t * H + i] = orc_bf16_from_double(v);
      xf[i] = g_mut == MUT_NORM_QUANT_UNROUNDED ? (float)v : (float)bf16r(v);
    }
    orc_quant_row(xf, H, group, codes + (size_t)t * H, scales + (size_t)t * (H / group));
  }
  free(h);
  free(xf);
}

/* One scale for a whole row of n values (the per-row activation variant): the
 * row quantised as one group, its scale repeated for each of the n / G weight
 * blocks, so that the block-FP8 dot below reads it per block unchanged. */
static void quant_row_one_scale(const float* v, int n, int G, uint8_t* codes, float* scales) {
  float s;
  orc_quant_row(v, n, n, codes, &s);
  for (int b = 0; b < n / G; ++b) scales[b] = s;
}

/* ---- router ([A], [E]) --------------------------------------------------- */
/* logits[e] = sum_i x_i * Wr[e,i] in double.  Selection: k largest by the
 * fp32-rounded logit, ties to the lower index, in rank order.  Weights: the
 * softmax of the selected (double) logits, which equals the full softmax
 * renormalised over the selection. */
static void router_impl(const uint16_t* x, int H, const float* wr, int E, int k,
                        int bf16_logits, double* logits, int32_t* idx, double* w) {
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    const float* row = wr + (size_t)e * H;
    for (int i = 0; i < H; ++i) acc += orc_bf16_to_double(x[i]) * (double)row[i];
    if (bf16_logits && g_mut != MUT_ROUTER_BF16_IGNORED) acc = bf16r((double)(float)acc);
    logits[e] = acc;
  }
  char* taken = (char*)calloc((size_t)E, 1);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    float bv = 0.0f;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      float v = (float)logits[e];
      if (best < 0 || v > bv || (v == bv && g_mut == MUT_TIE_HIGH)) {
        best = e;
        bv = v;
      }
    }
    taken[best] = 1;
    idx[j] = best;
  }
  free(taken);
  if (g_mut == MUT_NO_RENORM) {
    double mx = logits[0];
    for (int e = 1; e < E; ++e)
      if (logits[e] > mx) mx = logits[e];
    double den = 0.0;
    for (int e = 0; e < E; ++e) den += exp(logits[e] - mx);
    for (int j = 0; j < k; ++j) w[j] = exp(logits[idx[j]] - mx) / den;
    return;
  }
  double mx = logits[idx[0]];
  for (int j = 1; j < k; ++j)
    if (logits[idx[j]] > mx) mx = logits[idx[j]];
  double den = 0.0;
  for (int j = 0; j < k; ++j) den += exp(logits[idx[j]] - mx);
  for (int j = 0; j < k; ++j) w[j] = exp(logits[idx[j]] - mx) / den;
}

void orc_router(const uint16_t* x, int H, const float* wr, int E, int k,
                double* logits, int32_t* idx, double* w) {
  router_impl(x, H, wr, E, k, 0, logits, idx, w);
}

/* Router variant with bf16 logits ([E]: the reference's bf16 PyTorch oracle
 * routes on bf16 logits, where the 8th and 9th experts can tie exactly): each
 * logit is the fp32-rounded sum rounded once more to bf16 (nearest, ties to
 * even); selection (ties to the lower index) and the softmax over the
 * selection use those bf16 values. */
void orc_router_bf16(const uint16_t* x, int H, const float* wr, int E, int k,
                     double* logits, int32_t* idx, double* w) {
  router_impl(x, H, wr, E, k, 1, logits, idx, w);
}

/* ---- block-FP8 dot product ---------------------------------------------- */
/* One output of a block-scaled e4m3 GEMM:
 *   sum over K blocks kb of  a_scale[kb] * w_scale[kb] * sum_{k in kb} dec(a_k) dec(w_k)
 * Each e4m3 value times 2^9 is an integer (|.| <= 229376), so the inner sum
 * is exact in int64 and equals 2^18 times the real inner sum. */
static double block_fp8_dot(const uint8_t* a, const float* a_scale, const uint8_t* w,
                            const float* w_scale, int w_scale_stride, int K, int G) {
  e4m3_init();
  double acc = 0.0;
  for (int kb = 0; kb < K / G; ++kb) {
    int64_t s = 0;
    for (int i = kb * G; i < (kb + 1) * G; ++i) {
      int64_t ai = (int64_t)llround(ldexp(g_e4m3[a[i]], 9));
      int64_t wi = (int64_t)llround(ldexp(g_e4m3[w[i]], 9));
      s += ai * wi;
    }
    double ws = (double)w_scale[(size_t)kb * w_scale_stride];
    acc += ldexp((double)s, -18) * (double)a_scale[kb] * ws;
  }
  return acc;
}

double orc_block_fp8_dot(const uint8_t* a, const float* a_scale, const uint8_t* w,
                         const float* w_scale, int K, int G) {
  return block_fp8_dot(a, a_scale, w, w_scale, 1, K, G);
}

/* Dot product without activation quantisation (for the "quantisation off"
 * comparison of [B]): activations taken as given, weights dequantised. */
static double dequant_dot(const float* a, const uint8_t* w, const float* w_scale,
                          int w_scale_stride, int K, int G) {
  double acc = 0.0;
  for (int kb = 0; kb < K / G; ++kb) {
    double s = 0.0;
    for (int i = kb * G; i < (kb + 1) * G; ++i) s += (double)a[i] * g_e4m3[w[i]];
    acc += s * (double)w_scale[(size_t)kb * w_scale_stride];
  }
  return acc;
}

static double silu(double a) { return a / (1.0 + exp(-a)); }

/* ---- the layer ---------------------------------------------------------- */
typedef struct {
  int H, E, k, I, Is, G;
  const uint8_t* w13;    /* e4m3 [E][2I][H]; rows 0..I-1 gate, I..2I-1 up */
  const float* s13;      /* fp32 [E][2I/G][H/G] */
  const uint8_t* w2;     /* e4m3 [E][H][I] */
  const float* s2;       /* fp32 [E][H/G][I/G] */
  const float* wr;       /* fp32 [E][H] */
  const uint16_t* ws13;  /* bf16 [2Is][H]; rows 0..Is-1 gate, Is..2Is-1 up */
  const uint16_t* ws2;   /* bf16 [H][Is] */
  const uint16_t* gate;  /* bf16 [H] */
  int router_bf16;       /* 1: the bf16-logit router variant (orc_router_bf16) */
  int act_per_row;       /* 1: one activation scale per row (x and h) instead of per 1 x G */
} orc_layer;

/* Optional per-row intermediates; any pointer may be NULL. */
typedef struct {
  double* logits;  /* [T][E] */
  int32_t* idx;    /* [T][k] */
  double* w;       /* [T][k] */
  uint8_t* xq;     /* [T][H] */
  float* sx;       /* [T][H/G] */
  uint16_t* z;     /* [T][k][2I] bf16 */
  uint8_t* hq;     /* [T][k][I] */
  float* sh;       /* [T][k][I/G] */
  uint16_t* d;     /* [T][k][H] bf16 */
  uint16_t* zs;    /* [T][2Is] bf16 */
  uint16_t* hs;    /* [T][Is] bf16 */
  uint16_t* ds;    /* [T][H] bf16 */
  double* gamma;   /* [T] */
} orc_trace;

/* y[t] = sum_j w_j * d_j + gamma * d_s for each row t (double), also rounded
 * once to bf16.  act_quant = 0 skips both activation quantisations (the
 * comparison that [B] quotes); every other rounding point is kept. */
int orc_moe_rows(const orc_layer* L, const uint16_t* x, int T, int act_quant,
                 uint16_t* y_bf16, double* y_ref, const orc_trace* tr) {
  e4m3_init();
  const int H = L->H, E = L->E, k = L->k, I = L->I, Is = L->Is, G = L->G;
  if (H % G || I % G || k > E || k < 1) return -1;
  double* logits = (double*)malloc(sizeof(double) * E);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * k);
  double* w = (double*)malloc(sizeof(double) * k);
  float* xf = (float*)malloc(sizeof(float) * H);
  uint8_t* xq = (uint8_t*)malloc(H);
  float* sx = (float*)malloc(sizeof(float) * (H / G));
  double* z = (double*)malloc(sizeof(double) * 2 * I);
  float* hf = (float*)malloc(sizeof(float) * I);
  uint8_t* hq = (uint8_t*)malloc(I);
  float* sh = (float*)malloc(sizeof(float) * (I / G));
  double* dsum = (double*)malloc(sizeof(double) * H);
  double* zs = (double*)malloc(sizeof(double) * 2 * Is);
  double* hs = (double*)malloc(sizeof(double) * Is);
  double* ds = (double*)malloc(sizeof(double) * H);
  const int nb_h = H / G, nb_i = I / G;

  for (int t = 0; t < T; ++t) {
    const uint16_t* xt = x + (size_t)t * H;
    /* router */
    router_impl(xt, H, L->wr, E, k, L->router_bf16, logits, idx, w);
    if (tr && tr->logits) memcpy(tr->logits + (size_t)t * E, logits, sizeof(double) * E);
    if (tr && tr->idx) memcpy(tr->idx + (size_t)t * k, idx, sizeof(int32_t) * k);
    if (tr && tr->w) memcpy(tr->w + (size_t)t * k, w, sizeof(double) * k);
    /* activation quantisation */
    for (int i = 0; i < H; ++i) xf[i] = (float)orc_bf16_to_double(xt[i]);
    if (L->act_per_row && g_mut != MUT_PER_ROW_IGNORED)
      quant_row_one_scale(xf, H, G, xq, sx);
    else
      orc_quant_row(xf, H, G, xq, sx);
    if (tr && tr->xq) memcpy(tr->xq + (size_t)t * H, xq, H);
    if (tr && tr->sx) memcpy(tr->sx + (size_t)t * nb_h, sx, sizeof(float) * nb_h);

    for (int m = 0; m < H; ++m) dsum[m] = 0.0;
    const int k_used = (g_mut == MUT_DROP_EXPERT) ? k - 1 : k;
    for (int j = 0; j < k; ++j) {
      const int e = idx[j];
      const uint8_t* w13 = L->w13 + (size_t)e * 2 * I * H;
      const float* s13 = L->s13 + (size_t)e * (2 * I / G) * nb_h;
      /* gate/up: z[n] for n < 2I */
      for (int n = 0; n < 2 * I; ++n) {
        const float* srow;
        int sstride;
        if (g_mut == MUT_SCALE_TRANSPOSE) {
          /* reads s13 as if it were [H/G][2I/G] */
          srow = s13 + (n / G);
          sstride = 2 * I / G;
        } else {
          srow = s13 + (size_t)(n / G) * nb_h;
          sstride = 1;
        }
        double v = act_quant ? block_fp8_dot(xq, sx, w13 + (size_t)n * H, srow, sstride, H, G)
                             : dequant_dot(xf, w13 + (size_t)n * H, srow, sstride, H, G);
        z[n] = bf16r(v);
      }
      if (tr && tr->z)
        for (int n = 0; n < 2 * I; ++n)
          tr->z[((size_t)t * k + j) * 2 * I + n] = orc_bf16_from_double(z[n]);
      /* SwiGLU, rounded to fp32, then re-quantised */
      for (int n = 0; n < I; ++n) {
        double g = z[n], u = z[I + n];
        if (g_mut == MUT_SWAP_GATE_UP) {
          g = z[I + n];
          u = z[n];
        }
        hf[n] = (float)(silu(g) * u);
      }
      if (act_quant) {
        if (L->act_per_row && g_mut != MUT_PER_ROW_IGNORED)
          quant_row_one_scale(hf, I, G, hq, sh);
        else
          orc_quant_row(hf, I, G, hq, sh);
      }
      if (tr && tr->hq) memcpy(tr->hq + ((size_t)t * k + j) * I, hq, I);
      if (tr && tr->sh) memcpy(tr->sh + ((size_t)t * k + j) * nb_i, sh, sizeof(float) * nb_i);
      /* down */
      const uint8_t* w2 = L->w2 + (size_t)e * H * I;
      const float* s2 = L->s2 + (size_t)e * nb_h * nb_i;
      for (int m = 0; m < H; ++m) {
        const float* srow = s2 + (size_t)(m / G) * nb_i;
        double v = act_quant ? block_fp8_dot(hq, sh, w2 + (size_t)m * I, srow, 1, I, G)
                             : dequant_dot(hf, w2 + (size_t)m * I, srow, 1, I, G);
        double dv = bf16r(v);
        if (tr && tr->d) tr->d[((size_t)t * k + j) * H + m] = orc_bf16_from_double(dv);
        if (j < k_used) dsum[m] += w[j] * dv;
      }
    }
    /* shared expert, bf16 weights */
    for (int n = 0; n < 2 * Is; ++n) {
      double acc = 0.0;
      const uint16_t* row = L->ws13 + (size_t)n * H;
      for (int i = 0; i < H; ++i) acc += orc_bf16_to_double(xt[i]) * orc_bf16_to_double(row[i]);
      zs[n] = bf16r(acc);
    }
    for (int n = 0; n < Is; ++n) {
      double g = zs[n], u = zs[Is + n];
      if (g_mut == MUT_SWAP_GATE_UP) {
        g = zs[Is + n];
        u = zs[n];
      }
      hs[n] = bf16r(silu(g) * u);
    }
    for (int m = 0; m < H; ++m) {
      double acc = 0.0;
      const uint16_t* row = L->ws2 + (size_t)m * Is;
      for (int n = 0; n < Is; ++n) acc += hs[n] * orc_bf16_to_double(row[n]);
      ds[m] = bf16r(acc);
    }
    double xg = 0.0;
    for (int i = 0; i < H; ++i) xg += orc_bf16_to_double(xt[i]) * orc_bf16_to_double(L->gate[i]);
    if (g_mut == MUT_GATE_SIGN) xg = -xg;
    double gamma = 1.0 / (1.0 + exp(-xg));
    if (tr && tr->gamma) tr->gamma[t] = gamma;
    if (tr && tr->zs)
      for (int n = 0; n < 2 * Is; ++n) tr->zs[(size_t)t * 2 * Is + n] = orc_bf16_from_double(zs[n]);
    if (tr && tr->hs)
      for (int n = 0; n < Is; ++n) tr->hs[(size_t)t * Is + n] = orc_bf16_from_double(hs[n]);
    if (tr && tr->ds)
      for (int m = 0; m < H; ++m) tr->ds[(size_t)t * H + m] = orc_bf16_from_double(ds[m]);
    /* combine: routed terms in rank order, shared term last ([D]) */
    for (int m = 0; m < H; ++m) {
      double yv = dsum[m] + gamma * ds[m];
      if (y_ref) y_ref[(size_t)t * H + m] = yv;
      if (y_bf16) y_bf16[(size_t)t * H + m] = orc_bf16_from_double(yv);
    }
  }
  free(logits); free(idx); free(w); free(xf); free(xq); free(sx); free(z); free(hf);
  free(hq); free(sh); free(dsum); free(zs); free(hs); free(ds);
  return 0;
}

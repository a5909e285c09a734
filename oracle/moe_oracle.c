/*
 * moe_oracle.c -- plain, slow CPU oracle for the DFlash MoE verify layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Arithmetic is in double unless a step says otherwise.  bf16 rounding
 * (round to nearest, ties to even, straight from double) happens only at the
 * declared rounding points: the SwiGLU product h, the layer output y (after
 * the residual add), the RMSNorm output, the attention q/k/v projections,
 * the attention output and the attention residual.
 *
 * Sources (page title, section):
 *  - "mlxfast -- Poolside Laguna XS 2.1 (DFlash)" README, "Why this challenge
 *    exists": 256 routed experts plus one shared expert, 8 experts per token,
 *    MoE intermediate 512, hidden 2048; routed/shared expert projections are
 *    NVFP4 4-bit group-16, routers/attention/lm_head stay bf16; GQA with 8 KV
 *    heads at head_dim 128; decode advances by the longest correct prefix.
 *  - mlxfast-challenge-dev PR #844, "4. What I ported" and "5. Numerical
 *    safety": the expert tail silu(gate)*up; top-k selection of the router
 *    scores, renormalisation of the selected weights, weighted expert sum,
 *    routed scaling factor, shared-expert add and decoder residual add, in
 *    that order.
 *  - PR #844, "5. Numerical safety", the retired-model trap: the verifier
 *    takes a greedy argmax over every verify row.
 *  - PR #844, "8. What I looked at": the routed gather reads an expert once
 *    per (row, slot); the layer's unique experts are what has to be read.
 *  - NVFP4 format: each element is an E2M1 code, each run of 16 consecutive
 *    elements along a row shares one E4M3 scale, and the projection carries
 *    one FP32 tensor scale; value = e2m1 * e4m3 * tensor_scale.
 *
 * Readings where the pages are silent: softmax scoring with top-k
 * renormalisation; exact ties in selection go to the lower index; router
 * and lm_head logits are formed in one fixed FP32 order (below) because an
 * integer decision depends on them;
 * RMSNorm with unit gain and eps 1e-6 before every MoE block, attention
 * block and the lm_head; low nibble holds the even column.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Formats by definition                                               */
/* ------------------------------------------------------------------ */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: value = m * 2^-1. */
double orc_e2m1(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? ldexp((double)m, -1) : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* E4M3 (OCP E4M3FN): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa.  Exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there
 * are no infinities. */
double orc_e4m3(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) mag = ldexp((double)m / 8.0, -6);
  else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* bf16 bit pattern -> exact double. */
double orc_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to bf16 (8 significant bits, exponent range of binary32),
 * nearest-even, directly from double (no intermediate float rounding). */
uint16_t orc_round_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e;
  frexp(a, &e);                       /* a in [2^(e-1), 2^e) */
  int q = e - 8;                      /* unit in the last place for 8 bits */
  if (q < -133) q = -133;             /* subnormal spacing 2^-133 */
  double r = ldexp(rint(ldexp(a, -q)), q);
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  float f = (float)r;                 /* exact */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* Decode tables built once from the definitions above. */
static double T_E2M1[16];
static double T_E4M3[256];
static int T_READY = 0;
static void orc_tables(void) {
  if (T_READY) return;
  for (int c = 0; c < 16; ++c) T_E2M1[c] = orc_e2m1(c);
  for (int c = 0; c < 256; ++c) T_E4M3[c] = orc_e4m3(c);
  T_READY = 1;
}

/* ------------------------------------------------------------------ */
/* Layer description (host pointers, row-major)                        */
/* ------------------------------------------------------------------ */

typedef struct {
  const uint8_t* codes;   /* [n_exp][rows][cols/2], even column in the low nibble */
  const uint8_t* scales;  /* [n_exp][rows][cols/16], E4M3 */
  const float* tscale;    /* [n_exp] */
} orc_proj;

typedef struct {
  int H, E, top_k, I, Is;
  double routed_scale;
  const uint16_t* router_w;  /* bf16 [E][H] */
  const float* router_b;     /* [E] or NULL */
  orc_proj gate, up, down;   /* gate/up: rows I, cols H; down: rows H, cols I */
  orc_proj sh_gate, sh_up, sh_down;  /* one expert; used when Is > 0 */
  int scoring;               /* 0: softmax, bias added to the logits;
                                1: sigmoid, bias added to the scores for the selection only */
} orc_layer;

/* Value of element (row r, column c) of expert e of a projection. */
static inline double nv_elem(const orc_proj* p, int e, int rows, int cols, int r, int c) {
  size_t row = (size_t)e * rows + r;
  uint8_t byte = p->codes[row * (cols / 2) + c / 2];
  int code = (c & 1) ? (byte >> 4) : (byte & 15);
  uint8_t sc = p->scales[row * (cols / 16) + c / 16];
  return T_E2M1[code] * T_E4M3[sc] * (double)p->tscale[e];
}

/* Dequantise one row of one expert into out[cols]. */
void orc_nvfp4_row(const orc_proj* p, int e, int rows, int cols, int r, double* out) {
  orc_tables();
  for (int c = 0; c < cols; ++c) out[c] = nv_elem(p, e, rows, cols, r, c);
}

/* Dequantise a whole expert matrix into out[rows][cols]. */
void orc_nvfp4_matrix(const orc_proj* p, int e, int rows, int cols, double* out) {
  orc_tables();
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c) out[(size_t)r * cols + c] = nv_elem(p, e, rows, cols, r, c);
}

/* ------------------------------------------------------------------ */
/* Logits of a bf16 GEMV in the fixed FP32 order (router and lm_head)  */
/* ------------------------------------------------------------------ */
/*
 * The order: 32 partial sums ("lanes").  Lane l adds, in float, the product
 * x[k]*w[k] for k = 256*j + 8*l + t with j = 0 .. H/256-1 outer and
 * t = 0 .. 7 inner.  A bf16*bf16 product is exact in float, so a fused
 * multiply-add gives the same result.  The 32 partials are then combined by
 * five pairwise rounds with partner distances 16, 8, 4, 2, 1 (after each
 * round every lane holds partial[l] + partial[l ^ d]), and lane 0's value is
 * the dot product.  The bias is added last, in float.
 */
static float dot_fixed_order(const uint16_t* x, const uint16_t* w, int H) {
  float acc[32];
  for (int l = 0; l < 32; ++l) acc[l] = 0.0f;
  for (int j = 0; j < H / 256; ++j)
    for (int l = 0; l < 32; ++l)
      for (int t = 0; t < 8; ++t) {
        int k = 256 * j + 8 * l + t;
        float p = (float)orc_bf16(x[k]) * (float)orc_bf16(w[k]);
        acc[l] = acc[l] + p;
      }
  for (int d = 16; d >= 1; d >>= 1) {
    float nxt[32];
    for (int l = 0; l < 32; ++l) nxt[l] = acc[l] + acc[l ^ d];
    memcpy(acc, nxt, sizeof acc);
  }
  return acc[0];
}

/* Router logits, FP32 fixed order: out[K][E]. */
void orc_router_logits_f32(const orc_layer* L, const uint16_t* x, int K, float* out) {
  for (int r = 0; r < K; ++r)
    for (int e = 0; e < L->E; ++e) {
      float v = dot_fixed_order(x + (size_t)r * L->H, L->router_w + (size_t)e * L->H, L->H);
      if (L->router_b) v = v + L->router_b[e];
      out[(size_t)r * L->E + e] = v;
    }
}

/* Router logits in double (for margins): out[K][E]. */
void orc_router_logits_f64(const orc_layer* L, const uint16_t* x, int K, double* out) {
  for (int r = 0; r < K; ++r)
    for (int e = 0; e < L->E; ++e) {
      double s = 0.0;
      for (int k = 0; k < L->H; ++k)
        s += orc_bf16(x[(size_t)r * L->H + k]) * orc_bf16(L->router_w[(size_t)e * L->H + k]);
      if (L->router_b) s += (double)L->router_b[e];
      out[(size_t)r * L->E + e] = s;
    }
}

/* ------------------------------------------------------------------ */
/* Softmax, top-k, renormalisation                                     */
/* ------------------------------------------------------------------ */

/* "a ranks before b": larger logit first, lower index on an exact tie. */
static int ranks_before(float la, int a, float lb, int b) {
  return (la > lb) || (la == lb && a < b);
}

/* For each row: softmax over all E logits (double), the k best experts in
 * rank order, and their probabilities divided by the selected sum. */
void orc_topk(const float* logits, int K, int E, int k, int32_t* idx, float* w) {
  int* sel = (int*)malloc(sizeof(int) * E);
  double* p = (double*)malloc(sizeof(double) * E);
  for (int r = 0; r < K; ++r) {
    const float* l = logits + (size_t)r * E;
    double mx = -INFINITY;
    for (int e = 0; e < E; ++e) if ((double)l[e] > mx) mx = l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp((double)l[e] - mx); z += p[e]; }
    for (int e = 0; e < E; ++e) p[e] /= z;
    for (int e = 0; e < E; ++e) sel[e] = 0;
    double ssum = 0.0;
    for (int s = 0; s < k; ++s) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (sel[e]) continue;
        if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
      }
      sel[best] = 1;
      idx[(size_t)r * k + s] = best;
      ssum += p[best];
    }
    for (int s = 0; s < k; ++s) w[(size_t)r * k + s] = (float)(p[idx[(size_t)r * k + s]] / ssum);
  }
  free(sel);
  free(p);
}

/* ------------------------------------------------------------------ */
/* Sigmoid scoring with a selection-only bias (the Laguna router tail)  */
/* ------------------------------------------------------------------ */
/*
 * PR #844, "4. What I ported", router-tail row: the router logits are cast
 * to FP32 and passed through a sigmoid, and a bias is added to the scores
 * for the selection only (the top-k is taken over score + bias); the
 * selected experts' own scores, renormalised over the selection, weight
 * their outputs (the renormalisation is deferred into the combine, fusion
 * row 4), and the routed sum is scaled (x2.5 in the Laguna checkpoint,
 * "5. Numerical safety").
 *
 * The selection is an integer decision taken on FP32 values, so the sigmoid
 * is defined as a fixed sequence of correctly rounded FP32 operations (the
 * kernel evaluates the same sequence): exp by Cody and Waite's argument
 * reduction (ln 2 split into a 16-bit head and a tail, so n * head is exact)
 * and the degree-7 Taylor polynomial of e^r on |r| <= ln2/2 (truncation
 * below 1e-8 relative), then 1 / (1 + e):
 *   l <- clamp(l, -80, 80);  t = -l
 *   n = rint(t * log2(e));   r = fma(-n, LN2_HI, t);  r = fma(-n, LN2_LO, r)
 *   p = ((((((c7 r + c6) r + c5) r + c4) r + c3) r + c2) r + c1) r + c0,  c_i = 1/i!
 *   e = p * 2^n   (exact: |n| <= 116 keeps 2^n and the product normal)
 *   s = 1 / (1 + e)
 */
static const float SG_LOG2E = 0x1.715476p+0f;   /* log2(e) rounded to float */
static const float SG_LN2_HI = 0x1.62e4p-1f;    /* 45426 / 2^16 */
static const float SG_LN2_LO = 0x1.7f7d1cp-20f; /* ln 2 - SG_LN2_HI, rounded to float */

float orc_sigmoid_f32(float l) {
  static const float c[8] = {1.0f, 1.0f, 0.5f, 0x1.555556p-3f, 0x1.555556p-5f, 0x1.111112p-7f,
                             0x1.6c16c2p-10f, 0x1.a01a02p-13f};  /* 1/i! rounded to float */
  if (l < -80.0f) l = -80.0f;
  if (l > 80.0f) l = 80.0f;
  float t = -l;
  float n = rintf(t * SG_LOG2E);
  float r = fmaf(-n, SG_LN2_HI, t);
  r = fmaf(-n, SG_LN2_LO, r);
  float p = c[7];
  for (int i = 6; i >= 0; --i) p = fmaf(p, r, c[i]);
  float e = p * ldexpf(1.0f, (int)n);
  return 1.0f / (1.0f + e);
}

/* For each row: scores s_e = sigmoid(l_e) (l without bias), selection keys
 * s_e + bias_e (FP32 add; bias NULL = 0), the k largest keys in rank order
 * (lower index on an exact tie), and weights s / sum of the selected s
 * (double, stored as float). */
void orc_topk_sigmoid(const float* logits, const float* bias, int K, int E, int k, int32_t* idx, float* w) {
  int* sel = (int*)malloc(sizeof(int) * E);
  float* sc = (float*)malloc(sizeof(float) * E);
  float* key = (float*)malloc(sizeof(float) * E);
  for (int r = 0; r < K; ++r) {
    const float* l = logits + (size_t)r * E;
    for (int e = 0; e < E; ++e) {
      sc[e] = orc_sigmoid_f32(l[e]);
      key[e] = bias ? sc[e] + bias[e] : sc[e];
      sel[e] = 0;
    }
    double ssum = 0.0;
    for (int s = 0; s < k; ++s) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (sel[e]) continue;
        if (best < 0 || ranks_before(key[e], e, key[best], best)) best = e;
      }
      sel[best] = 1;
      idx[(size_t)r * k + s] = best;
      ssum += (double)sc[best];
    }
    for (int s = 0; s < k; ++s) w[(size_t)r * k + s] = (float)((double)sc[idx[(size_t)r * k + s]] / ssum);
  }
  free(sel);
  free(sc);
  free(key);
}

/* ------------------------------------------------------------------ */
/* Grouping of (row, slot) pairs by expert                             */
/* ------------------------------------------------------------------ */
/*
 * Output layout (int32), with G = min(E, K*k):
 *   g[0]                 number of distinct experts n
 *   g[1 .. 1+G)          the distinct experts in ascending order, then -1
 *   g[1+G .. 2+2G)       offsets: pairs of expert u are g[off[u] .. off[u+1]),
 *                        off[u] = K*k for u >= n
 *   g[2+2G .. 2+2G+K*k)  pair ids r*k + s, grouped by expert, rows ascending
 */
void orc_group(const int32_t* idx, int K, int E, int k, int32_t* g) {
  int G = E < K * k ? E : K * k;
  int32_t* uexp = g + 1;
  int32_t* off = g + 1 + G;
  int32_t* pairs = g + 2 + 2 * G;
  int n = 0, pos = 0;
  for (int e = 0; e < E; ++e) {
    int used = 0;
    for (int q = 0; q < K * k; ++q) if (idx[q] == e) used = 1;
    if (!used) continue;
    uexp[n] = e;
    off[n] = pos;
    for (int r = 0; r < K; ++r)
      for (int s = 0; s < k; ++s)
        if (idx[r * k + s] == e) pairs[pos++] = r * k + s;
    ++n;
  }
  g[0] = n;
  for (int u = n; u < G; ++u) uexp[u] = -1;
  for (int u = n; u <= G; ++u) off[u] = pos;
}

/* ------------------------------------------------------------------ */
/* One expert on one row                                               */
/* ------------------------------------------------------------------ */

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* d[H] = Down_e * bf16(silu(Gate_e x) * (Up_e x)), all in double except the
 * declared rounding of h. */
static void expert_row(const orc_proj* gp, const orc_proj* upj, const orc_proj* dp, int e,
                       int H, int I, const double* x, double* h_scratch, double* d) {
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += nv_elem(gp, e, I, H, i, c) * x[c];
      u += nv_elem(upj, e, I, H, i, c) * x[c];
    }
    h_scratch[i] = orc_bf16(orc_round_bf16(silu(g) * u));
  }
  for (int j = 0; j < H; ++j) {
    double s = 0.0;
    for (int i = 0; i < I; ++i) s += nv_elem(dp, e, H, I, j, i) * h_scratch[i];
    d[j] = s;
  }
}

/* Expert e applied to one bf16 row: out[H] (double), h_out[I] (optional). */
void orc_expert(const orc_proj* gp, const orc_proj* upj, const orc_proj* dp, int e, int H, int I,
                const uint16_t* x_bf16, double* out, double* h_out) {
  orc_tables();
  double* x = (double*)malloc(sizeof(double) * H);
  double* h = (double*)malloc(sizeof(double) * I);
  for (int c = 0; c < H; ++c) x[c] = orc_bf16(x_bf16[c]);
  expert_row(gp, upj, dp, e, H, I, x, h, out);
  if (h_out) memcpy(h_out, h, sizeof(double) * I);
  free(x);
  free(h);
}

/* ------------------------------------------------------------------ */
/* The MoE verify layer                                                */
/* ------------------------------------------------------------------ */
/*
 * For each row r: route (fixed-order FP32 logits, softmax, top-k,
 * renormalise; or, with scoring 1, sigmoid scores, top-k of score + bias,
 * renormalised scores), evaluate each selected expert, and form
 *   y_r = bf16( routed_scale * sum_{s=0..k-1} w_{r,s} d_{r,s}
 *               + d_shared_r + residual_r )
 * with the slot sum taken in slot order.  idx, w, group and y_f64 (the value
 * before the final rounding) are optional outputs.
 */
void orc_moe_layer(const orc_layer* L, const uint16_t* x_norm, int K, const uint16_t* residual,
                   uint16_t* y, int32_t* idx_out, float* w_out, int32_t* group_out, double* y_f64) {
  orc_tables();
  const int H = L->H, E = L->E, k = L->top_k, I = L->I;
  float* logits = (float*)malloc(sizeof(float) * (size_t)K * E);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)K * k);
  float* w = (float*)malloc(sizeof(float) * (size_t)K * k);
  if (L->scoring == 1) {  /* sigmoid scores; the bias only steers the selection */
    orc_layer nob = *L;
    nob.router_b = NULL;
    orc_router_logits_f32(&nob, x_norm, K, logits);
    orc_topk_sigmoid(logits, L->router_b, K, E, k, idx, w);
  } else {
    orc_router_logits_f32(L, x_norm, K, logits);
    orc_topk(logits, K, E, k, idx, w);
  }
  if (group_out) orc_group(idx, K, E, k, group_out);

  /* d[r][s][H], slot k holds the shared expert */
  double* d = (double*)calloc((size_t)K * (k + 1) * H, sizeof(double));
  #pragma omp parallel
  {
    double* x = (double*)malloc(sizeof(double) * H);
    double* h = (double*)malloc(sizeof(double) * (I > L->Is ? I : L->Is));
    #pragma omp for schedule(dynamic, 1)
    for (int q = 0; q < K * (k + 1); ++q) {
      int r = q / (k + 1), s = q % (k + 1);
      for (int c = 0; c < H; ++c) x[c] = orc_bf16(x_norm[(size_t)r * H + c]);
      double* dst = d + (size_t)q * H;
      if (s < k) expert_row(&L->gate, &L->up, &L->down, idx[r * k + s], H, I, x, h, dst);
      else if (L->Is > 0) expert_row(&L->sh_gate, &L->sh_up, &L->sh_down, 0, H, L->Is, x, h, dst);
    }
    free(x);
    free(h);
  }
  for (int r = 0; r < K; ++r)
    for (int j = 0; j < H; ++j) {
      double acc = 0.0;
      for (int s = 0; s < k; ++s) acc += (double)w[r * k + s] * d[((size_t)r * (k + 1) + s) * H + j];
      double v = L->routed_scale * acc + d[((size_t)r * (k + 1) + k) * H + j];
      if (residual) v += orc_bf16(residual[(size_t)r * H + j]);
      if (y_f64) y_f64[(size_t)r * H + j] = v;
      if (y) y[(size_t)r * H + j] = orc_round_bf16(v);
    }
  if (idx_out) memcpy(idx_out, idx, sizeof(int32_t) * (size_t)K * k);
  if (w_out) memcpy(w_out, w, sizeof(float) * (size_t)K * k);
  free(d);
  free(logits);
  free(idx);
  free(w);
}

/* ------------------------------------------------------------------ */
/* RMSNorm, attention, lm_head, acceptance                             */
/* ------------------------------------------------------------------ */

/* RMSNorm with unit gain: out = bf16( x * 1/sqrt(mean(x^2) + eps) ).
 * Its output feeds the router's top-k, an integer decision, so it is taken
 * in FP32 in the fixed order of the router logits: the sum of squares is the
 * fixed-order dot product of the row with itself, then mean = ss / H,
 * inv = 1 / sqrt(mean + eps) and x * inv, each a correctly rounded FP32
 * operation, and the product is rounded to bf16. */
void orc_rmsnorm(const uint16_t* x, int K, int H, double eps, uint16_t* out) {
  const float epsf = (float)eps;
  for (int r = 0; r < K; ++r) {
    const uint16_t* row = x + (size_t)r * H;
    float ss = dot_fixed_order(row, row, H);
    float mean = ss / (float)H;
    float inv = 1.0f / sqrtf(mean + epsf);
    for (int c = 0; c < H; ++c) {
      float v = (float)orc_bf16(row[c]) * inv;
      out[(size_t)r * H + c] = orc_round_bf16((double)v);
    }
  }
}

/* out[K][N] = bf16( x[K][D] . W[N][D]^T ), double accumulation. */
void orc_linear_bf16(const uint16_t* x, const uint16_t* W, int K, int D, int N, uint16_t* out) {
  #pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n)
    for (int r = 0; r < K; ++r) {
      double s = 0.0;
      for (int c = 0; c < D; ++c) s += orc_bf16(x[(size_t)r * D + c]) * orc_bf16(W[(size_t)n * D + c]);
      out[(size_t)r * N + n] = orc_round_bf16(s);
    }
}

/*
 * GQA attention of K new rows over a cache of C positions plus the K new
 * positions (row r sees cache 0..C-1 and new positions 0..r).
 *   x[K][H] (bf16): the block input (the residual stream)
 *   Wq [nq*hd][H], Wk, Wv [nkv*hd][H], Wo [H][nq*hd] (bf16)
 *   kc, vc [nkv][C][hd] (bf16): the cache
 *   x_out[K][H] = bf16( x + o . Wo^T ), o = bf16(softmax(q k^T / sqrt(hd)) v)
 *   o_out[K][nq*hd] (optional): o itself
 * The block's own input normalisation is applied first (orc_rmsnorm).
 */
void orc_attention(const uint16_t* x, int K, int H, int nq, int nkv, int hd, int C,
                   const uint16_t* Wq, const uint16_t* Wk, const uint16_t* Wv, const uint16_t* Wo,
                   const uint16_t* kc, const uint16_t* vc, double eps, uint16_t* x_out, uint16_t* o_out) {
  int QD = nq * hd, KD = nkv * hd, grp = nq / nkv;
  uint16_t* xn = (uint16_t*)malloc(2 * (size_t)K * H);
  uint16_t* q = (uint16_t*)malloc(2 * (size_t)K * QD);
  uint16_t* kn = (uint16_t*)malloc(2 * (size_t)K * KD);
  uint16_t* vn = (uint16_t*)malloc(2 * (size_t)K * KD);
  uint16_t* o = (uint16_t*)malloc(2 * (size_t)K * QD);
  orc_rmsnorm(x, K, H, eps, xn);
  orc_linear_bf16(xn, Wq, K, H, QD, q);
  orc_linear_bf16(xn, Wk, K, H, KD, kn);
  orc_linear_bf16(xn, Wv, K, H, KD, vn);
  double scale = 1.0 / sqrt((double)hd);
  #pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int r = 0; r < K; ++r)
    for (int h = 0; h < nq; ++h) {
      int kvh = h / grp;
      int n = C + r + 1;
      double* sc = (double*)malloc(sizeof(double) * n);
      const uint16_t* qv = q + (size_t)r * QD + (size_t)h * hd;
      double mx = -INFINITY;
      for (int p = 0; p < n; ++p) {
        const uint16_t* kv = (p < C) ? kc + ((size_t)kvh * C + p) * hd
                                     : kn + (size_t)(p - C) * KD + (size_t)kvh * hd;
        double s = 0.0;
        for (int c = 0; c < hd; ++c) s += orc_bf16(qv[c]) * orc_bf16(kv[c]);
        sc[p] = s * scale;
        if (sc[p] > mx) mx = sc[p];
      }
      double z = 0.0;
      for (int p = 0; p < n; ++p) { sc[p] = exp(sc[p] - mx); z += sc[p]; }
      for (int c = 0; c < hd; ++c) {
        double acc = 0.0;
        for (int p = 0; p < n; ++p) {
          const uint16_t* vv = (p < C) ? vc + ((size_t)kvh * C + p) * hd
                                       : vn + (size_t)(p - C) * KD + (size_t)kvh * hd;
          acc += (sc[p] / z) * orc_bf16(vv[c]);
        }
        o[(size_t)r * QD + (size_t)h * hd + c] = orc_round_bf16(acc);
      }
      free(sc);
    }
  for (int r = 0; r < K; ++r)
    for (int j = 0; j < H; ++j) {
      double s = 0.0;
      for (int c = 0; c < QD; ++c) s += orc_bf16(o[(size_t)r * QD + c]) * orc_bf16(Wo[(size_t)j * QD + c]);
      x_out[(size_t)r * H + j] = orc_round_bf16(orc_bf16(x[(size_t)r * H + j]) + s);
    }
  if (o_out) memcpy(o_out, o, 2 * (size_t)K * QD);
  free(xn); free(q); free(kn); free(vn); free(o);
}

/* ------------------------------------------------------------------ */
/* Rotary position embedding (RoPE) with YaRN frequency scaling         */
/* ------------------------------------------------------------------ */
/*
 * README, "Why this challenge exists": sliding-window layers use plain RoPE
 * at theta 10000, full-attention layers YaRN rotary with a 0.5
 * partial-rotary factor.  Rotary dims: the first rd of a head; pair i < rd/2
 * is (v[i], v[i + rd/2]) ("rotate half"), rotated by angle p * f_i at
 * position p, f_i = theta^(-2i/rd).  YaRN (Peng et al., "YaRN: Efficient
 * Context Window Extension of Large Language Models", NTK-by-parts) with
 * factor s > 1 and original context L0: r_i = L0 * f_i / (2 pi) (rotations
 * of pair i over L0 positions), ramp g_i = clamp((r_i - 1) / (32 - 1), 0, 1),
 * f_i <- (1 - g_i) f_i / s + g_i f_i; and the attention logits are scaled by
 * (0.1 ln s + 1)^2 (the temperature applied to both q and k).
 */
void orc_rope_freqs(int rd, double theta, double yarn_s, int yarn_l0, double* f) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < rd / 2; ++i) {
    double fi = pow(theta, -2.0 * i / rd);
    if (yarn_s > 1.0) {
      double r = (double)yarn_l0 * fi / two_pi;
      double g = (r - 1.0) / (32.0 - 1.0);
      if (g < 0.0) g = 0.0;
      if (g > 1.0) g = 1.0;
      fi = (1.0 - g) * fi / yarn_s + g * fi;
    }
    f[i] = fi;
  }
}

/* Rotates one head vector v[hd] (double, in place) at position p. */
void orc_rope_vec(double* v, int rd, const double* f, double p) {
  for (int i = 0; i < rd / 2; ++i) {
    double a = p * f[i], c = cos(a), s = sin(a);
    double x0 = v[i], x1 = v[i + rd / 2];
    v[i] = x0 * c - x1 * s;
    v[i + rd / 2] = x1 * c + x0 * s;
  }
}

/* The rows [K][n_heads * hd] (bf16) rotated at positions pos0 + r, rounded
 * to bf16 again. */
static void rope_rows_bf16(uint16_t* x, int K, int n_heads, int hd, int rd, const double* f, int pos0) {
  double* v = (double*)malloc(sizeof(double) * hd);
  for (int r = 0; r < K; ++r)
    for (int h = 0; h < n_heads; ++h) {
      uint16_t* xv = x + (size_t)r * n_heads * hd + (size_t)h * hd;
      for (int c = 0; c < hd; ++c) v[c] = orc_bf16(xv[c]);
      orc_rope_vec(v, rd, f, (double)(pos0 + r));
      for (int c = 0; c < hd; ++c) xv[c] = orc_round_bf16(v[c]);
    }
  free(v);
}

/*
 * The attention block of a Laguna layer: as orc_attention, with RoPE / YaRN
 * on q and the new keys (rd = 0: none), the rows at positions C .. C+K-1, and
 * a sliding window of `window` positions (0: none): row r at position
 * p = C + r sees positions max(0, p - window + 1) .. p.
 *   k_new_out, v_new_out [K][nkv*hd] (optional): the (rotated) new keys and
 *   the new values; o_out [K][nq*hd] (optional).
 */
void orc_attention_ex(const uint16_t* x, int K, int H, int nq, int nkv, int hd, int C, const uint16_t* Wq,
                      const uint16_t* Wk, const uint16_t* Wv, const uint16_t* Wo, const uint16_t* kc,
                      const uint16_t* vc, double eps, int window, int rd, double theta, double yarn_s, int yarn_l0,
                      uint16_t* x_out, uint16_t* k_new_out, uint16_t* v_new_out, uint16_t* o_out) {
  int QD = nq * hd, KD = nkv * hd, grp = nq / nkv;
  uint16_t* xn = (uint16_t*)malloc(2 * (size_t)K * H);
  uint16_t* q = (uint16_t*)malloc(2 * (size_t)K * QD);
  uint16_t* kn = (uint16_t*)malloc(2 * (size_t)K * KD);
  uint16_t* vn = (uint16_t*)malloc(2 * (size_t)K * KD);
  uint16_t* o = (uint16_t*)malloc(2 * (size_t)K * QD);
  double f[256];
  orc_rmsnorm(x, K, H, eps, xn);
  orc_linear_bf16(xn, Wq, K, H, QD, q);
  orc_linear_bf16(xn, Wk, K, H, KD, kn);
  orc_linear_bf16(xn, Wv, K, H, KD, vn);
  double temp = 1.0;
  if (rd > 0) {
    orc_rope_freqs(rd, theta, yarn_s, yarn_l0, f);
    rope_rows_bf16(q, K, nq, hd, rd, f, C);
    rope_rows_bf16(kn, K, nkv, hd, rd, f, C);
    if (yarn_s > 1.0) temp = (0.1 * log(yarn_s) + 1.0) * (0.1 * log(yarn_s) + 1.0);
  }
  double scale = temp / sqrt((double)hd);
  #pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int r = 0; r < K; ++r)
    for (int h = 0; h < nq; ++h) {
      int kvh = h / grp;
      int p_row = C + r;
      int lo = (window > 0 && p_row - window + 1 > 0) ? p_row - window + 1 : 0;
      int n = C + r + 1;
      double* sc = (double*)malloc(sizeof(double) * n);
      const uint16_t* qv = q + (size_t)r * QD + (size_t)h * hd;
      double mx = -INFINITY;
      for (int p = 0; p < n; ++p) {
        if (p < lo) { sc[p] = -INFINITY; continue; }
        const uint16_t* kv = (p < C) ? kc + ((size_t)kvh * C + p) * hd
                                     : kn + (size_t)(p - C) * KD + (size_t)kvh * hd;
        double s = 0.0;
        for (int c = 0; c < hd; ++c) s += orc_bf16(qv[c]) * orc_bf16(kv[c]);
        sc[p] = s * scale;
        if (sc[p] > mx) mx = sc[p];
      }
      double z = 0.0;
      for (int p = 0; p < n; ++p) { sc[p] = (p < lo) ? 0.0 : exp(sc[p] - mx); z += sc[p]; }
      for (int c = 0; c < hd; ++c) {
        double acc = 0.0;
        for (int p = lo; p < n; ++p) {
          const uint16_t* vv = (p < C) ? vc + ((size_t)kvh * C + p) * hd
                                       : vn + (size_t)(p - C) * KD + (size_t)kvh * hd;
          acc += (sc[p] / z) * orc_bf16(vv[c]);
        }
        o[(size_t)r * QD + (size_t)h * hd + c] = orc_round_bf16(acc);
      }
      free(sc);
    }
  for (int r = 0; r < K; ++r)
    for (int j = 0; j < H; ++j) {
      double s = 0.0;
      for (int c = 0; c < QD; ++c) s += orc_bf16(o[(size_t)r * QD + c]) * orc_bf16(Wo[(size_t)j * QD + c]);
      x_out[(size_t)r * H + j] = orc_round_bf16(orc_bf16(x[(size_t)r * H + j]) + s);
    }
  if (k_new_out) memcpy(k_new_out, kn, 2 * (size_t)K * KD);
  if (v_new_out) memcpy(v_new_out, vn, 2 * (size_t)K * KD);
  if (o_out) memcpy(o_out, o, 2 * (size_t)K * QD);
  free(xn); free(q); free(kn); free(vn); free(o);
}

/* The dense bf16 SwiGLU MLP of Laguna's layer 0 (README, "Why this
 * challenge exists": layer 0 has a dense MLP, intermediate 8192):
 *   h = bf16( silu(x_norm . Wg^T) * (x_norm . Wu^T) )   [K][I]
 *   y = bf16( residual + h . Wd^T )                      [K][H]
 * dot products in double, the same rounding points as the experts. */
void orc_dense_mlp(const uint16_t* x_norm, const uint16_t* residual, const uint16_t* Wg, const uint16_t* Wu,
                   const uint16_t* Wd, int K, int H, int I, uint16_t* y) {
  double* h = (double*)malloc(sizeof(double) * (size_t)K * I);
  #pragma omp parallel for schedule(static)
  for (int i = 0; i < I; ++i)
    for (int r = 0; r < K; ++r) {
      double g = 0.0, u = 0.0;
      for (int c = 0; c < H; ++c) {
        double xv = orc_bf16(x_norm[(size_t)r * H + c]);
        g += xv * orc_bf16(Wg[(size_t)i * H + c]);
        u += xv * orc_bf16(Wu[(size_t)i * H + c]);
      }
      h[(size_t)r * I + i] = orc_bf16(orc_round_bf16(silu(g) * u));
    }
  #pragma omp parallel for schedule(static)
  for (int j = 0; j < H; ++j)
    for (int r = 0; r < K; ++r) {
      double s = 0.0;
      for (int i = 0; i < I; ++i) s += h[(size_t)r * I + i] * orc_bf16(Wd[(size_t)j * I + i]);
      double v = s + (residual ? orc_bf16(residual[(size_t)r * H + j]) : 0.0);
      y[(size_t)r * H + j] = orc_round_bf16(v);
    }
  free(h);
}

/* lm_head greedy token per row: argmax over V of the fixed-order FP32
 * logits of x_norm[r] . W[v]; an exact tie goes to the lower index.
 * best_logit (optional) receives the winning FP32 logit. */
void orc_lm_argmax(const uint16_t* x_norm, const uint16_t* W, int K, int H, int V,
                   int32_t* tok, float* best_logit) {
  for (int r = 0; r < K; ++r) {
    int best = -1;
    float bl = 0.0f;
    #pragma omp parallel
    {
      int lb = -1;
      float ll = 0.0f;
      #pragma omp for schedule(static)
      for (int v = 0; v < V; ++v) {
        float l = dot_fixed_order(x_norm + (size_t)r * H, W + (size_t)v * H, H);
        if (lb < 0 || ranks_before(l, v, ll, lb)) { lb = v; ll = l; }
      }
      #pragma omp critical
      {
        if (lb >= 0 && (best < 0 || ranks_before(ll, lb, bl, best))) { best = lb; bl = ll; }
      }
    }
    tok[r] = best;
    if (best_logit) best_logit[r] = bl;
  }
}

/* Accepted prefix: the first i with draft[i] != target[i], else K. */
int orc_accept_prefix(const int32_t* draft, const int32_t* target, int K) {
  for (int i = 0; i < K; ++i) if (draft[i] != target[i]) return i;
  return K;
}

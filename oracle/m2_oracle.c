/*
 * m2_oracle.c -- plain, slow CPU oracle for the Nemotron-H Mamba-2 layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or constant generator with the CUDA
 * library: every function below is written from the definitions on the pages.
 *
 * Arithmetic is IEEE double.  Values are rounded to bfloat16 only at the six
 * rounding points the layer's "a16" activations imply (R1..R6 below); the SSM
 * state and everything between rounding points stay in double.
 *
 * Sources (page title, then the section on that page):
 *   [SRC]  spark_model/layers/nemotron_mamba2.rs -- module header "Forward pass"
 *          steps 1..8; `conv1d_update_biased` (conv with learned bias);
 *          `ssm_decode` (arguments of the SSM decode step, dt_min=1e-9,
 *          dt_max=1e9 "no effective clamp"); struct fields (h_state is fp32
 *          [num_heads, head_dim, state_size]).
 *   [QWEN] Struct Qwen3SsmLayer -- `set_fp8_decode_weights`: the w8a16 GEMV
 *          out[n] = sum_k A[k] * E4M3(B[n,k]) * block_scale[n/BS, k/BS], BS=128,
 *          scales [N/BS, K/BS] BF16.
 *   [NEMO] Struct NemotronMamba2Layer -- `set_fp8_weights`: the scale index
 *          block_scale[n/128 * k_blocks + k/128].
 *   [TRAIT] Trait TransformerLayer -- `decode` (hidden modified in place),
 *          `prefill` ("Default: falls back to sequential single-token decode
 *          calls"), `decode_multi_seq` (N sequences, one token each, own state).
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - E4M3 is the OCP "E4M3FN" encoding: bias 7, no infinities, S.1111.111 is NaN.
 *   - Rounding points: R1 hidden input is bf16; R2 RMSNorm output -> bf16;
 *     R3 in_proj output -> bf16; R4 conv output -> bf16; R5 gated-norm output ->
 *     bf16; R6 (hidden_in + out_proj) -> bf16 once.  bf16 rounding is
 *     round-to-nearest-even.
 *   - in_proj output order [z | xBC | dt]; xBC = [x | B (group-major) | C].
 *   - conv state: (d_conv-1) bf16 slots per channel used as a ring; `pos` counts
 *     tokens seen; token t is stored in slot t mod (d_conv-1).  The window from
 *     oldest to newest is slots pos, pos+1, .. (mod d_conv-1), then the current
 *     token; tap j multiplies window element j (tap d_conv-1 = current token).
 *   - head h uses group g = h / (H/G).
 *   - softplus(v) = log1p(exp(v)), and v itself for v > 20.
 *   - RMSNorm multiplies by the weight (not 1+weight); gated RMSNorm normalises
 *     y over groups of `group` elements (the whole d_inner by default), then
 *     multiplies by the weight and by silu(z).
 *   - residual: out = hidden_in + out_proj(...), a self-contained pre-norm block.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- formats */

/* E4M3FN closed form: for exponent field e>0, (-1)^s * 2^(e-7) * (1 + m/8);
 * for e=0, (-1)^s * 2^-6 * (m/8); 0x7F and 0xFF are NaN. */
double or_e4m3_to_f64(uint8_t b) {
  int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* bfloat16 is the top half of an IEEE binary32: sign, 8 exponent bits, 7
 * fraction bits. */
double or_bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bfloat16, ties to even, directly (one rounding,
 * not double->float->bf16).  Normal bf16 values carry 8 significant bits; below
 * 2^-126 the spacing is fixed at 2^-133 (subnormals).  Overflow goes to inf. */
uint16_t or_f64_to_bf16(double v) {
  if (isnan(v)) return signbit(v) ? 0xFFC0 : 0x7FC0;
  int neg = signbit(v) ? 1 : 0;
  double a = fabs(v);
  double r;
  if (a == 0.0) {
    r = 0.0;
  } else if (isinf(a)) {
    r = INFINITY;
  } else {
    int e;
    frexp(a, &e); /* a = f * 2^e, 0.5 <= f < 1 */
    int q_exp = (e - 1 >= -126) ? (e - 1 - 7) : -133; /* value of one ulp */
    double q = ldexp(a, -q_exp);                      /* exact scaling     */
    double qr = nearbyint(q);                         /* default mode: RNE */
    r = ldexp(qr, q_exp);
    /* largest finite bf16 = (2 - 2^-7) * 2^127; anything rounding above it
     * (i.e. a >= max + half ulp, ties going to the even "2^128") is inf */
    if (r > ldexp(2.0 - ldexp(1.0, -7), 127)) r = INFINITY;
  }
  float f = (float)r; /* exact: r is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t h = (uint16_t)(u >> 16);
  if (neg) h |= 0x8000;
  return h;
}

static double g_e4m3_table[256];
static int g_init = 0;

void or_init(void) {
  for (int b = 0; b < 256; ++b) g_e4m3_table[b] = or_e4m3_to_f64((uint8_t)b);
  g_init = 1;
}

static double e4m3(uint8_t b) {
  if (!g_init) or_init();
  return g_e4m3_table[b];
}

static double bf(uint16_t h) { return or_bf16_to_f64(h); }

/* ----------------------------------------------------------- elementwise */

double or_softplus(double v) { return v > 20.0 ? v : log1p(exp(v)); }

double or_silu(double v) { return v / (1.0 + exp(-v)); }

/* ---------------------------------------------------------------- step 1 */

/* RMSNorm with weight*x scaling ([SRC] step 1): out = x / sqrt(mean(x^2)+eps) * w,
 * rounded to bf16 (R2). */
void or_rmsnorm(const uint16_t* x, const uint16_t* w, int K, double eps, uint16_t* out) {
  double ss = 0.0;
  for (int k = 0; k < K; ++k) ss += bf(x[k]) * bf(x[k]);
  double r = 1.0 / sqrt(ss / (double)K + eps);
  for (int k = 0; k < K; ++k) out[k] = or_f64_to_bf16(bf(x[k]) * r * bf(w[k]));
}

/* ---------------------------------------------------------------- step 2 / 7 */

/* The w8a16 GEMV ([QWEN] set_fp8_decode_weights; [NEMO] set_fp8_weights):
 *   out[m][n] = sum_k A[m][k] * E4M3(W[n][k]) * S[(n/128)*kb + k/128],
 * with kb = ceil(K/128), summed with k ascending, unrounded (double). */
void or_w8a16_gemv(const uint16_t* A, int M, const uint8_t* W, const uint16_t* S, int N, int K,
                   double* out) {
  int kb = (K + 127) / 128;
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    const uint8_t* wrow = W + (size_t)n * K;
    const uint16_t* srow = S + (size_t)(n / 128) * kb;
    for (int m = 0; m < M; ++m) {
      const uint16_t* a = A + (size_t)m * K;
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += bf(a[k]) * e4m3(wrow[k]) * bf(srow[k / 128]);
      out[(size_t)m * N + n] = acc;
    }
  }
}

/* Dense BF16-weight GEMV of the unquantised projections ([SRC] struct field
 * comment on native BF16 projections): out[m][n] = sum_k A[m][k] * W[n][k]. */
void or_bf16_gemv(const uint16_t* A, int M, const uint16_t* W, int N, int K, double* out) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    const uint16_t* wrow = W + (size_t)n * K;
    for (int m = 0; m < M; ++m) {
      const uint16_t* a = A + (size_t)m * K;
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += bf(a[k]) * bf(wrow[k]);
      out[(size_t)m * N + n] = acc;
    }
  }
}

/* Sum of |terms| of the same products, sum_k |A[k] * W~[n][k]| (fmt 1: E4M3
 * with block scales, 2: bf16): the scale of the summation error of any
 * floating-point evaluation of the dot product.  Used only where tests judge
 * rounding decisions. */
void or_proj_abs(int fmt, const void* w, const uint16_t* s, const uint16_t* a, int N, int K, double* out) {
  int kb = (K + 127) / 128;
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int k = 0; k < K; ++k) {
      double wv = fmt == 1 ? e4m3(((const uint8_t*)w)[(size_t)n * K + k]) * bf(s[(size_t)(n / 128) * kb + k / 128])
                           : bf(((const uint16_t*)w)[(size_t)n * K + k]);
      acc += fabs(bf(a[k]) * wv);
    }
    out[n] = acc;
  }
}

/* ---------------------------------------------------------------- step 3 */

/* One-token causal depthwise conv update with learned bias and fused SiLU
 * ([SRC] step 3 and `conv1d_update_biased`).  ring is [(d_conv-1)][C] bf16;
 * *pos is the number of tokens seen so far (not advanced here).  The current
 * token x (bf16, R3) is used as tap d_conv-1 and then stored into slot
 * pos mod (d_conv-1).  Output rounded to bf16 (R4). */
void or_conv1d_update_exact(uint16_t* ring, const int32_t* pos, const uint16_t* x, const uint16_t* w,
                                const uint16_t* b, int C, int dconv, int silu, uint16_t* out, double* exact,
                                double* exact_abs) {
  int L = dconv - 1;
  int p = *pos;
  for (int c = 0; c < C; ++c) {
    double acc = b ? bf(b[c]) : 0.0;
    double aacc = fabs(acc);
    for (int j = 0; j < L; ++j) {
      int slot = (p + j) % L; /* oldest first */
      acc += bf(w[(size_t)c * dconv + j]) * bf(ring[(size_t)slot * C + c]);
      aacc += fabs(bf(w[(size_t)c * dconv + j]) * bf(ring[(size_t)slot * C + c]));
    }
    acc += bf(w[(size_t)c * dconv + L]) * bf(x[c]);
    aacc += fabs(bf(w[(size_t)c * dconv + L]) * bf(x[c]));
    double v = silu ? or_silu(acc) : acc;
    if (exact) exact[c] = v;
    if (exact_abs) exact_abs[c] = aacc;
    out[c] = or_f64_to_bf16(v);
  }
  int wslot = p % L;
  for (int c = 0; c < C; ++c) ring[(size_t)wslot * C + c] = x[c];
}

void or_conv1d_update(uint16_t* ring, const int32_t* pos, const uint16_t* x, const uint16_t* w,
                      const uint16_t* b, int C, int dconv, int silu, uint16_t* out) {
  or_conv1d_update_exact(ring, pos, x, w, b, C, dconv, silu, out, NULL, NULL);
}

/* ---------------------------------------------------------------- step 5 */

/* Mamba-2 SSM decode step ([SRC] step 5 and `ssm_decode`), one sequence:
 *   dt = clamp(softplus(dt_raw[h] + dt_bias[h]), 1e-9, 1e9)
 *   A  = -exp(A_log[h]);  dA = exp(dt * A)
 *   h[h][p][n] = dA * h[h][p][n] + dt * x[h*P+p] * B[g*N+n]
 *   y[h*P+p]   = sum_n C[g*N+n] * h[h][p][n] + D[h] * x[h*P+p]
 * with g = h / (H/G).  h and y in double; *clamp_hits counts clamp events. */
static void ssm_step_impl(double* hs, const uint16_t* x, const uint16_t* Bm, const uint16_t* Cm,
                          const uint16_t* dt_raw, const float* A_log, const float* D, const float* dt_bias,
                          int H, int P, int N, int G, double* y, double* y_abs, long* clamp_hits);

void or_ssm_step(double* hs, const uint16_t* x, const uint16_t* Bm, const uint16_t* Cm,
                 const uint16_t* dt_raw, const float* A_log, const float* D, const float* dt_bias,
                 int H, int P, int N, int G, double* y, long* clamp_hits) {
  ssm_step_impl(hs, x, Bm, Cm, dt_raw, A_log, D, dt_bias, H, P, N, G, y, NULL, clamp_hits);
}

/* The same step; y_abs (if not NULL) receives sum_n |C h| + |D x| per output,
 * the scale of the evaluation error of y. */
static void ssm_step_impl(double* hs, const uint16_t* x, const uint16_t* Bm, const uint16_t* Cm,
                          const uint16_t* dt_raw, const float* A_log, const float* D, const float* dt_bias,
                          int H, int P, int N, int G, double* y, double* y_abs, long* clamp_hits) {
  int hpg = H / G;
  for (int h = 0; h < H; ++h) {
    int g = h / hpg;
    double dt = or_softplus(bf(dt_raw[h]) + (double)dt_bias[h]);
    if (dt < 1e-9) { dt = 1e-9; if (clamp_hits) ++*clamp_hits; }
    if (dt > 1e9) { dt = 1e9; if (clamp_hits) ++*clamp_hits; }
    double A = -exp((double)A_log[h]);
    double dA = exp(dt * A);
    for (int p = 0; p < P; ++p) {
      double xv = bf(x[h * P + p]);
      double* hrow = hs + ((size_t)h * P + p) * N;
      double acc = 0.0, aacc = 0.0;
      for (int n = 0; n < N; ++n) {
        hrow[n] = dA * hrow[n] + dt * xv * bf(Bm[g * N + n]);
        acc += bf(Cm[g * N + n]) * hrow[n];
        aacc += fabs(bf(Cm[g * N + n]) * hrow[n]);
      }
      y[h * P + p] = acc + (double)D[h] * xv;
      if (y_abs) y_abs[h * P + p] = aacc + fabs((double)D[h] * xv);
    }
  }
}

/* ---------------------------------------------------------------- step 6 */

/* Gated RMSNorm ([SRC] step 6, "rms_norm(y, ssm_norm) * silu(z)"): for each
 * group of `group` consecutive elements, out = y / sqrt(mean(y^2)+eps) * w *
 * silu(z), rounded to bf16 (R5). */
void or_gated_rmsnorm(const double* y, const uint16_t* z, const uint16_t* w, int d, int group,
                      double eps, uint16_t* out) {
  for (int g0 = 0; g0 < d; g0 += group) {
    double ss = 0.0;
    for (int i = g0; i < g0 + group; ++i) ss += y[i] * y[i];
    double r = 1.0 / sqrt(ss / (double)group + eps);
    for (int i = g0; i < g0 + group; ++i)
      out[i] = or_f64_to_bf16(y[i] * r * bf(w[i]) * or_silu(bf(z[i])));
  }
}

/* The gated RMSNorm's unrounded outputs (exact[d]) and, from y's own scale
 * y_abs[d], the scale of their evaluation error: |r * w * silu(z)| * y_abs + |exact|. */
static void gated_rmsnorm_exact(const double* y, const double* y_abs, const uint16_t* z, const uint16_t* w, int d,
                                int group, double eps, double* exact, double* scale) {
  for (int g0 = 0; g0 < d; g0 += group) {
    double ss = 0.0;
    for (int i = g0; i < g0 + group; ++i) ss += y[i] * y[i];
    double r = 1.0 / sqrt(ss / (double)group + eps);
    for (int i = g0; i < g0 + group; ++i) {
      double f = r * bf(w[i]) * or_silu(bf(z[i]));
      exact[i] = y[i] * f;
      scale[i] = fabs(f) * y_abs[i] + fabs(exact[i]);
    }
  }
}

/* ---------------------------------------------------------------- W8A8 arm */

/* The W8A8 projections (FP8 activations as well as weights).  The pages give
 * FP8 GEMMs and a bf16 -> FP8 activation conversion for prefill but not its
 * scaling; the reading used here: per row and 128-element k block,
 * amax = max |a|; the block's codes are E4M3(a * (448 / amax)) and its scale
 * amax / 448, both computed in fp32 (an all-zero block has scale 0, codes 0).
 * E4M3 rounding is round-to-nearest-even with saturation to +-448. */

/* fp32 -> E4M3FN code, round to nearest even, saturating to +-448. */
uint8_t or_f32_to_e4m3_sat(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0;
  double a = fabs((double)v);
  if (a != a) return 0x7F; /* NaN (not produced by the quantizer) */
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormals: multiples of 2^-9; 8 * 2^-9 = 2^-6 is the first normal (code 0x08) */
    double r = nearbyint(a * 512.0);
    return sign | (uint8_t)r;
  }
  int e;
  double f = frexp(a, &e);  /* a = f * 2^e, f in [0.5, 1) */
  double r = nearbyint(f * 16.0); /* 8 + mantissa, in [8, 16] */
  int E = e + 6;                  /* biased exponent of 2^(e-1) */
  if (r == 16.0) {
    r = 8.0;
    E += 1;
  }
  if (E > 15 || (E == 15 && r - 8.0 > 6.0)) return sign | 0x7E;
  return sign | (uint8_t)((E << 3) | ((int)r - 8));
}

/* One row a[K] (bf16) -> codes q[K] and block scales s[ceil(K/128)] (fp32). */
void or_act_quant(const uint16_t* a, int K, uint8_t* q, float* s) {
  int kb = (K + 127) / 128;
  for (int b = 0; b < kb; ++b) {
    int k0 = b * 128, k1 = k0 + 128 < K ? k0 + 128 : K;
    float amax = 0.0f;
    for (int k = k0; k < k1; ++k) {
      float v = (float)fabs(bf(a[k]));
      if (v > amax) amax = v;
    }
    if (amax == 0.0f) {
      s[b] = 0.0f;
      for (int k = k0; k < k1; ++k) q[k] = 0;
      continue;
    }
    volatile float inv = 448.0f / amax; /* fp32 division, rounded */
    for (int k = k0; k < k1; ++k) {
      volatile float p = (float)bf(a[k]) * inv; /* fp32 product, rounded */
      q[k] = or_f32_to_e4m3_sat(p);
    }
    s[b] = amax / 448.0f;
  }
}

/* out[n] = sum over k blocks b of sa[b] * S[n/128][b] * sum_{k in b} E4M3(q[k]) * E4M3(W[n][k]). */
void or_w8a8_gemv(const uint8_t* q, const float* sa, const uint8_t* W, const uint16_t* S, int N, int K,
                  double* out) {
  int kb = (K + 127) / 128;
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int b = 0; b < kb; ++b) {
      int k0 = b * 128, k1 = k0 + 128 < K ? k0 + 128 : K;
      double part = 0.0;
      for (int k = k0; k < k1; ++k) part += e4m3(q[k]) * e4m3(W[(size_t)n * K + k]);
      acc += (double)sa[b] * bf(S[(size_t)(n / 128) * kb + b]) * part;
    }
    out[n] = acc;
  }
}

/* Sum of |terms| of the W8A8 product: sum_b |sa[b] * S[n/128][b]| * sum_{k in b} |E4M3(q[k]) * E4M3(W[n][k])|. */
void or_w8a8_abs(const uint8_t* q, const float* sa, const uint8_t* W, const uint16_t* S, int N, int K, double* out) {
  int kb = (K + 127) / 128;
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int b = 0; b < kb; ++b) {
      int k0 = b * 128, k1 = k0 + 128 < K ? k0 + 128 : K;
      double part = 0.0;
      for (int k = k0; k < k1; ++k) part += fabs(e4m3(q[k]) * e4m3(W[(size_t)n * K + k]));
      acc += fabs((double)sa[b] * bf(S[(size_t)(n / 128) * kb + b])) * part;
    }
    out[n] = acc;
  }
}

/* ---------------------------------------------------------------- layer */

typedef struct {
  int hidden, H, P, N, G, dconv, gnorm_group;
  double eps_in, eps_gated;
  const uint16_t* norm_w;   /* [hidden] */
  int in_fmt;               /* 1 = E4M3 + 128x128 bf16 block scales, 2 = bf16 */
  const void* in_w;         /* [n_in][hidden] */
  const uint16_t* in_s;     /* [ceil(n_in/128)][ceil(hidden/128)] */
  const uint16_t* conv_w;   /* [d_xbc][dconv] */
  const uint16_t* conv_b;   /* [d_xbc] */
  const float* A_log;       /* [H] */
  const float* D;           /* [H] */
  const float* dt_bias;     /* [H] */
  const uint16_t* gnorm_w;  /* [d_inner] */
  int out_fmt;
  const void* out_w;        /* [hidden][d_inner] */
  const uint16_t* out_s;    /* [ceil(hidden/128)][ceil(d_inner/128)] */
  int act_fp8;              /* 1: E4M3 projections use the W8A8 arm (FP8 activations) */
} or_layer;

static void proj(int fmt, int act_fp8, const void* w, const uint16_t* s, const uint16_t* a, int N, int K,
                 double* out) {
  if (fmt == 1 && act_fp8) {
    uint8_t* q = (uint8_t*)malloc((size_t)K);
    float* sa = (float*)malloc(sizeof(float) * (size_t)((K + 127) / 128));
    or_act_quant(a, K, q, sa);
    or_w8a8_gemv(q, sa, (const uint8_t*)w, s, N, K, out);
    free(q);
    free(sa);
  } else if (fmt == 1) {
    or_w8a16_gemv(a, 1, (const uint8_t*)w, s, N, K, out);
  } else {
    or_bf16_gemv(a, 1, (const uint16_t*)w, N, K, out);
  }
}

/* One token of one sequence through the whole layer, steps 1..8 in the order
 * of the [SRC] module header.  hidden [hidden] bf16 is modified in place
 * ([TRAIT] decode).  hs [H][P][N] double, ring [(dconv-1)][d_xbc] bf16 and
 * *pos are the sequence's state and are advanced by one token.  If tr_zx /
 * tr_u are non-NULL they receive the unrounded in_proj outputs [n_in] and conv
 * outputs [d_xbc] (the values rounded at R3 and R4), for tests that inspect
 * rounding decisions. */
long or_layer_token_traced(const or_layer* L, uint16_t* hidden, double* hs, uint16_t* ring, int32_t* pos,
                           double* tr_zx, double* tr_u, double* tr_zx_abs, double* tr_u_abs) {
  int d_inner = L->H * L->P;
  int d_xbc = d_inner + 2 * L->G * L->N;
  int n_in = d_inner + d_xbc + L->H;
  long hits = 0;
  uint16_t* xn = (uint16_t*)malloc(sizeof(uint16_t) * L->hidden);
  double* zx = (double*)malloc(sizeof(double) * n_in);
  uint16_t* zxb = (uint16_t*)malloc(sizeof(uint16_t) * n_in);
  uint16_t* u = (uint16_t*)malloc(sizeof(uint16_t) * d_xbc);
  double* y = (double*)malloc(sizeof(double) * d_inner);
  uint16_t* gout = (uint16_t*)malloc(sizeof(uint16_t) * d_inner);
  double* o = (double*)malloc(sizeof(double) * L->hidden);

  /* 1. RMSNorm (R2) */
  or_rmsnorm(hidden, L->norm_w, L->hidden, L->eps_in, xn);
  /* 2. in_proj -> [z, xBC, dt] (R3) */
  proj(L->in_fmt, L->act_fp8, L->in_w, L->in_s, xn, n_in, L->hidden, zx);
  for (int i = 0; i < n_in; ++i) zxb[i] = or_f64_to_bf16(zx[i]);
  if (tr_zx) memcpy(tr_zx, zx, sizeof(double) * n_in);
  if (tr_zx_abs) or_proj_abs(L->in_fmt, L->in_w, L->in_s, xn, n_in, L->hidden, tr_zx_abs);
  const uint16_t* z = zxb;
  const uint16_t* xbc = zxb + d_inner;
  const uint16_t* dt = zxb + d_inner + d_xbc;
  /* 3. conv1d update on xBC with bias and SiLU (R4) */
  or_conv1d_update_exact(ring, pos, xbc, L->conv_w, L->conv_b, d_xbc, L->dconv, 1, u, tr_u, tr_u_abs);
  *pos += 1;
  /* 4. split into x, B, C */
  const uint16_t* xs = u;
  const uint16_t* Bm = u + d_inner;
  const uint16_t* Cm = u + d_inner + L->G * L->N;
  /* 5. SSM state update and output */
  or_ssm_step(hs, xs, Bm, Cm, dt, L->A_log, L->D, L->dt_bias, L->H, L->P, L->N, L->G, y, &hits);
  /* 6. gated RMSNorm (R5) */
  or_gated_rmsnorm(y, z, L->gnorm_w, d_inner, L->gnorm_group, L->eps_gated, gout);
  /* 7. out_proj, 8. residual add, rounded once (R6) */
  proj(L->out_fmt, L->act_fp8, L->out_w, L->out_s, gout, L->hidden, d_inner, o);
  for (int i = 0; i < L->hidden; ++i) hidden[i] = or_f64_to_bf16(bf(hidden[i]) + o[i]);

  free(xn); free(zx); free(zxb); free(u); free(y); free(gout); free(o);
  return hits;
}

long or_layer_token(const or_layer* L, uint16_t* hidden, double* hs, uint16_t* ring, int32_t* pos) {
  return or_layer_token_traced(L, hidden, hs, ring, pos, NULL, NULL, NULL, NULL);
}

/* Prefill of T tokens of one sequence, by its definition: T sequential
 * single-token decode steps ([TRAIT] prefill default).  hidden is [T][hidden]. */
long or_layer_prefill(const or_layer* L, uint16_t* hidden, int T, double* hs, uint16_t* ring,
                      int32_t* pos) {
  long hits = 0;
  for (int t = 0; t < T; ++t)
    hits += or_layer_token(L, hidden + (size_t)t * L->hidden, hs, ring, pos);
  return hits;
}

/* The same, recording per token the unrounded in_proj and conv outputs
 * (tr_zx [T][n_in], tr_u [T][d_xbc]) and their sums of |terms|. */
long or_layer_prefill_traced(const or_layer* L, uint16_t* hidden, int T, double* hs, uint16_t* ring,
                             int32_t* pos, double* tr_zx, double* tr_u, double* tr_zx_abs, double* tr_u_abs) {
  int d_inner = L->H * L->P;
  int d_xbc = d_inner + 2 * L->G * L->N;
  int n_in = d_inner + d_xbc + L->H;
  long hits = 0;
  for (int t = 0; t < T; ++t)
    hits += or_layer_token_traced(L, hidden + (size_t)t * L->hidden, hs, ring, pos, tr_zx + (size_t)t * n_in,
                                  tr_u + (size_t)t * d_xbc, tr_zx_abs + (size_t)t * n_in,
                                  tr_u_abs + (size_t)t * d_xbc);
  return hits;
}

/* Vector form of or_f64_to_bf16. */
void or_f64_to_bf16_array(const double* v, uint16_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = or_f64_to_bf16(v[i]);
}

/* ------------------------------------------------------- rounding decisions */

/* Where a value lies within floating-point evaluation error of a bfloat16
 * rounding boundary, an fp32 evaluation and this double one may round to the
 * two neighbouring codes, and both are correct roundings of a correct value.
 * The functions below let the oracle follow another evaluation's decision at
 * the rounding points R3..R6 -- but only after checking it: the candidate code
 * is taken only if the exact value lies within tol * scale of the interval of
 * reals that round to that code, scale being the point's sum of |terms| (the
 * size of any evaluation's error).  Every other difference is refused (the
 * oracle keeps its own code) and counted.  The oracle still computes every
 * value itself. */

/* The interval [lo, hi] of reals that round (to nearest) to the finite bf16
 * code c; returns 0 for NaN and infinity codes. */
int or_bf16_round_interval(uint16_t c, double* lo, double* hi) {
  uint16_t mag = c & 0x7FFF;
  if (mag >= 0x7F80) return 0;
  double v = bf(mag);
  double below = mag == 0 ? -bf(1) : bf((uint16_t)(mag - 1));
  double above = mag == 0x7F7F ? ldexp(1.0, 128) : bf((uint16_t)(mag + 1));
  double a = 0.5 * (below + v), b = 0.5 * (v + above);
  if (c & 0x8000) {
    *lo = -b;
    *hi = -a;
  } else {
    *lo = a;
    *hi = b;
  }
  return 1;
}

/* Distance of `exact` from the rounding interval of code c, over `scale`
 * (0 inside the interval; infinite for a NaN or infinity code or a zero
 * scale with a nonzero distance). */
double or_decision_excess(uint16_t c, double exact, double scale) {
  double lo, hi;
  if (!or_bf16_round_interval(c, &lo, &hi)) return INFINITY;
  double dist = exact < lo ? lo - exact : (exact > hi ? exact - hi : 0.0);
  if (dist == 0.0) return 0.0;
  return scale > 0.0 ? dist / scale : INFINITY;
}

typedef struct {
  const uint16_t* cand[4]; /* candidate codes at R3 [n_in], R4 [d_xbc], R5 [d_inner], R6 [hidden]; NULL: none */
  long ld[4];              /* row stride of each candidate array (prefill: next token) */
  double tol[4];           /* relative tolerance of each point */
  long taken[4];           /* candidates that differed from the oracle's code and were legitimate */
  long refused[4];         /* candidates that differed and were not */
  double worst_taken[4];   /* largest excess among taken candidates */
  double worst_refused[4]; /* largest excess among refused ones */
  long first_refused[4];   /* token * row + index of the first refused candidate, -1 if none */
  /* W8A8 arm: the out_proj's E4M3 input codes [d_inner] and block scales
   * [d_inner/128] ("Q5"), rows q5_ld / q5_lds apart; judged per 128-block */
  const uint8_t* q5_codes;
  const float* q5_scales;
  long q5_ld, q5_lds;
  long q5_taken, q5_refused, q5_first_refused;
  uint16_t* r5_trace; /* if not NULL: the decided R5 codes of each token [T][d_inner] */
  double* q5_diag;    /* if not NULL: the first refused Q5 block, [4][128] + 2: exact R5 values,
                         their scales, own codes, candidate codes, candidate scale, own scale */
} or_decisions;

/* One rounding point: codes[i] = the candidate where it is legitimate, else
 * the oracle's own rounding of exact[i]. */
static void decide(or_decisions* dec, int pt, long token, const double* exact, const double* scale, int n,
                   uint16_t* codes) {
  const uint16_t* cand = dec && dec->cand[pt] ? dec->cand[pt] + token * dec->ld[pt] : NULL;
  for (int i = 0; i < n; ++i) {
    uint16_t own = or_f64_to_bf16(exact[i]);
    codes[i] = own;
    if (!cand || cand[i] == own) continue;
    double ex = or_decision_excess(cand[i], exact[i], scale[i] > fabs(exact[i]) ? scale[i] : fabs(exact[i]));
    if (ex <= dec->tol[pt]) {
      codes[i] = cand[i];
      dec->taken[pt]++;
      if (ex > dec->worst_taken[pt]) dec->worst_taken[pt] = ex;
    } else {
      dec->refused[pt]++;
      if (ex > dec->worst_refused[pt]) dec->worst_refused[pt] = ex;
      if (dec->first_refused[pt] < 0) dec->first_refused[pt] = token * (long)n + i;
    }
  }
}

/* bf16 codes as ordered integers (value order) and back; finite codes only. */
static int code_ord(uint16_t c) { return (c & 0x8000) ? -(int)(c & 0x7FFF) : (int)(c & 0x7FFF); }
static uint16_t ord_code(int o) { return o < 0 ? (uint16_t)(0x8000 | (-o)) : (uint16_t)o; }
/* E4M3 codes as ordered integers. */
static int e4m3_ord(uint8_t q) { return (q & 0x80) ? -(int)(q & 0x7F) : (int)(q & 0x7F); }

/* The range [*lo, *hi] (ordered bf16 codes) of the codes decide() would take
 * for an exact value with this scale: the own code c and every code next to
 * the range whose excess is <= tol. */
static void legit_code_range(uint16_t c, double exact, double scale, double tol, int* lo, int* hi) {
  double sc = scale > fabs(exact) ? scale : fabs(exact);
  int o = code_ord(c), l = o, h = o;
  for (int it = 0; it < 65536 && l - 1 >= -0x7F7F && or_decision_excess(ord_code(l - 1), exact, sc) <= tol; ++it) --l;
  for (int it = 0; it < 65536 && h + 1 <= 0x7F7F && or_decision_excess(ord_code(h + 1), exact, sc) <= tol; ++it) ++h;
  *lo = l;
  *hi = h;
}

/* Whether an E4M3 block (codes gq[n], scale gs) is what the W8A8 activation
 * quantization makes of some choice of bf16 inputs, each element a code that
 * decide() would take at R5 (the oracle's own code c[i], or any code whose
 * excess is <= tol: a contiguous range of codes).  The quantization is the
 * oracle's own (or_act_quant): amax over the block, scale amax / 448 and codes
 * E4M3(v * (448 / amax)) in fp32, which is monotonic in v; so for a given amax
 * each element reaches a contiguous range of E4M3 codes. */
static int q5_block_legit(const double* exact, const double* scale, const uint16_t* c, int n, const uint8_t* gq,
                          float gs, double tol) {
  int lo[128], hi[128];
  for (int i = 0; i < n; ++i) legit_code_range(c[i], exact[i], scale[i], tol, &lo[i], &hi[i]);
  if (gs == 0.0f) {  /* an all-zero block: every element must be able to be zero */
    for (int i = 0; i < n; ++i)
      if (lo[i] > 0 || hi[i] < 0 || gq[i] != 0) return 0;
    return 1;
  }
  /* amax candidates: the bf16 magnitudes m with m / 448 == gs in fp32 */
  uint16_t m0 = or_f64_to_bf16((double)gs * 448.0);
  for (int dm = -3; dm <= 3; ++dm) {
    int om = code_ord(m0) + dm;
    if (om <= 0 || om > 0x7F7F) continue;
    float m = (float)bf(ord_code(om));
    if (m / 448.0f != gs) continue;
    volatile float inv = 448.0f / m;
    int ok = 1, attained = 0;
    for (int i = 0; i < n && ok; ++i) {
      /* the element's values within [-m, m] */
      int l = lo[i] > -om ? lo[i] : -om, h = hi[i] < om ? hi[i] : om;
      if (l > h) {
        ok = 0;
        break;
      }
      volatile float vl = (float)bf(ord_code(l)) * inv, vh = (float)bf(ord_code(h)) * inv;
      int ql = e4m3_ord(or_f32_to_e4m3_sat(vl)), qh = e4m3_ord(or_f32_to_e4m3_sat(vh)), g = e4m3_ord(gq[i]);
      if (g < ql || g > qh) ok = 0;
      /* an element that can be +-m and whose code is the one +-m gives */
      if ((h == om && g == qh) || (l == -om && g == ql)) attained = 1;
    }
    if (ok && attained) return 1;
  }
  return 0;
}

/* The layer's token (steps 1..8 as or_layer_token_traced) with the decisions
 * at R3..R6 judged against `dec`; token is the row index into the candidates. */
static long layer_token_decided(const or_layer* L, uint16_t* hidden, double* hs, uint16_t* ring, int32_t* pos,
                                or_decisions* dec, long token) {
  int d_inner = L->H * L->P;
  int d_xbc = d_inner + 2 * L->G * L->N;
  int n_in = d_inner + d_xbc + L->H;
  int kmax = L->hidden > d_inner ? L->hidden : d_inner;
  long hits = 0;
  uint16_t* xn = (uint16_t*)malloc(sizeof(uint16_t) * L->hidden);
  double* zx = (double*)malloc(sizeof(double) * n_in);
  double* zxa = (double*)malloc(sizeof(double) * n_in);
  uint16_t* zxb = (uint16_t*)malloc(sizeof(uint16_t) * n_in);
  uint16_t* u = (uint16_t*)malloc(sizeof(uint16_t) * d_xbc);
  double* ue = (double*)malloc(sizeof(double) * d_xbc);
  double* ua = (double*)malloc(sizeof(double) * d_xbc);
  double* y = (double*)malloc(sizeof(double) * d_inner);
  double* ya = (double*)malloc(sizeof(double) * d_inner);
  double* ge = (double*)malloc(sizeof(double) * d_inner);
  double* ga = (double*)malloc(sizeof(double) * d_inner);
  uint16_t* gout = (uint16_t*)malloc(sizeof(uint16_t) * d_inner);
  double* o = (double*)malloc(sizeof(double) * L->hidden);
  double* oa = (double*)malloc(sizeof(double) * L->hidden);
  uint8_t* q = (uint8_t*)malloc((size_t)kmax);
  float* sa = (float*)malloc(sizeof(float) * (size_t)((kmax + 127) / 128));

  /* 1. RMSNorm (R2) */
  or_rmsnorm(hidden, L->norm_w, L->hidden, L->eps_in, xn);
  /* 2. in_proj -> [z, xBC, dt] (R3) */
  if (L->in_fmt == 1 && L->act_fp8) {
    or_act_quant(xn, L->hidden, q, sa);
    or_w8a8_gemv(q, sa, (const uint8_t*)L->in_w, L->in_s, n_in, L->hidden, zx);
    or_w8a8_abs(q, sa, (const uint8_t*)L->in_w, L->in_s, n_in, L->hidden, zxa);
  } else {
    proj(L->in_fmt, 0, L->in_w, L->in_s, xn, n_in, L->hidden, zx);
    or_proj_abs(L->in_fmt, L->in_w, L->in_s, xn, n_in, L->hidden, zxa);
  }
  decide(dec, 0, token, zx, zxa, n_in, zxb);
  /* 3. conv1d update with bias and SiLU (R4) */
  or_conv1d_update_exact(ring, pos, zxb + d_inner, L->conv_w, L->conv_b, d_xbc, L->dconv, 1, u, ue, ua);
  for (int c = 0; c < d_xbc; ++c) ua[c] *= 1.1; /* |silu'| <= 1.1: the pre-activation's error, carried through */
  decide(dec, 1, token, ue, ua, d_xbc, u);
  *pos += 1;
  /* 4, 5. split, SSM step */
  ssm_step_impl(hs, u, u + d_inner, u + d_inner + L->G * L->N, zxb + d_inner + d_xbc, L->A_log, L->D, L->dt_bias,
                L->H, L->P, L->N, L->G, y, ya, &hits);
  /* 6. gated RMSNorm (R5) */
  gated_rmsnorm_exact(y, ya, zxb, L->gnorm_w, d_inner, L->gnorm_group, L->eps_gated, ge, ga);
  decide(dec, 2, token, ge, ga, d_inner, gout);
  if (dec && dec->r5_trace) memcpy(dec->r5_trace + token * (long)d_inner, gout, sizeof(uint16_t) * d_inner);
  /* 7, 8. out_proj and residual (R6) */
  if (L->out_fmt == 1 && L->act_fp8) {
    or_act_quant(gout, d_inner, q, sa);
    if (dec && dec->q5_codes) {
      /* the quantized input, block by block, as the candidate has it where
       * that is what legitimate R5 decisions would give */
      const uint8_t* gq = dec->q5_codes + token * dec->q5_ld;
      const float* gs = dec->q5_scales + token * dec->q5_lds;
      for (int b = 0; b * 128 < d_inner; ++b) {
        int k0 = b * 128, n = d_inner - k0 < 128 ? d_inner - k0 : 128;
        if (!memcmp(gq + k0, q + k0, (size_t)n) && gs[b] == sa[b]) continue;
        if (q5_block_legit(ge + k0, ga + k0, gout + k0, n, gq + k0, gs[b], dec->tol[2])) {
          memcpy(q + k0, gq + k0, (size_t)n);
          sa[b] = gs[b];
          dec->q5_taken++;
        } else {
          dec->q5_refused++;
          if (dec->q5_first_refused < 0) {
            dec->q5_first_refused = token * (long)d_inner + k0;
            if (dec->q5_diag) {
              for (int i = 0; i < n; ++i) {
                dec->q5_diag[i] = ge[k0 + i];
                dec->q5_diag[128 + i] = ga[k0 + i];
                dec->q5_diag[256 + i] = gout[k0 + i];
                dec->q5_diag[384 + i] = gq[k0 + i];
              }
              dec->q5_diag[512] = gs[b];
              dec->q5_diag[513] = sa[b];
            }
          }
        }
      }
    }
    or_w8a8_gemv(q, sa, (const uint8_t*)L->out_w, L->out_s, L->hidden, d_inner, o);
    or_w8a8_abs(q, sa, (const uint8_t*)L->out_w, L->out_s, L->hidden, d_inner, oa);
  } else {
    proj(L->out_fmt, 0, L->out_w, L->out_s, gout, L->hidden, d_inner, o);
    or_proj_abs(L->out_fmt, L->out_w, L->out_s, gout, L->hidden, d_inner, oa);
  }
  for (int i = 0; i < L->hidden; ++i) {
    o[i] += bf(hidden[i]);
    oa[i] += fabs(bf(hidden[i]));
  }
  decide(dec, 3, token, o, oa, L->hidden, hidden);

  free(xn); free(zx); free(zxa); free(zxb); free(u); free(ue); free(ua); free(y); free(ya); free(ge); free(ga);
  free(gout); free(o); free(oa); free(q); free(sa);
  return hits;
}

/* T tokens of one sequence (hidden [T][hidden], in place), each decision
 * judged against the candidates of its token row. */
long or_layer_prefill_decided(const or_layer* L, uint16_t* hidden, int T, double* hs, uint16_t* ring, int32_t* pos,
                              or_decisions* dec) {
  long hits = 0;
  for (int t = 0; t < T; ++t)
    hits += layer_token_decided(L, hidden + (size_t)t * L->hidden, hs, ring, pos, dec, t);
  return hits;
}

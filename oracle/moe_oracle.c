/*
 * moe_oracle.c -- plain, slow fp64 CPU reference of the fused MoE expert
 * computation.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library; the product path never
 * does.  It shares no code, header, table or constant generator with the CUDA
 * library: every codec, rule and formula below is written out here on its own.
 *
 * What it computes, and where each part comes from (page title, then the
 * class / function / passage on that page):
 *
 *  - Element codecs.  "vllm.model_executor.layers.quantization.quark.quark_moe",
 *    QuarkNvfp4MoEMethod.create_weights (two e2m1 values packed per uint8,
 *    e4m3 group scales, fp32 global scales) and
 *    "vLLM/vllm/model_executor/layers/quantization/mxfp4.py",
 *    GptOssMxfp4MoEMethod.create_weights (packed e2m1 codes, uint8 e8m0 scales
 *    per 32 elements of the reduction dimension).  The code->value tables are
 *    the OCP microscaling element formats: e2m1 (bias 1), e4m3fn (bias 7, no
 *    infinity, S.1111.111 = NaN, max 448) and e8m0 (2^(c-127), 255 = NaN).
 *  - Routing (softmax -> top-k -> renormalise): the router that produces
 *    topk_ids / topk_weights for "rocm_aiter_fused_experts".
 *  - Expert sort and block padding: the dispatch step named by
 *    moe_sorting_dispatch_policy in AiterExperts.apply.  The pages do not give
 *    the rule; the one used here is: per local expert (ascending id) the flat
 *    slot ids t*T+k in ascending order, padded with the sentinel S = M*T to a
 *    multiple of the block size; empty experts get no block.
 *  - Activation quantisers (per-tensor static/dynamic, per-token, 1x128 group
 *    fp8; NVFP4 x16 with an fp32 global): AiterFp8TensorExperts,
 *    AiterFp8ChannelExperts, AiterFp8BlockExperts and QuarkNvfp4MoEMethod.
 *  - The fused experts (route -> gate/up GEMM -> activation -> down GEMM ->
 *    top-k weighted reduce): "rocm_aiter_fused_experts" and AiterExperts.apply
 *    (output (M, K) written into a caller-owned buffer), the activation set of
 *    _resolve_aiter_activation, the gate/up layouts of the gate-mode selection
 *    (SEPARATED = [gate_all; up_all], INTERLEAVE = row 2j gate, 2j+1 up) and
 *    the SwiGLU constants of GptOssMxfp4MoEMethod.get_fused_moe_quant_config
 *    (alpha 1.702, beta 1.0, limit 7.0).
 *
 * Precision: every sum, product and activation is evaluated in fp64.  Where a
 * floating-point value decides an integer code, the decision is taken on the
 * fp32 value the quantiser spec names (fl32(x / scale)); an fp64 divide of two
 * fp32 values rounded once to fp32 equals the correctly rounded fp32 divide.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- enumerations (this file's own numbering; the Python wrapper maps names) */
enum { ORC_W_BF16 = 0, ORC_W_FP8_TENSOR = 1, ORC_W_FP8_CHANNEL = 2,
       ORC_W_FP8_BLOCK128 = 3, ORC_W_MXFP4 = 4, ORC_W_NVFP4 = 5 };
enum { ORC_A_BF16 = 0, ORC_A_FP8_TENSOR_STATIC = 1, ORC_A_FP8_TENSOR_DYN = 2,
       ORC_A_FP8_TOKEN_DYN = 3, ORC_A_FP8_GROUP128_DYN = 4, ORC_A_NVFP4_DYN = 5,
       ORC_A_MXFP4_DYN = 6, ORC_A_MXFP8_DYN = 7 };
enum { ORC_ACT_SILU = 0, ORC_ACT_GELU = 1, ORC_ACT_SWIGLU_OAI = 2 };
enum { ORC_GATE_SEPARATED = 0, ORC_GATE_INTERLEAVED = 1 };

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ============================== codecs ================================== */

/* e2m1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa. */
double orc_e2m1_decode(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double v = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
  return s ? -v : v;
}

/* e4m3fn: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa;
 * exponent 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN; no infinity. */
double orc_e4m3_decode(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = m * ldexp(1.0, -9);
  else v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
  return s ? -v : v;
}

/* e8m0: an unsigned biased exponent, value 2^(c-127); 255 is NaN. */
double orc_e8m0_decode(int code) {
  code &= 255;
  return code == 255 ? NAN : ldexp(1.0, code - 127);
}

/* Nearest entry of an ascending table of non-negative magnitudes, ties to the
 * even code (for these formats the even code is the one with an even
 * mantissa).  Magnitudes above the last entry saturate to it. */
static int nearest_code(double a, const double *table, int n) {
  int best = 0;
  double bd = fabs(a - table[0]);
  for (int c = 1; c < n; ++c) {
    double d = fabs(a - table[c]);
    if (d < bd || (d == bd && (c % 2) == 0)) { best = c; bd = d; }
  }
  return best;
}

static double g_e4m3_mag[127];
static double g_e2m1_mag[8];
static int g_tables_ready = 0;
static void init_tables(void) {
  if (g_tables_ready) return;
  for (int c = 0; c < 127; ++c) g_e4m3_mag[c] = orc_e4m3_decode(c);
  for (int c = 0; c < 8; ++c) g_e2m1_mag[c] = orc_e2m1_decode(c);
  g_tables_ready = 1;
}

/* Round-to-nearest-even, saturating at +-448; the sign is kept (so -0 gives
 * 0x80).  `v` is an fp32 value (passed widened). */
int orc_e4m3_encode(double v) {
  init_tables();
  int sign = signbit(v) ? 0x80 : 0;
  return sign | nearest_code(fabs(v), g_e4m3_mag, 127);
}

/* Round-to-nearest-even, saturating at +-6; the sign is kept (-0 gives 0x8). */
int orc_e2m1_encode(double v) {
  init_tables();
  int sign = signbit(v) ? 0x8 : 0;
  return sign | nearest_code(fabs(v), g_e2m1_mag, 8);
}

/* bf16 bits <-> value; round-to-nearest-even straight from fp64. */
double orc_bf16_decode(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

double orc_round_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e;
  frexp(v, &e); /* v = f * 2^e with 0.5 <= |f| < 1 */
  int ulp_exp = e - 8;            /* 8 significant bits for normals */
  if (e - 1 < -126) ulp_exp = -133; /* subnormal spacing 2^-133 */
  double q = ldexp(v, -ulp_exp);
  return ldexp(nearbyint(q), ulp_exp);
}

uint16_t orc_bf16_encode(double v) {
  float f = (float)orc_round_bf16(v); /* exact: the value is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

static double fl32(double v) { return (double)(float)v; }

/* ============================== routing ================================= */
/* softmax over E logits, top-k (largest first, ties to the lower expert id),
 * optional renormalisation of the selected probabilities to sum to one. */
void orc_route_topk(const double *logits, int M, int E, int k, int renorm,
                    int32_t *ids, double *weights) {
  double *p = (double *)malloc(sizeof(double) * E);
  char *taken = (char *)malloc(E);
  for (int t = 0; t < M; ++t) {
    const double *l = logits + (size_t)t * E;
    double mx = l[0];
    for (int e = 1; e < E; ++e) if (l[e] > mx) mx = l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - mx); z += p[e]; }
    for (int e = 0; e < E; ++e) p[e] /= z;
    memset(taken, 0, E);
    double sel = 0.0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || p[e] > p[best])) best = e;
      taken[best] = 1;
      ids[(size_t)t * k + j] = best;
      weights[(size_t)t * k + j] = p[best];
      sel += p[best];
    }
    if (renorm)
      for (int j = 0; j < k; ++j) weights[(size_t)t * k + j] /= sel;
  }
  free(p);
  free(taken);
}

/* Router of the apply_monolithic path (router logits, num_expert_group,
 * topk_group, e_score_correction_bias, routed_scaling_factor), read as:
 *   s_e   = softmax(l)_e (scoring 0) or 1 / (1 + exp(-l_e)) (scoring 1)
 *   key_e = s_e + bias_e with a bias, else l_e (the same order as s_e)
 *   G > 1: group g (experts g*E/G .. (g+1)*E/G - 1) scores the sum of its two
 *          largest keys (bias) or its largest key (no bias); the TG best
 *          groups, ties to the lower group, stay eligible
 *   ids   = the k eligible experts with the largest keys, descending, ties to
 *           the lower id
 *   w_j   = s_{id_j}, divided by their sum when renorm, times scale. */
void orc_route_grouped(const double *logits, int M, int E, int k, int scoring, int renorm, int G,
                       int TG, const double *bias, double scale, int32_t *ids, double *weights) {
  double *sc = (double *)malloc(sizeof(double) * E);
  double *key = (double *)malloc(sizeof(double) * E);
  char *ok = (char *)malloc(E);
  double *gscore = (double *)malloc(sizeof(double) * (G > 1 ? G : 1));
  char *gkeep = (char *)malloc(G > 1 ? G : 1);
  for (int t = 0; t < M; ++t) {
    const double *l = logits + (size_t)t * E;
    if (scoring == 0) {
      double mx = l[0];
      for (int e = 1; e < E; ++e) if (l[e] > mx) mx = l[e];
      double z = 0.0;
      for (int e = 0; e < E; ++e) { sc[e] = exp(l[e] - mx); z += sc[e]; }
      for (int e = 0; e < E; ++e) sc[e] /= z;
    } else {
      for (int e = 0; e < E; ++e) sc[e] = 1.0 / (1.0 + exp(-l[e]));
    }
    for (int e = 0; e < E; ++e) {
      key[e] = bias ? sc[e] + bias[e] : l[e];
      ok[e] = 1;
    }
    if (G > 1) {
      const int gs = E / G;
      for (int g = 0; g < G; ++g) {
        double b1 = -INFINITY, b2 = -INFINITY;
        for (int e = g * gs; e < (g + 1) * gs; ++e) {
          if (key[e] > b1) { b2 = b1; b1 = key[e]; }
          else if (key[e] > b2) b2 = key[e];
        }
        gscore[g] = bias ? b1 + b2 : b1;
        gkeep[g] = 0;
      }
      for (int j = 0; j < TG; ++j) {
        int best = -1;
        for (int g = 0; g < G; ++g)
          if (!gkeep[g] && (best < 0 || gscore[g] > gscore[best])) best = g;
        gkeep[best] = 1;
      }
      for (int e = 0; e < E; ++e) ok[e] = gkeep[e / gs];
    }
    double sel = 0.0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (ok[e] && (best < 0 || key[e] > key[best])) best = e;
      ok[best] = 0;
      ids[(size_t)t * k + j] = best;
      weights[(size_t)t * k + j] = sc[best];
      sel += sc[best];
    }
    for (int j = 0; j < k; ++j) {
      double w = weights[(size_t)t * k + j];
      if (renorm) w /= sel;
      weights[(size_t)t * k + j] = w * scale;
    }
  }
  free(sc);
  free(key);
  free(ok);
  free(gscore);
  free(gkeep);
}

/* ========================= expert sort / padding ======================== */

static int local_expert(int32_t g, const int32_t *emap, int E, int El) {
  if (g < 0 || g >= E) return -1;
  int l = emap ? emap[g] : g;
  return (l >= 0 && l < El) ? l : -1;
}

/* Capacity of the sorted-id buffer: every live slot plus at most BM-1 pad
 * entries for each expert that has at least one slot, rounded up to a whole
 * number of blocks. */
long orc_align_capacity(int M, int T, int El, int BM) {
  long S = (long)M * T;
  long nonempty = S < El ? S : El;
  long cap = S + nonempty * (BM - 1);
  return ((cap + BM - 1) / BM) * BM;
}

/* Returns 0 on success.  sorted_ids has orc_align_capacity() entries,
 * expert_ids has capacity/BM entries, counts has El entries. */
int orc_align_block_size(const int32_t *ids, int M, int T, const int32_t *emap,
                         int E, int El, int BM, int32_t *sorted_ids,
                         int32_t *expert_ids, int32_t *num_post_pad,
                         int32_t *counts) {
  long S = (long)M * T;
  long cap = orc_align_capacity(M, T, El, BM);
  for (int e = 0; e < El; ++e) counts[e] = 0;
  for (long s = 0; s < S; ++s) {
    int l = local_expert(ids[s], emap, E, El);
    if (l >= 0) counts[l]++;
  }
  long off = 0;
  for (int e = 0; e < El; ++e) {
    if (counts[e] == 0) continue;
    long start = off, n = 0;
    for (long s = 0; s < S; ++s)
      if (local_expert(ids[s], emap, E, El) == e) sorted_ids[start + n++] = (int32_t)s;
    long padded = ((n + BM - 1) / BM) * BM;
    for (long i = n; i < padded; ++i) sorted_ids[start + i] = (int32_t)S;
    for (long b = start / BM; b < (start + padded) / BM; ++b) expert_ids[b] = e;
    off += padded;
  }
  *num_post_pad = (int32_t)off;
  for (long i = off; i < cap; ++i) sorted_ids[i] = (int32_t)S;
  for (long b = off / BM; b < cap / BM; ++b) expert_ids[b] = -1;
  return 0;
}

/* ========================== activation quantisers ======================= */

#define ORC_FP8_MAX 448.0
#define ORC_E2M1_MAX 6.0

/* fp8 scale of a group with absolute maximum `amax` (an fp32 value):
 * fl32(max(amax, fl32(1e-12)) / 448). */
static double fp8_dyn_scale(double amax) {
  double floor_ = fl32(1e-12);
  return fl32((amax > floor_ ? amax : floor_) / ORC_FP8_MAX);
}

/* Quantise `n` fp32 values with one fp8 scale; writes codes, returns nothing. */
static void fp8_encode_group(const float *x, long n, double scale, uint8_t *codes) {
  for (long i = 0; i < n; ++i) codes[i] = (uint8_t)orc_e4m3_encode(fl32((double)x[i] / scale));
}

/* NVFP4 group of 16 with fp32 global g: the e4m3 scale code is
 * e4m3(fl32(fl32(amax/6)/g)); element codes are e2m1(fl32(x / fl32(s*g)));
 * a zero scale gives zero codes.  Codes are written one per byte here. */
static int nvfp4_encode_group(const float *x, double g, uint8_t *codes16) {
  double amax = 0.0;
  for (int i = 0; i < 16; ++i) { double a = fabs((double)x[i]); if (a > amax) amax = a; }
  int s = orc_e4m3_encode(fl32(fl32(amax / ORC_E2M1_MAX) / g));
  double sv = orc_e4m3_decode(s);
  if (sv == 0.0) { for (int i = 0; i < 16; ++i) codes16[i] = 0; return s; }
  double denom = fl32(sv * g);
  for (int i = 0; i < 16; ++i) codes16[i] = (uint8_t)orc_e2m1_encode(fl32((double)x[i] / denom));
  return s;
}

/* OCP MX block of 32 fp32 values (MXFP4: e2m1 elements, emax 2; MXFP8: e4m3
 * elements, emax 8), the conversion of the OCP Microscaling Formats (MX) v1.0
 * specification: shared exponent X = floor(log2(amax)) - emax, clamped to the
 * e8m0 range [-127, 127]; scale code X + 127; element code = RNE with
 * saturation of x / 2^X (an exact power-of-two division).  amax == 0 gives
 * scale code 0 and zero codes.  Element codes one per byte. */
static int mx_encode_group(const float *x, int elem_fp4, uint8_t *codes32) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) { double a = fabs((double)x[i]); if (a > amax) amax = a; }
  if (amax == 0.0) { for (int i = 0; i < 32; ++i) codes32[i] = 0; return 0; }
  int ex;
  frexp(amax, &ex);                 /* amax = f * 2^ex, 0.5 <= f < 1 */
  int X = (ex - 1) - (elem_fp4 ? 2 : 8);
  if (X < -127) X = -127;
  if (X > 127) X = 127;
  for (int i = 0; i < 32; ++i) {
    double v = ldexp((double)x[i], -X);
    codes32[i] = (uint8_t)(elem_fp4 ? orc_e2m1_encode(v) : orc_e4m3_encode(v));
  }
  return X + 127;
}

/* Quantise fp32 rows.  Layouts (row-major):
 *   fp8 codes  u8 [rows, cols];  NVFP4 codes u8 [rows, cols/2] (even column in
 *   the low nibble);
 *   scales: tensor f32[1]; token f32[rows]; group128 f32[rows, ceil(cols/128)];
 *   NVFP4 e4m3 u8 [rows, cols/16].
 * `param`: the static fp8 scale (tensor static) or, for NVFP4, the global of
 * each row (`per_row_param` != 0) or one global for all rows. */
static int quant_rows(const float *x, long rows, long cols, int afmt,
                      const float *param, int per_row_param, uint8_t *codes,
                      void *scales) {
  if (afmt == ORC_A_FP8_TENSOR_STATIC || afmt == ORC_A_FP8_TENSOR_DYN) {
    double scale;
    if (afmt == ORC_A_FP8_TENSOR_STATIC) scale = (double)param[0];
    else {
      double amax = 0.0;
      for (long i = 0; i < rows * cols; ++i) { double a = fabs((double)x[i]); if (a > amax) amax = a; }
      scale = fp8_dyn_scale(amax);
    }
    ((float *)scales)[0] = (float)scale;
    fp8_encode_group(x, rows * cols, scale, codes);
    return 0;
  }
  if (afmt == ORC_A_FP8_TOKEN_DYN) {
    for (long r = 0; r < rows; ++r) {
      double amax = 0.0;
      for (long c = 0; c < cols; ++c) { double a = fabs((double)x[r * cols + c]); if (a > amax) amax = a; }
      double scale = fp8_dyn_scale(amax);
      ((float *)scales)[r] = (float)scale;
      fp8_encode_group(x + r * cols, cols, scale, codes + r * cols);
    }
    return 0;
  }
  if (afmt == ORC_A_FP8_GROUP128_DYN) {
    long G = (cols + 127) / 128;
    for (long r = 0; r < rows; ++r)
      for (long g = 0; g < G; ++g) {
        long c0 = g * 128, n = (cols - c0) < 128 ? (cols - c0) : 128;
        double amax = 0.0;
        for (long c = 0; c < n; ++c) { double a = fabs((double)x[r * cols + c0 + c]); if (a > amax) amax = a; }
        double scale = fp8_dyn_scale(amax);
        ((float *)scales)[r * G + g] = (float)scale;
        fp8_encode_group(x + r * cols + c0, n, scale, codes + r * cols + c0);
      }
    return 0;
  }
  if (afmt == ORC_A_MXFP4_DYN || afmt == ORC_A_MXFP8_DYN) {
    if (cols % 32) return -1;
    const int fp4 = afmt == ORC_A_MXFP4_DYN;
    long G = cols / 32;
    uint8_t q[32];
    for (long r = 0; r < rows; ++r)
      for (long gi = 0; gi < G; ++gi) {
        int sc = mx_encode_group(x + r * cols + gi * 32, fp4, q);
        ((uint8_t *)scales)[r * G + gi] = (uint8_t)sc;
        if (fp4) {
          for (int i = 0; i < 16; ++i)
            codes[r * (cols / 2) + gi * 16 + i] = (uint8_t)(q[2 * i] | (q[2 * i + 1] << 4));
        } else {
          memcpy(codes + r * cols + gi * 32, q, 32);
        }
      }
    return 0;
  }
  if (afmt == ORC_A_NVFP4_DYN) {
    if (cols % 16) return -1;
    long G = cols / 16;
    uint8_t q[16];
    for (long r = 0; r < rows; ++r) {
      double g = (double)(per_row_param ? param[r] : param[0]);
      for (long gi = 0; gi < G; ++gi) {
        int s = nvfp4_encode_group(x + r * cols + gi * 16, g, q);
        ((uint8_t *)scales)[r * G + gi] = (uint8_t)s;
        for (int i = 0; i < 8; ++i)
          codes[r * (cols / 2) + gi * 8 + i] = (uint8_t)(q[2 * i] | (q[2 * i + 1] << 4));
      }
    }
    return 0;
  }
  return -1;
}

/* Dequantise the rows produced by quant_rows back to fp64. */
static void dequant_rows(const uint8_t *codes, const void *scales, long rows,
                         long cols, int afmt, const float *param,
                         int per_row_param, double *out) {
  for (long r = 0; r < rows; ++r)
    for (long c = 0; c < cols; ++c) {
      double v;
      switch (afmt) {
        case ORC_A_FP8_TENSOR_STATIC:
        case ORC_A_FP8_TENSOR_DYN:
          v = orc_e4m3_decode(codes[r * cols + c]) * ((const float *)scales)[0];
          break;
        case ORC_A_FP8_TOKEN_DYN:
          v = orc_e4m3_decode(codes[r * cols + c]) * ((const float *)scales)[r];
          break;
        case ORC_A_FP8_GROUP128_DYN: {
          long G = (cols + 127) / 128;
          v = orc_e4m3_decode(codes[r * cols + c]) * ((const float *)scales)[r * G + c / 128];
          break;
        }
        case ORC_A_NVFP4_DYN: {
          uint8_t b = codes[r * (cols / 2) + c / 2];
          int q = (c & 1) ? (b >> 4) : (b & 15);
          double g = (double)(per_row_param ? param[r] : param[0]);
          v = orc_e2m1_decode(q) * orc_e4m3_decode(((const uint8_t *)scales)[r * (cols / 16) + c / 16]) * g;
          break;
        }
        case ORC_A_MXFP4_DYN: {
          uint8_t b = codes[r * (cols / 2) + c / 2];
          int q = (c & 1) ? (b >> 4) : (b & 15);
          v = orc_e2m1_decode(q) * orc_e8m0_decode(((const uint8_t *)scales)[r * (cols / 32) + c / 32]);
          break;
        }
        case ORC_A_MXFP8_DYN:
          v = orc_e4m3_decode(codes[r * cols + c]) *
              orc_e8m0_decode(((const uint8_t *)scales)[r * (cols / 32) + c / 32]);
          break;
        default: v = NAN;
      }
      out[r * cols + c] = v;
    }
}

/* Public stage-1 quantiser on bf16 input (one global / static scale). */
int orc_quant_act(const uint16_t *x_bf16, long rows, long cols, int afmt,
                  const float *scale_in, uint8_t *codes, void *scales) {
  float *xf = (float *)malloc(sizeof(float) * rows * cols);
  for (long i = 0; i < rows * cols; ++i) xf[i] = (float)orc_bf16_decode(x_bf16[i]);
  int rc = quant_rows(xf, rows, cols, afmt, scale_in, 0, codes, scales);
  free(xf);
  return rc;
}

/* Public quantise-dequantise of fp32 rows, with per-row NVFP4 globals when
 * per_row_param is set (used for the stage-2 intermediate). */
int orc_qdq_rows(const float *x, long rows, long cols, int afmt,
                 const float *param, int per_row_param, double *out) {
  long ncodes = (afmt == ORC_A_NVFP4_DYN || afmt == ORC_A_MXFP4_DYN) ? rows * cols / 2 : rows * cols;
  long nscales = rows * ((cols + 15) / 16) + rows * ((cols + 127) / 128) + rows + 1;
  uint8_t *codes = (uint8_t *)malloc(ncodes > 0 ? ncodes : 1);
  float *scales = (float *)malloc(sizeof(float) * nscales);
  int rc = quant_rows(x, rows, cols, afmt, param, per_row_param, codes, scales);
  if (rc == 0) dequant_rows(codes, scales, rows, cols, afmt, param, per_row_param, out);
  free(codes);
  free(scales);
  return rc;
}

/* ============================ weight dequant ============================ */

typedef struct {
  const void *codes;        /* see layouts below */
  const void *scales;
  const float *global_scale; /* NVFP4: f32 [El] */
  const void *bias;          /* optional [El, R] */
  int bias_is_f32;
} orc_weight;

/* Dequantise row r of expert l of a weight tensor [El, R, C] into out[C].
 *   BF16        codes bf16 [El,R,C]
 *   FP8_TENSOR  codes e4m3 [El,R,C], scales f32 [El]
 *   FP8_CHANNEL codes e4m3 [El,R,C], scales f32 [El,R]
 *   FP8_BLOCK128 codes e4m3 [El,R,C], scales f32 [El,ceil(R/128),ceil(C/128)]
 *   MXFP4       codes u8 [El,R,C/2] (even column low nibble), scales e8m0 u8 [El,R,C/32]
 *   NVFP4       codes u8 [El,R,C/2], scales e4m3 u8 [El,R,C/16], global f32 [El] */
static void dequant_weight_row(int wfmt, const orc_weight *w, long l, long r,
                               long R, long C, double *out) {
  if (wfmt == ORC_W_BF16) {
    const uint16_t *p = (const uint16_t *)w->codes + (l * R + r) * C;
    for (long c = 0; c < C; ++c) out[c] = orc_bf16_decode(p[c]);
  } else if (wfmt == ORC_W_FP8_TENSOR || wfmt == ORC_W_FP8_CHANNEL || wfmt == ORC_W_FP8_BLOCK128) {
    const uint8_t *p = (const uint8_t *)w->codes + (l * R + r) * C;
    const float *s = (const float *)w->scales;
    long RB = (R + 127) / 128, CB = (C + 127) / 128;
    for (long c = 0; c < C; ++c) {
      double sc = (wfmt == ORC_W_FP8_TENSOR) ? s[l]
                : (wfmt == ORC_W_FP8_CHANNEL) ? s[l * R + r]
                : s[(l * RB + r / 128) * CB + c / 128];
      out[c] = orc_e4m3_decode(p[c]) * sc;
    }
  } else if (wfmt == ORC_W_MXFP4) {
    const uint8_t *p = (const uint8_t *)w->codes + (l * R + r) * (C / 2);
    const uint8_t *s = (const uint8_t *)w->scales + (l * R + r) * (C / 32);
    for (long c = 0; c < C; ++c) {
      int q = (c & 1) ? (p[c / 2] >> 4) : (p[c / 2] & 15);
      out[c] = orc_e2m1_decode(q) * orc_e8m0_decode(s[c / 32]);
    }
  } else if (wfmt == ORC_W_NVFP4) {
    const uint8_t *p = (const uint8_t *)w->codes + (l * R + r) * (C / 2);
    const uint8_t *s = (const uint8_t *)w->scales + (l * R + r) * (C / 16);
    double g = (double)w->global_scale[l];
    for (long c = 0; c < C; ++c) {
      int q = (c & 1) ? (p[c / 2] >> 4) : (p[c / 2] & 15);
      out[c] = orc_e2m1_decode(q) * orc_e4m3_decode(s[c / 16]) * g;
    }
  } else {
    for (long c = 0; c < C; ++c) out[c] = NAN;
  }
}

static double weight_bias(const orc_weight *w, long l, long r, long R) {
  if (!w->bias) return 0.0;
  if (w->bias_is_f32) return (double)((const float *)w->bias)[l * R + r];
  return orc_bf16_decode(((const uint16_t *)w->bias)[l * R + r]);
}

/* =============================== activations ============================ */

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* act-and-mul of one (gate, up) pair. */
static double act_and_mul(int act, double g, double u, double alpha, double beta,
                          double limit) {
  if (act == ORC_ACT_SILU) return g * sigmoid(g) * u;
  if (act == ORC_ACT_GELU) return 0.5 * g * (1.0 + erf(g / sqrt(2.0))) * u;
  if (act == ORC_ACT_SWIGLU_OAI) {
    if (limit > 0.0) {
      if (g > limit) g = limit;
      if (u > limit) u = limit;
      if (u < -limit) u = -limit;
    }
    return (u + beta) * g * sigmoid(alpha * g);
  }
  return NAN;
}

/* ============================== fused experts =========================== */

typedef struct {
  int M, K, N, T, E, El;
  int wfmt, afmt, act, gate;
  double swiglu_alpha, swiglu_beta, swiglu_limit;
  const float *a1_scale; /* fp8 tensor static: [1]; NVFP4: one global [1] */
  const float *a2_scale; /* fp8 tensor static: [1]; NVFP4: per expert [El] */
  int weight_on_stage1;  /* apply_router_weight_on_input: w scales the stage-1 output */
  int n_valid_tokens;    /* num_local_tokens: tokens t >= it take no part; -1 = all */
} orc_problem;

/* Stage-2 (intermediate) quantiser implied by the weight / activation format. */
static int stage2_afmt(const orc_problem *p) {
  switch (p->wfmt) {
    case ORC_W_FP8_TENSOR: return p->afmt; /* static or dynamic per tensor */
    case ORC_W_FP8_CHANNEL: return ORC_A_FP8_TOKEN_DYN;
    case ORC_W_FP8_BLOCK128: return ORC_A_FP8_GROUP128_DYN;
    case ORC_W_NVFP4: return ORC_A_NVFP4_DYN;
    case ORC_W_MXFP4: /* w4a4 / w4a8: the intermediate in the activation format */
      return (p->afmt == ORC_A_MXFP4_DYN || p->afmt == ORC_A_MXFP8_DYN) ? p->afmt : ORC_A_BF16;
    default: return ORC_A_BF16; /* no requantisation */
  }
}

/* Computes out[n_tokens, K] (fp64, before the final bf16 rounding) for the
 * listed tokens.  Returns 0, or -1 for an unsupported request (per-tensor
 * dynamic stage-2 needs every token, because its scale spans all slots). */
/* The fused experts of the requested tokens.  When z_pre / z_post are given
 * ([n_tokens * T, N] each, zeroed here), row i*T + k receives the stage-1
 * output of slot k of tokens[i] before and after the stage-2 quantiser (the
 * same values step 4 computes; dropped slots stay zero). */
int orc_fused_experts_x(const orc_problem *p, const uint16_t *x_bf16,
                        const orc_weight *w13, const orc_weight *w2,
                        const int32_t *topk_ids, const float *topk_weights,
                        const int32_t *expert_map, const int32_t *tokens,
                        int n_tokens, double *out, double *z_pre, double *z_post) {
  const long M = p->M, K = p->K, N = p->N, T = p->T;
  const int s2 = stage2_afmt(p);
  if (s2 == ORC_A_FP8_TENSOR_DYN && n_tokens != M) return -1;
  if ((p->afmt == ORC_A_FP8_TENSOR_STATIC || p->afmt == ORC_A_NVFP4_DYN) && !p->a1_scale) return -2;
  if ((s2 == ORC_A_FP8_TENSOR_STATIC || s2 == ORC_A_NVFP4_DYN) && !p->a2_scale) return -2;
  if (p->wfmt == ORC_W_NVFP4 && (!w13->global_scale || !w2->global_scale)) return -2;
  /* apply_router_weight_on_input is defined for one slot per token */
  if (p->weight_on_stage1 && T != 1) return -3;

  /* 1. stage-1 activations of the requested tokens (QDQ where quantised). */
  double *a = (double *)malloc(sizeof(double) * n_tokens * K);
  if (p->afmt == ORC_A_BF16) {
    for (long i = 0; i < n_tokens; ++i)
      for (long c = 0; c < K; ++c) a[i * K + c] = orc_bf16_decode(x_bf16[(long)tokens[i] * K + c]);
  } else if (p->afmt == ORC_A_FP8_TENSOR_DYN) {
    /* the scale spans the whole batch: quantise all rows, keep the requested */
    float *xf = (float *)malloc(sizeof(float) * M * K);
    double *q = (double *)malloc(sizeof(double) * M * K);
    for (long i = 0; i < M * K; ++i) xf[i] = (float)orc_bf16_decode(x_bf16[i]);
    orc_qdq_rows(xf, M, K, p->afmt, p->a1_scale, 0, q);
    for (long i = 0; i < n_tokens; ++i) memcpy(a + i * K, q + (long)tokens[i] * K, sizeof(double) * K);
    free(xf);
    free(q);
  } else {
    float *xf = (float *)malloc(sizeof(float) * n_tokens * K);
    for (long i = 0; i < n_tokens; ++i)
      for (long c = 0; c < K; ++c) xf[i * K + c] = (float)orc_bf16_decode(x_bf16[(long)tokens[i] * K + c]);
    orc_qdq_rows(xf, n_tokens, K, p->afmt, p->a1_scale, 0, a);
    free(xf);
  }

  /* 2. live slots of the requested tokens. */
  long ns = 0;
  long *slot_tok = (long *)malloc(sizeof(long) * n_tokens * T + 1);
  long *slot_row = (long *)malloc(sizeof(long) * n_tokens * T + 1);
  int *slot_exp = (int *)malloc(sizeof(int) * n_tokens * T + 1);
  double *slot_w = (double *)malloc(sizeof(double) * n_tokens * T + 1);
  for (long i = 0; i < n_tokens; ++i)
    for (long k = 0; k < T; ++k) {
      long t = tokens[i];
      if (p->n_valid_tokens >= 0 && t >= p->n_valid_tokens) continue;  /* padding row */
      int l = local_expert(topk_ids[t * T + k], expert_map, p->E, p->El);
      if (l < 0) continue;
      slot_tok[ns] = i;
      slot_row[ns] = i * T + k;
      slot_exp[ns] = l;
      slot_w[ns] = (double)topk_weights[t * T + k];
      ++ns;
    }

  /* 3. gate/up GEMM: h[s][j] = a[t(s)] . W13[l(s), j, :] + b13[l(s), j]. */
  double *h = (double *)malloc(sizeof(double) * (ns ? ns : 1) * 2 * N);
  for (int l = 0; l < p->El; ++l) {
    int any = 0;
    for (long s = 0; s < ns; ++s) if (slot_exp[s] == l) { any = 1; break; }
    if (!any) continue;
#pragma omp parallel
    {
      double *row = (double *)malloc(sizeof(double) * K);
#pragma omp for schedule(static)
      for (long j = 0; j < 2 * N; ++j) {
        dequant_weight_row(p->wfmt, w13, l, j, 2 * N, K, row);
        double b = weight_bias(w13, l, j, 2 * N);
        for (long s = 0; s < ns; ++s) {
          if (slot_exp[s] != l) continue;
          const double *av = a + slot_tok[s] * K;
          double acc = 0.0;
          for (long c = 0; c < K; ++c) acc += av[c] * row[c];
          h[s * 2 * N + j] = acc + b;
        }
      }
      free(row);
    }
  }

  /* 4. activation on (gate, up) pairs, then the stage-2 quantiser. */
  double *z = (double *)malloc(sizeof(double) * (ns ? ns : 1) * N);
  for (long s = 0; s < ns; ++s)
    for (long j = 0; j < N; ++j) {
      double g, u;
      if (p->gate == ORC_GATE_SEPARATED) { g = h[s * 2 * N + j]; u = h[s * 2 * N + N + j]; }
      else { g = h[s * 2 * N + 2 * j]; u = h[s * 2 * N + 2 * j + 1]; }
      z[s * N + j] = act_and_mul(p->act, g, u, p->swiglu_alpha, p->swiglu_beta, p->swiglu_limit);
      /* doweight_stage1 / tkw1: the router weight scales the stage-1 output
       * (before the stage-2 quantiser) instead of the stage-2 output */
      if (p->weight_on_stage1) z[s * N + j] *= slot_w[s];
    }
  if (z_pre) {
    memset(z_pre, 0, sizeof(double) * n_tokens * T * N);
    for (long s = 0; s < ns; ++s) memcpy(z_pre + slot_row[s] * N, z + s * N, sizeof(double) * N);
  }
  if (s2 != ORC_A_BF16 && ns > 0) {
    float *zf = (float *)malloc(sizeof(float) * ns * N);
    for (long i = 0; i < ns * N; ++i) zf[i] = (float)z[i];
    if (s2 == ORC_A_NVFP4_DYN) {
      float *g_row = (float *)malloc(sizeof(float) * ns);
      for (long s = 0; s < ns; ++s) g_row[s] = p->a2_scale[slot_exp[s]];
      orc_qdq_rows(zf, ns, N, s2, g_row, 1, z);
      free(g_row);
    } else {
      orc_qdq_rows(zf, ns, N, s2, p->a2_scale, 0, z);
    }
    free(zf);
  }

  if (z_post) {
    memset(z_post, 0, sizeof(double) * n_tokens * T * N);
    for (long s = 0; s < ns; ++s) memcpy(z_post + slot_row[s] * N, z + s * N, sizeof(double) * N);
  }

  /* 5. down GEMM and the top-k weighted reduce. */
  memset(out, 0, sizeof(double) * n_tokens * K);
  for (int l = 0; l < p->El; ++l) {
    int any = 0;
    for (long s = 0; s < ns; ++s) if (slot_exp[s] == l) { any = 1; break; }
    if (!any) continue;
#pragma omp parallel
    {
      double *row = (double *)malloc(sizeof(double) * N);
#pragma omp for schedule(static)
      for (long i = 0; i < K; ++i) {
        dequant_weight_row(p->wfmt, w2, l, i, K, N, row);
        double b = weight_bias(w2, l, i, K);
        for (long s = 0; s < ns; ++s) {
          if (slot_exp[s] != l) continue;
          const double *zv = z + s * N;
          double acc = 0.0;
          for (long j = 0; j < N; ++j) acc += zv[j] * row[j];
          out[slot_tok[s] * K + i] += (p->weight_on_stage1 ? 1.0 : slot_w[s]) * (acc + b);
        }
      }
      free(row);
    }
  }

  free(a); free(slot_tok); free(slot_row); free(slot_exp); free(slot_w); free(h); free(z);
  return 0;
}

int orc_fused_experts(const orc_problem *p, const uint16_t *x_bf16,
                      const orc_weight *w13, const orc_weight *w2,
                      const int32_t *topk_ids, const float *topk_weights,
                      const int32_t *expert_map, const int32_t *tokens,
                      int n_tokens, double *out) {
  return orc_fused_experts_x(p, x_bf16, w13, w2, topk_ids, topk_weights, expert_map, tokens,
                             n_tokens, out, NULL, NULL);
}

/*
 * beam_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, FP64 CPU definition of the group-limited Mixture-of-Experts
 * block of the Beam model.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this code; the product path
 * (the CUDA library) never does, and the two share no code.
 *
 * Source of the definition (two translations of the same launch post):
 *   [zh] "Reflection 发布 501B 开放模型 Beam，支持自托管定制与扩展" (sihot.dev),
 *        section 混合专家（Mixture of Experts）, and section 残差流 for the
 *        list of places computed in FP32.
 *   [de] "Willkommen Beam: ein offenes 501B-Modell, das Sie besitzen,
 *        anpassen und skalieren können" (spke.com), section "Mixture of
 *        Experts", and section "Residual Stream" for the FP32 list.
 *
 * What the pages fix (restated):
 *   - 256 experts, each a SwiGLU MLP with intermediate size 2560 on hidden
 *     size 5120;
 *   - the router scores every expert with a sigmoid, splits the experts into
 *     8 groups of 32, ranks each group by the sum of its two best scores,
 *     keeps the 4 best groups and takes the 8 best experts inside them;
 *   - no shared expert; the expert outputs are combined with the normalised
 *     router weights multiplied by 2.5;
 *   - the router and the SwiGLU product are computed (at least) in FP32.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - experts 32j..32j+31 form group j (contiguous groups);
 *   - an optional per-expert bias b is added to the sigmoid scores for the
 *     SELECTION only (group ranking and top-8); the combine weights use the
 *     unbiased scores.  With b = 0 this is exactly the pages' text;
 *   - ties: the lower group index / lower expert index wins; selected ids
 *     are listed by descending biased score, ties by lower id;
 *   - weights are oriented like a linear layer, [out, in]:
 *     gate/up [I, H], down [H, I];
 *   - NVFP4: E2M1 codes two per byte, even K index in the low nibble, one
 *     E4M3 scale per 16 consecutive K elements, one FP32 global scale per
 *     weight matrix; value = e2m1 * e4m3 * global.
 *
 * Arithmetic is IEEE double throughout (the exact definition; the pages'
 * FP32 is the minimum precision of the product path).  Inputs are the exact
 * bytes the product path sees (FP32, BF16 bit patterns, packed NVFP4);
 * every format is decoded exactly to double by the small decoders below.
 * No blocking, fusion or reordering of any sum: every dot product runs
 * h = 0..H-1 (or i = 0..I-1) in order.  Threads split independent outputs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_NVFP4 2
#define ORACLE_FP8 3

/* ------------------------------------------------------------------ */
/* Exact decoders (each format written out from its bit layout).      */
/* ------------------------------------------------------------------ */

/* BF16: the upper 16 bits of an IEEE binary32. */
double oracle_decode_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* E4M3 ("fn" variant of the OCP 8-bit float): 1 sign, 4 exponent bits
 * (bias 7), 3 mantissa bits, no infinities, S.1111.111 is NaN. */
double oracle_decode_e4m3(uint8_t code) {
  int sign = (code >> 7) & 1;
  int ex = (code >> 3) & 0xF;
  int man = code & 7;
  double v;
  if (ex == 0xF && man == 7) return NAN;
  if (ex == 0)
    v = ldexp((double)man / 8.0, -6); /* subnormal: 0.mmm * 2^(1-7) */
  else
    v = ldexp(1.0 + (double)man / 8.0, ex - 7);
  return sign ? -v : v;
}

/* Float -> E4M3 (layout above): round to nearest, ties to even; magnitudes
 * of 448 (the largest finite value) and above give +-448 (saturation, as the
 * FP8 formats have no infinity).  Written from the layout: the binade of |v|
 * fixes the quantum 2^(e-3) (2^-9 below 2^-6, the subnormal range), |v| is
 * rounded to a whole number of quanta, and a carry into 16 quanta moves to
 * the next binade. */
uint8_t oracle_encode_e4m3(float v) {
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs((double)v);
  if (isnan(v)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1): binade 2^(e2-1) */
  int e = e2 - 1;
  if (e < -6) e = -6;
  double m = nearbyint(ldexp(a, 3 - e)); /* quanta of 2^(e-3); default mode: ties to even */
  if (m >= 16.0) {
    e += 1;
    m = 8.0;
  }
  if (m < 8.0) return sign | (uint8_t)m; /* subnormal (only reachable for e = -6): exponent field 0 */
  return sign | (uint8_t)(((e + 7) << 3) | ((int)m - 8));
}

/* Per-row dynamic quantisation of a GEMM input row to E4M3, the reading used
 * for FP8 expert weights: the row's scale is s = amax / 448 (amax = the
 * largest magnitude in the row; FP32 division; s = 1 when that is 0), each
 * element is encoded as E4M3(a / s) with the division in FP32, and stands for
 * e4m3 * s.  Both decisions are taken in FP32 so that the product path, which
 * makes them in FP32 too, picks the same codes from the same inputs. */
void oracle_quantize_e4m3_row(const float* a, int64_t K, uint8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int64_t j = 0; j < K; ++j) {
    const float m = fabsf(a[j]);
    if (m > amax) amax = m;
  }
  volatile float s = amax / 448.0f; /* one FP32 rounding */
  float sf = s;
  if (sf == 0.0f) sf = 1.0f;
  for (int64_t j = 0; j < K; ++j) {
    volatile float q = a[j] / sf;
    codes[j] = oracle_encode_e4m3(q);
  }
  *scale = sf;
}

/* E2M1 (OCP 4-bit float): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit,
 * no infinities or NaN. */
double oracle_decode_e2m1(uint8_t nibble) {
  int sign = (nibble >> 3) & 1;
  int ex = (nibble >> 1) & 3;
  int man = nibble & 1;
  double v;
  if (ex == 0)
    v = 0.5 * (double)man; /* subnormal: 0.m * 2^(1-1) */
  else
    v = ldexp(1.0 + 0.5 * (double)man, ex - 1);
  return sign ? -v : v;
}

/* double -> the nearest BF16 value (ties to even), as a float, rounded from
 * the double's own value (no intermediate FP32 rounding): |v| is written in
 * quanta of 2^(e-7) (8 significant bits in its binade 2^e) and rounded to a
 * whole number of them. */
float oracle_round_bf16(double v) {
  if (v != v) return (float)v;
  if (v == 0.0) return (float)v;
  int e2;
  const double a = fabs(v);
  frexp(a, &e2); /* a in [2^(e2-1), 2^e2) */
  int e = e2 - 1;
  if (e < -126) e = -126; /* BF16 subnormals share FP32's exponent range */
  const double q = nearbyint(ldexp(a, 7 - e)); /* quanta of 2^(e-7): 8 significant bits */
  double r = ldexp(q, e - 7);
  if (r > 0x1.FEp127) r = INFINITY; /* beyond the largest finite BF16 */
  return (float)(v < 0 ? -r : r);
}

/* Float -> E2M1 code (layout at oracle_decode_e2m1): the nearest of the
 * eight magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, ties to the even code,
 * magnitudes above 6 giving 6 (no infinity in the format); a search over the
 * magnitudes in code order. */
uint8_t oracle_encode_e2m1(float v) {
  const uint8_t sign = signbit(v) ? 0x8 : 0x0;
  const double a = fabs((double)v);
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    const double d = fabs(a - oracle_decode_e2m1((uint8_t)c));
    if (d < bd || (d == bd && c % 2 == 0)) {
      best = c;
      bd = d;
    }
  }
  return sign | (uint8_t)best;
}

/* Per-row dynamic NVFP4 quantisation of a GEMM input row -- the reading used
 * for NVFP4 activations (W4A4; the launch post names NVFP4 only as a weight
 * format): the row's global scale g = amax / (6 * 448) in FP32 (1 when amax is
 * 0), the same recipe as the weights' per-matrix scale but per row; each
 * block of 16 consecutive elements the E4M3 scale s = E4M3((bmax / 6) / g)
 * (FP32 divisions, nearest even, saturating at 448); each element the E2M1
 * code of a / (s * g) (FP32 product and division; code 0 when s is 0).  The
 * element stands for e2m1 * s * g.  codes: one code per byte, [K]. */
void oracle_quantize_nvfp4_row(const float* a, int64_t K, uint8_t* codes, uint8_t* scales, float* global) {
  float amax = 0.0f;
  for (int64_t j = 0; j < K; ++j) {
    const float m = fabsf(a[j]);
    if (m > amax) amax = m;
  }
  volatile float g = amax / (6.0f * 448.0f);
  float gf = g;
  if (gf == 0.0f) gf = 1.0f;
  for (int64_t b = 0; b < K / 16; ++b) {
    float bmax = 0.0f;
    for (int j = 0; j < 16; ++j) {
      const float m = fabsf(a[b * 16 + j]);
      if (m > bmax) bmax = m;
    }
    volatile float t = bmax / 6.0f;
    volatile float q = t / gf;
    const uint8_t sc = oracle_encode_e4m3(q);
    scales[b] = sc;
    volatile float sv = (float)oracle_decode_e4m3(sc);
    volatile float d = sv * gf;
    for (int j = 0; j < 16; ++j) {
      if (sv == 0.0f || d == 0.0f) {
        codes[b * 16 + j] = 0;
        continue;
      }
      volatile float e = a[b * 16 + j] / d;
      codes[b * 16 + j] = oracle_encode_e2m1(e);
    }
  }
  *global = gf;
}

/* One element [row, k] of a weight matrix with `cols` columns (K). */
typedef struct {
  int dtype;            /* ORACLE_F32 / ORACLE_BF16 / ORACLE_NVFP4 / ORACLE_FP8 */
  const void* data;     /* f32 [rows, cols] | bf16 [rows, cols] | u8 [rows, cols/2] | u8 [rows, cols] */
  const uint8_t* scale; /* NVFP4 only: E4M3 [rows, cols/16] */
  double global_scale;  /* NVFP4 only */
  int64_t cols;
  const float* row_scale; /* FP8 only: FP32 scale per row [rows] */
} oracle_matrix_t;

static double mat_elem(const oracle_matrix_t* m, int64_t row, int64_t k) {
  if (m->dtype == ORACLE_F32) return (double)((const float*)m->data)[row * m->cols + k];
  if (m->dtype == ORACLE_BF16) return oracle_decode_bf16(((const uint16_t*)m->data)[row * m->cols + k]);
  if (m->dtype == ORACLE_FP8)
    return oracle_decode_e4m3(((const uint8_t*)m->data)[row * m->cols + k]) * (double)m->row_scale[row];
  /* NVFP4: byte k/2 of the row holds elements k (low nibble, k even) and k+1. */
  {
    uint8_t byte = ((const uint8_t*)m->data)[row * (m->cols / 2) + k / 2];
    uint8_t nib = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    uint8_t sc = m->scale[row * (m->cols / 16) + k / 16];
    return oracle_decode_e2m1(nib) * oracle_decode_e4m3(sc) * m->global_scale;
  }
}

static double act_elem(const void* x, int dtype, int64_t idx) {
  if (dtype == ORACLE_F32) return (double)((const float*)x)[idx];
  return oracle_decode_bf16(((const uint16_t*)x)[idx]);
}

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* ------------------------------------------------------------------ */
/* A tiny fork/join helper: run fn(arg, lo, hi) over [0, n) in nthreads */
/* contiguous slices.                                                 */
/* ------------------------------------------------------------------ */
typedef void (*range_fn)(void* arg, int64_t lo, int64_t hi);
typedef struct {
  range_fn fn;
  void* arg;
  int64_t lo, hi;
} slice_t;

static void* slice_main(void* p) {
  slice_t* s = (slice_t*)p;
  s->fn(s->arg, s->lo, s->hi);
  return NULL;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void* arg) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
  if (nthreads == 1) {
    fn(arg, 0, n);
    return;
  }
  pthread_t th[512];
  slice_t sl[512];
  int started[512];
  for (int i = 0; i < nthreads; ++i) {
    sl[i].fn = fn;
    sl[i].arg = arg;
    sl[i].lo = n * i / nthreads;
    sl[i].hi = n * (i + 1) / nthreads;
    started[i] = pthread_create(&th[i], NULL, slice_main, &sl[i]) == 0;
    if (!started[i]) slice_main(&sl[i]); /* could not start a thread: run inline */
  }
  for (int i = 0; i < nthreads; ++i)
    if (started[i]) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------ */
/* Routing                                                            */
/* ------------------------------------------------------------------ */
typedef struct {
  int64_t H;
  int E, G, KG, K;
  double scale;
  const void* x;
  int x_dtype;
  const float* wr;
  const float* bias;
  int32_t* ids;
  double* weights;
  double* margin_group;
  double* margin_expert;
  double* scores;
  double* logits;
  int status;
} route_args_t;

/* "a better than b" for (value, index) pairs: larger value, then lower index. */
static int better(double va, int ia, double vb, int ib) { return va > vb || (va == vb && ia < ib); }

static void route_tokens(void* p, int64_t lo, int64_t hi) {
  route_args_t* a = (route_args_t*)p;
  const int E = a->E, G = a->G, KG = a->KG, K = a->K;
  const int per = E / G;
  double* l = (double*)malloc(sizeof(double) * E);
  double* s = (double*)malloc(sizeof(double) * E);
  double* sel = (double*)malloc(sizeof(double) * E);
  double* g = (double*)malloc(sizeof(double) * G);
  int* kept = (int*)malloc(sizeof(int) * G);
  int* taken = (int*)malloc(sizeof(int) * E);
  if (!l || !s || !sel || !g || !kept || !taken) {
    a->status = -2;
    free(l); free(s); free(sel); free(g); free(kept); free(taken);
    return;
  }
  for (int64_t t = lo; t < hi; ++t) {
    /* 1. logits: l[e] = sum_h x[t,h] * Wr[e,h]; 2. s = sigmoid(l). */
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int64_t h = 0; h < a->H; ++h)
        acc += act_elem(a->x, a->x_dtype, t * a->H + h) * (double)a->wr[(int64_t)e * a->H + h];
      l[e] = acc;
      s[e] = sigmoid(acc);
      sel[e] = s[e] + (a->bias ? (double)a->bias[e] : 0.0);
    }
    if (a->logits) memcpy(a->logits + t * E, l, sizeof(double) * E);
    if (a->scores) memcpy(a->scores + t * E, s, sizeof(double) * E);

    /* 3. group score: sum of the two largest selection scores in the group. */
    for (int j = 0; j < G; ++j) {
      int i1 = -1, i2 = -1;
      for (int e = j * per; e < (j + 1) * per; ++e)
        if (i1 < 0 || better(sel[e], e, sel[i1], i1)) i1 = e;
      for (int e = j * per; e < (j + 1) * per; ++e)
        if (e != i1 && (i2 < 0 || better(sel[e], e, sel[i2], i2))) i2 = e;
      g[j] = sel[i1] + (per > 1 ? sel[i2] : 0.0);
      kept[j] = 0;
    }
    /* 4. keep the KG best groups (repeated selection of the best remaining). */
    double g_last = 0.0;
    for (int r = 0; r < KG; ++r) {
      int best = -1;
      for (int j = 0; j < G; ++j)
        if (!kept[j] && (best < 0 || better(g[j], j, g[best], best))) best = j;
      kept[best] = 1;
      g_last = g[best];
    }
    {
      int next = -1;
      for (int j = 0; j < G; ++j)
        if (!kept[j] && (next < 0 || better(g[j], j, g[next], next))) next = j;
      a->margin_group[t] = next < 0 ? INFINITY : g_last - g[next];
    }
    /* 5. the K best experts among the kept groups, best first. */
    for (int e = 0; e < E; ++e) taken[e] = 0;
    double ssum = 0.0, sel_last = 0.0;
    for (int k = 0; k < K; ++k) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (kept[e / per] && !taken[e] && (best < 0 || better(sel[e], e, sel[best], best))) best = e;
      taken[best] = 1;
      a->ids[t * K + k] = best;
      sel_last = sel[best];
    }
    {
      int next = -1;
      for (int e = 0; e < E; ++e)
        if (kept[e / per] && !taken[e] && (next < 0 || better(sel[e], e, sel[next], next))) next = e;
      a->margin_expert[t] = next < 0 ? INFINITY : sel_last - sel[next];
    }
    /* 6. weights: unbiased scores normalised over the K chosen, times scale. */
    for (int k = 0; k < K; ++k) ssum += s[a->ids[t * K + k]];
    for (int k = 0; k < K; ++k) a->weights[t * K + k] = s[a->ids[t * K + k]] / ssum * a->scale;
  }
  free(l); free(s); free(sel); free(g); free(kept); free(taken);
}

/*
 * oracle_route: routing decision for T tokens.
 *   x        [T, H]   FP32 or BF16 bits (x_dtype)
 *   wr       [E, H]   FP32 router weight
 *   bias     [E]      FP32 selection bias, or NULL
 *   ids      [T, K]   out: chosen experts, best first
 *   weights  [T, K]   out: combine weights (sum = scale)
 *   margin_group  [T] out: g(4th kept) - g(best dropped)
 *   margin_expert [T] out: sel(8th chosen) - sel(best unchosen in kept groups)
 *   scores   [T, E]   out (nullable): unbiased sigmoid scores
 *   logits   [T, E]   out (nullable): router logits
 * Returns 0, or -1 on a bad shape, -2 on allocation failure.
 */
int oracle_route(int64_t T, int64_t H, int E, int G, int KG, int K, double scale, const void* x,
                 int x_dtype, const float* wr, const float* bias, int32_t* ids, double* weights,
                 double* margin_group, double* margin_expert, double* scores, double* logits,
                 int nthreads) {
  if (T < 0 || H <= 0 || E <= 0 || G <= 0 || E % G != 0 || KG <= 0 || KG > G || K <= 0 ||
      K > KG * (E / G))
    return -1;
  route_args_t a = {H, E, G, KG, K, scale, x, x_dtype, wr, bias, ids, weights,
                    margin_group, margin_expert, scores, logits, 0};
  parallel_for(T, nthreads, route_tokens, &a);
  return a.status;
}

/* ------------------------------------------------------------------ */
/* One expert's SwiGLU MLP on a batch of rows                         */
/* ------------------------------------------------------------------ */
typedef struct {
  int64_t H, I, n;
  const void* x;
  int x_dtype;
  oracle_matrix_t wg, wu, wd;
  double* h; /* [n, I] */
  double* out; /* [n, H] */
  const double* xq; /* FP8 only: quantised x values [n, H] (NULL: read x) */
} ffn_args_t;

/* h[r, i] = silu(a) * u with a = x_r . Wg[i,:], u = x_r . Wu[i,:]. */
static void ffn_hidden(void* p, int64_t lo, int64_t hi) {
  ffn_args_t* a = (ffn_args_t*)p;
  for (int64_t q = lo; q < hi; ++q) {
    int64_t r = q / a->I, i = q % a->I;
    double ga = 0.0, ua = 0.0;
    for (int64_t hh = 0; hh < a->H; ++hh) {
      double xv = a->xq ? a->xq[r * a->H + hh] : act_elem(a->x, a->x_dtype, r * a->H + hh);
      ga += xv * mat_elem(&a->wg, i, hh);
      ua += xv * mat_elem(&a->wu, i, hh);
    }
    a->h[q] = ga * sigmoid(ga) * ua; /* SiLU(gate) * up */
  }
}

/* out[r, j] = h_r . Wd[j,:] */
static void ffn_down(void* p, int64_t lo, int64_t hi) {
  ffn_args_t* a = (ffn_args_t*)p;
  for (int64_t q = lo; q < hi; ++q) {
    int64_t r = q / a->H, j = q % a->H;
    double acc = 0.0;
    for (int64_t i = 0; i < a->I; ++i) acc += a->h[r * a->I + i] * mat_elem(&a->wd, j, i);
    a->out[q] = acc;
  }
}

/*
 * oracle_expert_ffn: one expert applied to n rows.
 *   x        [n, H]   FP32 or BF16 bits (x_dtype)
 *   wg, wu   [I, H]   w_dtype: FP32 | BF16 bits | NVFP4 packed [I, H/2]
 *   wd       [H, I]   same dtype; NVFP4 packed [H, I/2]
 *   sg,su,sd          NVFP4 only: E4M3 block scales [I, H/16], [I, H/16], [H, I/16]
 *   gg,gu,gd          NVFP4 only: global scales
 *   out      [n, H]   out
 *   h_out    [n, I]   out (nullable): SwiGLU activations
 */
int oracle_expert_ffn(int64_t H, int64_t I, int64_t n, const void* x, int x_dtype, int w_dtype,
                      const void* wg, const void* wu, const void* wd, const uint8_t* sg,
                      const uint8_t* su, const uint8_t* sd, double gg, double gu, double gd,
                      double* out, double* h_out, int nthreads) {
  if (H <= 0 || I <= 0 || n < 0) return -1;
  if (w_dtype == ORACLE_NVFP4 && (H % 16 != 0 || I % 16 != 0 || !sg || !su || !sd)) return -1;
  ffn_args_t a;
  a.H = H;
  a.I = I;
  a.n = n;
  a.x = x;
  a.x_dtype = x_dtype;
  a.xq = NULL;
  if (w_dtype == ORACLE_FP8) return -1; /* oracle_expert_ffn_fp8 */
  a.wg = (oracle_matrix_t){w_dtype, wg, sg, gg, H, NULL};
  a.wu = (oracle_matrix_t){w_dtype, wu, su, gu, H, NULL};
  a.wd = (oracle_matrix_t){w_dtype, wd, sd, gd, I, NULL};
  a.out = out;
  a.h = h_out ? h_out : (double*)malloc(sizeof(double) * (size_t)(n * I > 0 ? n * I : 1));
  if (!a.h) return -2;
  parallel_for(n * I, nthreads, ffn_hidden, &a);
  parallel_for(n * H, nthreads, ffn_down, &a);
  if (!h_out) free(a.h);
  return 0;
}

/*
 * oracle_expert_ffn_fp8: one expert with FP8 weights applied to n rows.  The
 * launch post names an FP8 checkpoint beside BF16 and NVFP4 (section
 * "Mixture of Experts") without giving its layout; it is read as E4M3
 * weights with one FP32 scale per output row (weight = e4m3 * row_scale) and
 * FP8 activations quantised per row at run time (oracle_quantize_e4m3_row):
 * the rows of x before gate/up, the rows of h before down.  The quantised
 * inputs are the block's activations in their storage type: x as given
 * (FP32 or BF16), h as a BF16 tensor, i.e. rounded to BF16 (nearest even)
 * before its row is quantised.
 *   x          [n, H]  FP32 or BF16 bits (x_dtype), quantised from its own values
 *   wg, wu     [I, H]  E4M3 codes; rg, ru [I] row scales
 *   wd         [H, I]  E4M3 codes; rd [H] row scales
 *   out        [n, H]  out;  h_out [n, I] out (nullable): h before rounding
 * h = silu(xq . wg) * (xq . wu) in double; each h row is rounded to BF16 and
 * quantised; out = hq . wd.  Sums run in index order, in double.
 */
int oracle_expert_ffn_fp8(int64_t H, int64_t I, int64_t n, const void* x, int x_dtype, const uint8_t* wg,
                          const uint8_t* wu, const uint8_t* wd, const float* rg, const float* ru, const float* rd,
                          double* out, double* h_out, int nthreads) {
  if (H <= 0 || I <= 0 || n < 0 || !rg || !ru || !rd) return -1;
  const int64_t nn = n > 0 ? n : 1;
  float* rowf = (float*)malloc(sizeof(float) * (size_t)(H > I ? H : I));
  uint8_t* codes = (uint8_t*)malloc((size_t)(H > I ? H : I));
  double* xq = (double*)malloc(sizeof(double) * (size_t)(nn * H));
  double* hq = (double*)malloc(sizeof(double) * (size_t)(nn * I));
  double* h = h_out ? h_out : (double*)malloc(sizeof(double) * (size_t)(nn * I));
  int rc = 0;
  if (!rowf || !codes || !xq || !hq || !h) {
    rc = -2;
    goto done;
  }
  /* x rows -> E4M3 codes and scales -> the values the GEMM multiplies */
  for (int64_t r = 0; r < n; ++r) {
    float sc;
    for (int64_t j = 0; j < H; ++j) rowf[j] = (float)act_elem(x, x_dtype, r * H + j);
    oracle_quantize_e4m3_row(rowf, H, codes, &sc);
    for (int64_t j = 0; j < H; ++j) xq[r * H + j] = oracle_decode_e4m3(codes[j]) * (double)sc;
  }
  {
    ffn_args_t a;
    a.H = H;
    a.I = I;
    a.n = n;
    a.x = NULL;
    a.x_dtype = -1;
    a.wg = (oracle_matrix_t){ORACLE_FP8, wg, NULL, 1.0, H, rg};
    a.wu = (oracle_matrix_t){ORACLE_FP8, wu, NULL, 1.0, H, ru};
    a.wd = (oracle_matrix_t){ORACLE_FP8, wd, NULL, 1.0, I, rd};
    a.h = h;
    a.out = out;
    a.xq = xq;
    parallel_for(n * I, nthreads, ffn_hidden, &a);
    /* h rows -> BF16 -> E4M3 codes and scales */
    for (int64_t r = 0; r < n; ++r) {
      float sc;
      for (int64_t i = 0; i < I; ++i) rowf[i] = oracle_round_bf16(h[r * I + i]);
      oracle_quantize_e4m3_row(rowf, I, codes, &sc);
      for (int64_t i = 0; i < I; ++i) hq[r * I + i] = oracle_decode_e4m3(codes[i]) * (double)sc;
    }
    a.h = hq;
    parallel_for(n * H, nthreads, ffn_down, &a);
  }
done:
  free(rowf);
  free(codes);
  free(xq);
  free(hq);
  if (!h_out) free(h);
  return rc;
}

/*
 * oracle_expert_ffn_w4a4: one expert with NVFP4 weights (layout as in
 * oracle_expert_ffn) whose GEMM inputs are quantised per row to NVFP4 at run
 * time (oracle_quantize_nvfp4_row): x as given before gate/up, h rounded to
 * BF16 before down.  Values are decoded exactly and summed in double in
 * index order.  h_out (nullable) receives h before rounding.
 */
int oracle_expert_ffn_w4a4(int64_t H, int64_t I, int64_t n, const void* x, int x_dtype, const uint8_t* wg,
                           const uint8_t* wu, const uint8_t* wd, const uint8_t* sg, const uint8_t* su,
                           const uint8_t* sd, double gg, double gu, double gd, double* out, double* h_out,
                           int nthreads) {
  if (H <= 0 || I <= 0 || n < 0 || H % 16 != 0 || I % 16 != 0 || !sg || !su || !sd) return -1;
  const int64_t nn = n > 0 ? n : 1, KM = H > I ? H : I;
  float* rowf = (float*)malloc(sizeof(float) * (size_t)KM);
  uint8_t* codes = (uint8_t*)malloc((size_t)KM);
  uint8_t* scales = (uint8_t*)malloc((size_t)(KM / 16));
  double* xq = (double*)malloc(sizeof(double) * (size_t)(nn * H));
  double* hq = (double*)malloc(sizeof(double) * (size_t)(nn * I));
  double* h = h_out ? h_out : (double*)malloc(sizeof(double) * (size_t)(nn * I));
  int rc = 0;
  if (!rowf || !codes || !scales || !xq || !hq || !h) {
    rc = -2;
    goto done;
  }
  for (int64_t r = 0; r < n; ++r) {
    float g;
    for (int64_t j = 0; j < H; ++j) rowf[j] = (float)act_elem(x, x_dtype, r * H + j);
    oracle_quantize_nvfp4_row(rowf, H, codes, scales, &g);
    for (int64_t j = 0; j < H; ++j)
      xq[r * H + j] = oracle_decode_e2m1(codes[j]) * oracle_decode_e4m3(scales[j / 16]) * (double)g;
  }
  {
    ffn_args_t a;
    a.H = H;
    a.I = I;
    a.n = n;
    a.x = NULL;
    a.x_dtype = -1;
    a.wg = (oracle_matrix_t){ORACLE_NVFP4, wg, sg, gg, H, NULL};
    a.wu = (oracle_matrix_t){ORACLE_NVFP4, wu, su, gu, H, NULL};
    a.wd = (oracle_matrix_t){ORACLE_NVFP4, wd, sd, gd, I, NULL};
    a.h = h;
    a.out = out;
    a.xq = xq;
    parallel_for(n * I, nthreads, ffn_hidden, &a);
    for (int64_t r = 0; r < n; ++r) {
      float g;
      for (int64_t i = 0; i < I; ++i) rowf[i] = oracle_round_bf16(h[r * I + i]);
      oracle_quantize_nvfp4_row(rowf, I, codes, scales, &g);
      for (int64_t i = 0; i < I; ++i)
        hq[r * I + i] = oracle_decode_e2m1(codes[i]) * oracle_decode_e4m3(scales[i / 16]) * (double)g;
    }
    a.h = hq;
    parallel_for(n * H, nthreads, ffn_down, &a);
  }
done:
  free(rowf);
  free(codes);
  free(scales);
  free(xq);
  free(hq);
  if (!h_out) free(h);
  return rc;
}

/*
 * oracle_combine: y[t, :] = sum_k weights[t,k] * o[t,k,:], k = 0..K-1 in order.
 * No shared-expert term.
 */
int oracle_combine(int64_t n, int K, int64_t H, const double* weights, const double* o, double* y) {
  if (n < 0 || K <= 0 || H <= 0) return -1;
  for (int64_t t = 0; t < n; ++t)
    for (int64_t j = 0; j < H; ++j) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) acc += weights[t * K + k] * o[(t * K + k) * H + j];
      y[t * H + j] = acc;
    }
  return 0;
}

/*
 * oracle_residual_update: the step that follows the MoE sublayer in the
 * residual stream (Beam launch post, section "Residual Stream"): the input
 * embedding is step 1; at step k >= 2 the stream is kept with weight
 * sqrt((k-1)/k) and the sublayer output is added with weight 1/sqrt(k), the
 * two weights' squares summing to one.  Every sublayer's output is
 * normalised after the sublayer.  The post does not say which norm; it is
 * read as RMSNorm (the norm the post names elsewhere, in section "Attention",
 * for queries and keys) with a learned scale w and eps inside the root; here,
 * in double:
 *   yn[t, j]  = y[t, j] / sqrt(mean_j' y[t, j']^2 + eps) * w[j]
 *   out[t, j] = sqrt((k-1)/k) * stream[t, j] + yn[t, j] / sqrt(k)
 */
int oracle_residual_update(int64_t n, int64_t H, const double* y, const double* stream, const double* w, double eps,
                           int k, double* out) {
  if (n < 0 || H <= 0 || k < 2 || !(eps >= 0.0)) return -1;
  const double keep = sqrt((double)(k - 1) / (double)k), add = 1.0 / sqrt((double)k);
  for (int64_t t = 0; t < n; ++t) {
    double ss = 0.0;
    for (int64_t j = 0; j < H; ++j) ss += y[t * H + j] * y[t * H + j];
    const double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int64_t j = 0; j < H; ++j)
      out[t * H + j] = keep * stream[t * H + j] + y[t * H + j] * inv * w[j] * add;
  }
  return 0;
}

/*
 * oracle_dispatch: per-expert route lists implied by "each token runs only
 * its 8 experts".  Route r = t*K + k goes to expert ids[r].
 *   counts  [E]    routes per expert
 *   offsets [E+1]  exclusive prefix sum of counts
 *   perm    [R]    route ids grouped by expert, ascending r inside an expert
 *   pos     [R]    inverse: perm[pos[r]] == r
 */
int oracle_dispatch(int64_t R, int E, const int32_t* ids, int32_t* counts, int32_t* offsets,
                    int32_t* perm, int32_t* pos) {
  if (R < 0 || E <= 0) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t r = 0; r < R; ++r) {
    if (ids[r] < 0 || ids[r] >= E) return -1;
    counts[ids[r]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * E);
  if (!fill) return -2;
  for (int e = 0; e < E; ++e) fill[e] = offsets[e];
  for (int64_t r = 0; r < R; ++r) {
    int32_t p = fill[ids[r]]++;
    perm[p] = (int32_t)r;
    pos[r] = p;
  }
  free(fill);
  return 0;
}

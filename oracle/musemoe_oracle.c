/* CPU oracle of the MuseSpark1x MoE decode block in plain C (float64, one
 * thread; no BLAS, every sum a sequential loop).
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, __graft_entry__.smoke() and the
 * CPU-baseline / reference legs of bench.py load this library. It shares no
 * code with the CUDA path and restates, step by step and in the same order,
 * what oracle/musemoe_oracle.py restates from the pages:
 *
 *  - router GEMV and routing rule: page "vllm.models.muse_spark.amd.
 *    muse_moe_runner", MuseSpark1xRouter (docstring and
 *    _compute_routing_native): optional output multiplier -> sigmoid or
 *    softmax -> expert bias added for SELECTION only -> top-k -> gather the
 *    UNBIASED scores -> divide by (sum + division_eps) -> times route_scale;
 *  - pooler + pre_expert_norm, routed experts, tail, unpooler: page
 *    "vllm.models.muse_spark.nvidia.specialized_decode.runtime.providers",
 *    MoEProvider docstring and RoutedMoE.run;
 *  - routed experts with unit weights, the router weight applied after the
 *    post-expert norm, summed over k: muse_moe_runner page,
 *    MuseSparkAiterExperts and MuseSparkTopKWeightAndReduce.apply;
 *  - FFN boundary: providers page, BoundaryProvider docstring.
 *
 * Rounding points (the storage dtypes the pages show): fp32 logits, scores
 * and selection scores, fp32 routing weights, bf16 h, bf16 MoE activations,
 * bf16 moe_out, fp32 stream, bf16 out. Readings where the pages are silent:
 * ties in the top-k go to the lower expert id; fused w13 rows [0, I) are the
 * gate and [I, 2I) the up rows; element 2j of a packed FP4 row sits in the
 * low nibble of byte j; RMSNorm is v / sqrt(mean(v^2) + eps) * w; the gated
 * add is stream + gate * post_ffn_norm(u); FP8 W8A8 requantizes h per token
 * and the activation per route with scale fp32(amax / 448); the W4A4 forms
 * round both expert inputs to the weights' FP4 format (MXFP4: scale
 * 2^(floor(log2 amax) - 2) per 32; NVFP4: e4m3 scale nearest fp32(amax / 6)
 * per 16; nearest e2m1 magnitude, ties to the even code).
 *
 * Built twice: single-threaded (the oracle) and with -fopenmp (the same
 * source, rows and routes spread over the host's cores; labelled as such
 * wherever it is timed). */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { Q_MXFP4 = 0, Q_NVFP4 = 1, Q_FP8 = 2, Q_BF16 = 3, Q_MXFP4_A4 = 4, Q_NVFP4_A4 = 5 };

typedef struct {
  int32_t rows, hidden, pooled, inter, experts, top_k;
  int32_t quant;       /* Q_* */
  int32_t softmax;     /* 0 sigmoid, 1 softmax */
  int32_t has_multiplier, has_division_eps, pre_norm;
  float route_scale, multiplier, division_eps;
  double norm_eps;
} oc_config;

typedef struct {
  const float *w_router, *expert_bias;            /* [E, H], [E] */
  const uint16_t *w_pool, *w_pre_norm;            /* bf16 [P, H], [P] */
  const uint8_t *w13, *w2;                        /* plain layouts, see below */
  const void *w13_scale, *w2_scale;               /* UE8M0 / e4m3 bytes, FP8 fp32 per row */
  const float *w13_gscale, *w2_gscale;            /* NVFP4 [E] */
  const uint16_t *w_post_norm, *w_unpool;         /* bf16 [P], [H, P] */
  const uint16_t *w_ffn_norm, *w_next_norm;       /* bf16 [H], [H] */
  float gate;
} oc_weights;

/* ---- number formats --------------------------------------------------- */
static double bf16_val(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}
static double round_f32(double v) { return (double)(float)v; }
/* nearest value with mant_bits fraction bits in the binade of v (never below
 * the binade 2^min_exp), ties to even */
static double round_minifloat(double v, int mant_bits, int min_exp) {
  if (v == 0.0 || !isfinite(v)) return v;
  int e;
  frexp(v, &e);
  int binade = e - 1;
  if (binade < min_exp) binade = min_exp;
  const double step = ldexp(1.0, binade - mant_bits);
  return nearbyint(v / step) * step;
}
static double round_bf16(double v) {
  const double r = round_minifloat(v, 7, -126);
  if (fabs(r) > 3.3895313892515355e38) return copysign(INFINITY, r);
  return r;
}
static uint16_t bf16_bits(double v) { /* v bf16-representable */
  const float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}
static const double E2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
static double e2m1_val(unsigned code) {
  const double m = E2M1[code & 7u];
  return (code & 8u) ? -m : m;
}
static double e4m3_val(unsigned c) { /* OCP float8 e4m3fn */
  const int ex = (c >> 3) & 0xF, m = c & 7;
  if ((c & 0x7F) == 0x7F) return NAN;
  const double v = ex == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, ex - 7);
  return (c & 0x80) ? -v : v;
}
/* e4m3 value nearest v: round to nearest even, saturating to +-448 */
static double e4m3_round(double v) {
  double r = round_minifloat(fabs(v), 3, -6);
  if (r > 448.0) r = 448.0;
  return copysign(r, v);
}
static double ue8m0_val(unsigned s) { return s == 255u ? NAN : ldexp(1.0, (int)s - 127); }
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* nearest e2m1 magnitude of a >= 0, ties to the even code (saturating at 6) */
static double e2m1_nearest(double a) {
  int best = 0;
  double bd = fabs(a - E2M1[0]);
  for (int c = 1; c < 8; ++c) {
    const double d = fabs(a - E2M1[c]);
    if (d < bd || (d == bd && (c & 1) == 0 && (best & 1))) {
      bd = d;
      best = c;
    }
  }
  return E2M1[best];
}

/* The W4A4 expert input: bf16-valued v [K] rounded in place to MXFP4 (fmt 1,
 * blocks of 32) or NVFP4 (fmt 2, blocks of 16), then decoded. */
static void fp4_round_row(double* v, int K, int fmt) {
  const int B = fmt == 1 ? 32 : 16;
  for (int b0 = 0; b0 < K; b0 += B) {
    double amax = 0.0;
    for (int i = 0; i < B; ++i)
      if (fabs(v[b0 + i]) > amax) amax = fabs(v[b0 + i]);
    if (fmt == 1) {
      int e = 0;
      if (amax > 0.0) {
        int ex;
        frexp(amax, &ex);
        e = ex - 1 - 2;
      }
      if (e < -126) e = -126;
      if (e > 127) e = 127;
      const double sc = ldexp(1.0, e);
      for (int i = 0; i < B; ++i) {
        const double x = v[b0 + i];
        v[b0 + i] = copysign(e2m1_nearest(fabs(x) / sc) * sc, x);
      }
    } else {
      const double sf = e4m3_round(round_f32(amax / 6.0));
      for (int i = 0; i < B; ++i) {
        const double x = v[b0 + i];
        double a = sf > 0.0 ? round_f32(fabs(x) / sf) : 0.0;
        if (a > 8.0) a = 8.0;
        v[b0 + i] = copysign(e2m1_nearest(a) * sf, x);
      }
    }
  }
}

/* FP8 W8A8: bf16-valued v [K] -> its e4m3 requantization times the row scale
 * fp32(amax / 448) (an all-zero row stays zero) */
static void fp8_round_row(double* v, int K) {
  double amax = 0.0;
  for (int i = 0; i < K; ++i)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  const double s = round_f32(amax / 448.0);
  for (int i = 0; i < K; ++i) v[i] = s > 0.0 ? e4m3_round(round_f32(v[i] / s)) * s : 0.0;
}

/* RMSNorm of v [n] with bf16 weight w (NULL: weightless), in place */
static void rms_norm(double* v, int n, const uint16_t* w, double eps) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += v[i] * v[i];
  const double r = sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) v[i] = v[i] / r * (w ? bf16_val(w[i]) : 1.0);
}

/* ---- expert weights ------------------------------------------------------ */
/* Row n of expert e's matrix (w13: N = 2I rows of K = P; w2: N = P rows of
 * K = I) dequantized exactly into out [K]. Plain layouts: FP4 codes
 * [E, N, K/2] (low nibble first), MXFP4 UE8M0 [E, N, K/32], NVFP4 e4m3
 * [E, N, K/16] and fp32 global [E]; FP8 e4m3 [E, N, K] and fp32 [E, N];
 * BF16 bf16 [E, N, K]. */
static void weight_row(int q, const uint8_t* codes, const void* scale, const float* gscale, int e,
                       int n, int N, int K, double* out) {
  if (q == Q_MXFP4_A4) q = Q_MXFP4;
  if (q == Q_NVFP4_A4) q = Q_NVFP4;
  if (q == Q_MXFP4 || q == Q_NVFP4) {
    const uint8_t* row = codes + ((size_t)e * N + n) * (K / 2);
    const uint8_t* sc = (const uint8_t*)scale + ((size_t)e * N + n) * (K / (q == Q_MXFP4 ? 32 : 16));
    const double g = q == Q_NVFP4 ? (double)gscale[e] : 1.0;
    for (int k = 0; k < K; ++k) {
      const unsigned c = (k & 1) ? (row[k / 2] >> 4) : (row[k / 2] & 0xF);
      const double s = q == Q_MXFP4 ? ue8m0_val(sc[k / 32]) : e4m3_val(sc[k / 16]);
      out[k] = e2m1_val(c) * s * g;
    }
  } else if (q == Q_FP8) {
    const uint8_t* row = codes + ((size_t)e * N + n) * K;
    const double s = (double)((const float*)scale)[(size_t)e * N + n];
    for (int k = 0; k < K; ++k) out[k] = e4m3_val(row[k]) * s;
  } else {
    const uint16_t* row = (const uint16_t*)codes + ((size_t)e * N + n) * K;
    for (int k = 0; k < K; ++k) out[k] = bf16_val(row[k]);
  }
}

/* ---- routing ------------------------------------------------------------- */
/* One row of the routing rule: logits [E] (fp32 values) -> ids [k] by
 * descending selection score (ties: lower id first), fp32 weights [k]. */
static void route_row(const oc_config* c, const float* bias, const double* logit, int32_t* ids,
                      float* weights, double* s, double* sel) {
  const int E = c->experts, k = c->top_k;
  for (int e = 0; e < E; ++e) {
    double g = logit[e];
    if (c->has_multiplier) g = round_f32(g * (double)c->multiplier);
    s[e] = g;
  }
  if (!c->softmax) {
    for (int e = 0; e < E; ++e) s[e] = round_f32(1.0 / (1.0 + exp(-s[e])));
  } else {
    double mx = s[0];
    for (int e = 1; e < E; ++e)
      if (s[e] > mx) mx = s[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) {
      s[e] = exp(s[e] - mx);
      z += s[e];
    }
    for (int e = 0; e < E; ++e) s[e] = round_f32(s[e] / z);
  }
  for (int e = 0; e < E; ++e) sel[e] = round_f32(s[e] + (double)bias[e]);
  for (int j = 0; j < k; ++j) {  /* k rounds of arg-max, the lower id on ties */
    int best = -1;
    for (int e = 0; e < E; ++e) {
      int taken = 0;
      for (int i = 0; i < j; ++i) taken |= ids[i] == e;
      if (!taken && (best < 0 || sel[e] > sel[best])) best = e;
    }
    ids[j] = best;
  }
  double denom = 0.0;
  for (int j = 0; j < k; ++j) denom += s[ids[j]];
  if (c->has_division_eps) denom += (double)c->division_eps;
  for (int j = 0; j < k; ++j)
    weights[j] = (float)(s[ids[j]] / denom * (double)c->route_scale);
}

/* Routing only: logits fp32 [rows, E] -> ids [rows, k], weights [rows, k]. */
int musemoe_oracle_route(const oc_config* c, const float* logits, const float* bias,
                         int32_t* ids, float* weights) {
  const int E = c->experts;
  double* buf = (double*)malloc(sizeof(double) * 3 * (size_t)E);
  if (!buf) return 1;
  for (int t = 0; t < c->rows; ++t) {
    for (int e = 0; e < E; ++e) buf[e] = (double)logits[(size_t)t * E + e];
    route_row(c, bias, buf, ids + (size_t)t * c->top_k, weights + (size_t)t * c->top_k, buf + E,
              buf + 2 * E);
  }
  free(buf);
  return 0;
}

/* ---- the block --------------------------------------------------------------
 * x bf16 [rows, H], stream_in fp32 [rows, H] -> ids int32 [rows, k], weights
 * fp32 [rows, k], h bf16 [rows, P], moe_out bf16 [rows, P], stream_out fp32
 * [rows, H], out bf16 [rows, H]. Returns 0, or 1 if memory ran out. */
int musemoe_oracle_block(const oc_config* c, const oc_weights* w, const uint16_t* x,
                         const float* stream_in, int32_t* ids, float* weights, uint16_t* h_out,
                         uint16_t* moe_out, float* stream_out, uint16_t* out) {
  const int b = c->rows, H = c->hidden, P = c->pooled, I = c->inter, E = c->experts, k = c->top_k;
  const int q = c->quant;
  const int act4 = q == Q_MXFP4_A4 ? 1 : q == Q_NVFP4_A4 ? 2 : 0;
  double* h = (double*)calloc((size_t)b * P, sizeof(double));     /* bf16 values */
  double* hin = (double*)calloc((size_t)b * P, sizeof(double));   /* the w13 input */
  double* y = (double*)calloc((size_t)b * k * P, sizeof(double)); /* route outputs */
  double* mo = (double*)calloc((size_t)b * P, sizeof(double));    /* moe_out values */
  if (!h || !hin || !y || !mo) {
    free(h), free(hin), free(y), free(mo);
    return 1;
  }
  int fail = 0;

  /* router and routing rule, pooler and pre-expert norm: per row */
#pragma omp parallel for schedule(dynamic) reduction(| : fail)
  for (int t = 0; t < b; ++t) {
    double* buf = (double*)malloc(sizeof(double) * ((size_t)3 * E + H));
    if (!buf) {
      fail = 1;
      continue;
    }
    double* xr = buf + 3 * E;
    for (int j = 0; j < H; ++j) xr[j] = bf16_val(x[(size_t)t * H + j]);
    for (int e = 0; e < E; ++e) {
      double a = 0.0;
      for (int j = 0; j < H; ++j) a += xr[j] * (double)w->w_router[(size_t)e * H + j];
      buf[e] = round_f32(a);
    }
    route_row(c, w->expert_bias, buf, ids + (size_t)t * k, weights + (size_t)t * k, buf + E,
              buf + 2 * E);
    double* hr = h + (size_t)t * P;
    for (int p = 0; p < P; ++p) {
      double a = 0.0;
      for (int j = 0; j < H; ++j) a += xr[j] * bf16_val(w->w_pool[(size_t)p * H + j]);
      hr[p] = a;
    }
    if (c->pre_norm) rms_norm(hr, P, w->w_pre_norm, (double)c->norm_eps);
    for (int p = 0; p < P; ++p) hr[p] = round_bf16(hr[p]);
    double* hi = hin + (size_t)t * P;
    memcpy(hi, hr, sizeof(double) * P);
    if (q == Q_FP8) fp8_round_row(hi, P);
    if (act4) fp4_round_row(hi, P, act4);
    free(buf);
  }

  /* routed experts: per route, unit router weight */
#pragma omp parallel for schedule(dynamic) reduction(| : fail)
  for (int r = 0; r < b * k; ++r) {
    const int t = r / k, e = ids[r];
    double* buf = (double*)malloc(sizeof(double) * ((size_t)2 * I + P + I));
    if (!buf) {
      fail = 1;
      continue;
    }
    double* gu = buf;          /* [2I] */
    double* row = buf + 2 * I; /* [max(P, I)] */
    const double* hi = hin + (size_t)t * P;
    for (int n = 0; n < 2 * I; ++n) {
      weight_row(q, w->w13, w->w13_scale, w->w13_gscale, e, n, 2 * I, P, row);
      double a = 0.0;
      for (int p = 0; p < P; ++p) a += row[p] * hi[p];
      gu[n] = a;
    }
    double* act = gu;  /* a = bf16(silu(gate) * up), into gu[0..I) */
    for (int i = 0; i < I; ++i) act[i] = round_bf16(silu(gu[i]) * gu[I + i]);
    if (q == Q_FP8) fp8_round_row(act, I);
    if (act4) fp4_round_row(act, I, act4);
    for (int p = 0; p < P; ++p) {
      weight_row(q, w->w2, w->w2_scale, w->w2_gscale, e, p, P, I, row);
      double a = 0.0;
      for (int i = 0; i < I; ++i) a += row[i] * act[i];
      y[(size_t)r * P + p] = a;
    }
    free(buf);
  }

  /* post-expert norm, router weight, sum over k; unpooler; FFN boundary */
#pragma omp parallel for schedule(dynamic) reduction(| : fail)
  for (int t = 0; t < b; ++t) {
    double* u = (double*)malloc(sizeof(double) * ((size_t)H + P));
    if (!u) {
      fail = 1;
      continue;
    }
    double* n = u + H;
    double* m = mo + (size_t)t * P;
    for (int j = 0; j < k; ++j) {
      memcpy(n, y + ((size_t)t * k + j) * P, sizeof(double) * P);
      rms_norm(n, P, w->w_post_norm, (double)c->norm_eps);
      const double wt = (double)weights[(size_t)t * k + j];
      for (int p = 0; p < P; ++p) m[p] += n[p] * wt;
    }
    for (int p = 0; p < P; ++p) m[p] = round_bf16(m[p]);
    for (int i = 0; i < H; ++i) {
      double a = 0.0;
      for (int p = 0; p < P; ++p) a += m[p] * bf16_val(w->w_unpool[(size_t)i * P + p]);
      u[i] = a;
    }
    rms_norm(u, H, w->w_ffn_norm, (double)c->norm_eps);
    double* s = (double*)malloc(sizeof(double) * (size_t)H);
    if (!s) {
      free(u);
      fail = 1;
      continue;
    }
    for (int i = 0; i < H; ++i)
      s[i] = round_f32((double)stream_in[(size_t)t * H + i] + (double)w->gate * u[i]);
    for (int i = 0; i < H; ++i) stream_out[(size_t)t * H + i] = (float)s[i];
    rms_norm(s, H, w->w_next_norm, (double)c->norm_eps);
    for (int i = 0; i < H; ++i) out[(size_t)t * H + i] = bf16_bits(round_bf16(s[i]));
    for (int p = 0; p < P; ++p) {
      h_out[(size_t)t * P + p] = bf16_bits(h[(size_t)t * P + p]);
      moe_out[(size_t)t * P + p] = bf16_bits(m[p]);
    }
    free(s);
    free(u);
  }
  free(h), free(hin), free(y), free(mo);
  return fail;
}

/* 1 if built with OpenMP (the all-cores build), else 0 */
int musemoe_oracle_threads(void) {
#ifdef _OPENMP
  return 1;
#else
  return 0;
#endif
}

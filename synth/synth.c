/*
 * Seeded synthetic inputs for the MuseSpark1x MoE decode block.
 *
 * This file only draws random bytes and numbers and stores them in the
 * storage formats of the block's tensors. It holds none of the block's
 * arithmetic, and both the CUDA path's tests and the oracle take their
 * inputs from it.
 *
 * Every value is a pure function of (seed, tensor id, element index): the
 * counter-based SplitMix64 generator (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) is evaluated at state
 * key + (i + 1) * golden_gamma, so any sub-range of a tensor can be
 * regenerated on its own and the bytes do not depend on generation order.
 *
 * Normals use the Box-Muller transform: uniforms 2j and 2j+1 give normals
 * 2j (cosine branch) and 2j+1 (sine branch). Fillers run on OpenMP threads;
 * every element is still a pure function of its index.
 * libm's log/cos/sqrt may differ in the last bit between machines; the tests
 * always generate the inputs and the expected values in the same process.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tensor) {
  return mix64(mix64(seed + GOLDEN_GAMMA) ^ (tensor * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * GOLDEN_GAMMA);
}

/* Uniform in [0, 1) with 53 random bits. */
static inline double uniform01(uint64_t key, uint64_t i) {
  return (double)(draw(key, i) >> 11) * 0x1.0p-53;
}

/* Standard normals 2j and 2j+1 from uniforms 2j and 2j+1 (Box-Muller: the
 * cosine branch gives the even element, the sine branch the odd one). */
static inline double normal01(uint64_t key, uint64_t i) {
  uint64_t j = i >> 1;
  double u1 = 1.0 - uniform01(key, 2 * j); /* (0, 1]: log never sees 0 */
  double u2 = uniform01(key, 2 * j + 1);
  double r = sqrt(-2.0 * log(u1)), t = 6.283185307179586476925 * u2;
  return (i & 1) ? r * sin(t) : r * cos(t);
}

/* Fills normals [start, start + n) of a stream, computing each Box-Muller
 * pair once. */
static void normals(uint64_t key, uint64_t start, uint64_t n, double *out) {
  for (uint64_t j = 0; j < n;) {
    uint64_t i = start + j;
    if ((i & 1) == 0 && j + 1 < n) {
      double u1 = 1.0 - uniform01(key, i), u2 = uniform01(key, i + 1);
      double r = sqrt(-2.0 * log(u1)), t = 6.283185307179586476925 * u2;
      out[j] = r * cos(t);
      out[j + 1] = r * sin(t);
      j += 2;
    } else {
      out[j] = normal01(key, i);
      j += 1;
    }
  }
}

#define CHUNK 4096

/* float -> bfloat16 bits, round to nearest even (NaN kept quiet). */
static inline uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
    return (uint16_t)((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* float -> OCP float8 e4m3fn code, round to nearest even, saturating to
 * +-448 (the format has no infinity). */
static uint8_t f32_to_e4m3_satfinite(float v) {
  uint8_t sign = (v < 0.0f || (v == 0.0f && signbit(v))) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;
  if (a < 0x1.0p-6) {                       /* subnormal range, step 2^-9 */
    double m = nearbyint(a * 512.0);        /* 0..8 */
    return sign | (uint8_t)m;               /* m == 8 is the code of 2^-6 */
  }
  int e;
  frexp(a, &e);                             /* a = f * 2^e, f in [0.5, 1) */
  int unb = e - 1;                          /* a in [2^unb, 2^(unb+1)) */
  double m = nearbyint(ldexp(a, 3 - unb));  /* 8..16 */
  if (m == 16.0) { unb += 1; m = 8.0; }
  int code = ((unb + 7) << 3) | ((int)m - 8);
  if (code > 0x7E) code = 0x7E;
  return sign | (uint8_t)code;
}

/* ---- exported fillers: element i of the tensor is out[i - start] ---- */

void synth_bytes(uint64_t seed, uint64_t tensor, uint8_t *out, uint64_t start,
                 uint64_t n) {
  uint64_t key = stream_key(seed, tensor);
#pragma omp parallel for schedule(static)
  for (uint64_t j = 0; j < n; ++j) {
    uint64_t i = start + j;
    out[j] = (uint8_t)(draw(key, i >> 3) >> (8 * (i & 7)));
  }
}

void synth_normal_f32(uint64_t seed, uint64_t tensor, float *out,
                      uint64_t start, uint64_t n, double mean, double std) {
  uint64_t key = stream_key(seed, tensor);
#pragma omp parallel for schedule(static)
  for (uint64_t c = 0; c < n; c += CHUNK) {
    double buf[CHUNK];
    uint64_t m = n - c < CHUNK ? n - c : CHUNK;
    normals(key, start + c, m, buf);
    for (uint64_t j = 0; j < m; ++j) out[c + j] = (float)(mean + std * buf[j]);
  }
}

void synth_normal_bf16(uint64_t seed, uint64_t tensor, uint16_t *out,
                       uint64_t start, uint64_t n, double mean, double std) {
  uint64_t key = stream_key(seed, tensor);
#pragma omp parallel for schedule(static)
  for (uint64_t c = 0; c < n; c += CHUNK) {
    double buf[CHUNK];
    uint64_t m = n - c < CHUNK ? n - c : CHUNK;
    normals(key, start + c, m, buf);
    for (uint64_t j = 0; j < m; ++j)
      out[c + j] = f32_to_bf16_bits((float)(mean + std * buf[j]));
  }
}

void synth_uniform_f32(uint64_t seed, uint64_t tensor, float *out,
                       uint64_t start, uint64_t n, double lo, double hi) {
  uint64_t key = stream_key(seed, tensor);
#pragma omp parallel for schedule(static)
  for (uint64_t j = 0; j < n; ++j)
    out[j] = (float)(lo + (hi - lo) * uniform01(key, start + j));
}

/* Integers uniform in [lo, hi], stored as (value + offset) in a byte. */
void synth_int_u8(uint64_t seed, uint64_t tensor, uint8_t *out, uint64_t start,
                  uint64_t n, int32_t lo, int32_t hi, int32_t offset) {
  uint64_t key = stream_key(seed, tensor);
  uint64_t span = (uint64_t)(hi - lo + 1);
#pragma omp parallel for schedule(static)
  for (uint64_t j = 0; j < n; ++j) {
    uint64_t r = (uint64_t)(uniform01(key, start + j) * (double)span);
    out[j] = (uint8_t)((int32_t)r + lo + offset);
  }
}

/* e4m3 codes of 2^u with u uniform in [lo, hi). */
void synth_e4m3_pow2(uint64_t seed, uint64_t tensor, uint8_t *out,
                     uint64_t start, uint64_t n, double lo, double hi) {
  uint64_t key = stream_key(seed, tensor);
#pragma omp parallel for schedule(static)
  for (uint64_t j = 0; j < n; ++j) {
    double u = lo + (hi - lo) * uniform01(key, start + j);
    out[j] = f32_to_e4m3_satfinite((float)exp2(u));
  }
}

/* A row-quantized fp8 weight: W ~ N(0, std) in fp32 per element, one fp32
 * scale per row = amax / 448 (fp32 division), codes = e4m3(W / scale). Rows
 * [row0, row0 + nrows) of a tensor whose rows have `cols` elements. */
void synth_fp8_rows(uint64_t seed, uint64_t tensor, uint8_t *codes,
                    float *scales, uint64_t row0, uint64_t nrows,
                    uint64_t cols, double std) {
  uint64_t key = stream_key(seed, tensor);
#pragma omp parallel
  {
    double *buf = (double *)malloc(cols * sizeof(double));
#pragma omp for schedule(static)
    for (uint64_t r = 0; r < nrows; ++r) {
      normals(key, (row0 + r) * cols, cols, buf);
      float amax = 0.0f;
      for (uint64_t c = 0; c < cols; ++c) {
        float w = (float)(std * buf[c]);
        if (fabsf(w) > amax) amax = fabsf(w);
      }
      float s = amax / 448.0f;
      scales[r] = s;
      for (uint64_t c = 0; c < cols; ++c) {
        float w = (float)(std * buf[c]);
        codes[r * cols + c] = s > 0.0f ? f32_to_e4m3_satfinite(w / s) : 0;
      }
    }
    free(buf);
  }
}

/* A permutation of 0..n-1 (Fisher-Yates driven by draws 0..n-2). */
void synth_permutation(uint64_t seed, uint64_t tensor, int32_t *out,
                       uint64_t n) {
  uint64_t key = stream_key(seed, tensor);
  for (uint64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (uint64_t i = n; i > 1; --i) {
    uint64_t j = (uint64_t)(uniform01(key, n - i) * (double)i);
    int32_t t = out[i - 1];
    out[i - 1] = out[j];
    out[j] = t;
  }
}

/*
 * gen.c -- seeded synthetic inputs for the PTQ1_0 tests and benchmark.
 *
 * This module holds random-number generation and storage-format rounding
 * only: no step of the ternary matmul, the rotation or the feed-forward block.
 * Both sides of every parity test (the CPU oracle and the CUDA library) are
 * fed the very arrays it writes.
 *
 * Generator: counter-based.  Value i of stream s under seed q is
 *   mix(key(q, s) + (i + 1) * G),  key(q, s) = mix(q * G + s + 1),
 * where mix is the splitmix64 output function (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014) and G is
 * 0x9E3779B97F4A7C15.  Because each value depends only on (q, s, i), the
 * loops below can run in any order and on any number of threads.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t key_of(uint64_t seed, uint64_t stream) {
  return mix(seed * GOLDEN + stream + 1);
}

static inline uint64_t draw(uint64_t key, uint64_t i) {
  return mix(key + (i + 1) * GOLDEN);
}

/* uniform double in (0, 1]: 53 random bits */
static inline double unit_open0(uint64_t h) {
  return ((double)(h >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}

/* uniform double in [0, 1) */
static inline double unit(uint64_t h) {
  return (double)(h >> 11) * (1.0 / 9007199254740992.0);
}

/* standard normal number i of the stream, Box-Muller from draws 2i, 2i+1 */
static inline double normal_at(uint64_t key, uint64_t i) {
  double u1 = unit_open0(draw(key, 2 * i));
  double u2 = unit(draw(key, 2 * i + 1));
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925 * u2);
}

/* IEEE binary16 bit pattern nearest to v (round to nearest, ties to even).
   Handles subnormal results and overflow to infinity. */
static uint16_t to_half_bits(double v) {
  uint16_t sign = 0;
  if (v < 0 || (v == 0 && signbit(v))) {
    sign = 0x8000;
    v = -v;
  }
  if (isnan(v)) return 0x7e00;
  if (v >= 65520.0) return sign | 0x7c00; /* rounds past the largest finite */
  if (v == 0) return sign;
  int e;
  (void)frexp(v, &e); /* v = m * 2^e, m in [0.5, 1) */
  /* unit in the last place: normal results have 11 significant bits,
     subnormal results are multiples of 2^-24 */
  int exp_unbiased = e - 1; /* v in [2^(e-1), 2^e) */
  int ulp_exp = exp_unbiased >= -14 ? exp_unbiased - 10 : -24;
  double q = ldexp(v, -ulp_exp); /* v / ulp, >= 0 */
  double r = nearbyint(q);       /* default rounding mode: ties to even */
  uint64_t mant = (uint64_t)r;   /* v ~= mant * 2^ulp_exp */
  if (ulp_exp == -24) {
    /* subnormal (mant < 1024) or rounded up to the smallest normal (1024) */
    return sign | (uint16_t)mant;
  }
  /* normal: mant in [1024, 2048]; 2048 carries into the exponent */
  int biased = exp_unbiased + 15;
  if (mant == 2048) {
    mant = 1024;
    biased += 1;
  }
  if (biased >= 31) return sign | 0x7c00;
  return sign | (uint16_t)(biased << 10) | (uint16_t)(mant - 1024);
}

/* bfloat16 bit pattern nearest to a float (ties to even) */
static uint16_t to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* ---- public entry points ------------------------------------------------ */

void syn_trits_uniform(uint64_t seed, uint64_t stream, int8_t* out, int64_t n) {
  uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t h = draw(key, (uint64_t)i);
    out[i] = (int8_t)((int)(((h >> 32) * 3u) >> 32) - 1);
  }
}

/* P(0) = p_zero, P(-1) = P(+1) = (1 - p_zero) / 2 */
void syn_trits_sparse(uint64_t seed, uint64_t stream, double p_zero, int8_t* out,
                      int64_t n) {
  uint64_t key = key_of(seed, stream);
  double p_neg = p_zero + 0.5 * (1.0 - p_zero);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double u = unit(draw(key, (uint64_t)i));
    out[i] = (int8_t)(u < p_zero ? 0 : (u < p_neg ? -1 : 1));
  }
}

void syn_signs(uint64_t seed, uint64_t stream, int8_t* out, int64_t n) {
  uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = (int8_t)((draw(key, (uint64_t)i) >> 63) ? 1 : -1);
}

void syn_normal_f64(uint64_t seed, uint64_t stream, double* out, int64_t n) {
  uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(key, (uint64_t)i);
}

void syn_normal_f32(uint64_t seed, uint64_t stream, float* out, int64_t n) {
  uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)normal_at(key, (uint64_t)i);
}

void syn_normal_bf16(uint64_t seed, uint64_t stream, uint16_t* out, int64_t n) {
  uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = to_bf16_bits((float)normal_at(key, (uint64_t)i));
}

/* fp16 bit patterns of sigma * |z|, z standard normal */
void syn_abs_normal_f16(uint64_t seed, uint64_t stream, double sigma, uint16_t* out,
                        int64_t n) {
  uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = to_half_bits(sigma * fabs(normal_at(key, (uint64_t)i)));
}

/* storage rounding helpers, exported so the tests can pin them */
/* token ids uniform over [0, V): draw mod V (the bias, below V / 2^64, is
   immaterial for a test input) */
void syn_token_ids(uint64_t seed, uint64_t stream, int64_t V, int32_t* out, int64_t n) {
  uint64_t key = key_of(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(draw(key, (uint64_t)i) % (uint64_t)V);
}

uint16_t syn_half_bits(double v) { return to_half_bits(v); }
uint16_t syn_bf16_bits(float f) { return to_bf16_bits(f); }

/*
 * ptq_oracle.c -- plain, slow, fp64 CPU oracle (TEST INFRASTRUCTURE ONLY).
 *
 * See ptq_oracle.h for the sources and the readings.  Every loop here follows
 * a definition directly; there is no blocking, fusion or reordering beyond
 * what the definition states.  The only parallelism is an OpenMP loop over
 * independent output rows, which does not change any result.
 */
#include "ptq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
  ORC_WEIGHTS_PER_BLOCK = 128, /* [P1] "What Bonsai is" */
  ORC_TRITS_PER_BYTE = 5,      /* [P1] "What Bonsai is" */
  ORC_BYTES_PER_BLOCK = 26,    /* ceil(128 / 5) */
  ORC_ROT = 1024,              /* [P1] "What Bonsai is": 1024-wide butterfly */
  ORC_PQ2_PER_BYTE = 4,        /* [P2] "Level 2": 2 bits per weight */
  ORC_PQ2_BYTES_PER_BLOCK = 32 /* 128 weights x 2 bits */
};

static int g_threads = 0; /* 0 = OpenMP default */

void orc_set_threads(int n) {
  g_threads = n;
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
  return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- exact storage decodes (IEEE-754 bit fields) ---------------------- */

double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

double orc_bf16_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int m = b & 0x7f;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -133); /* subnormal: m * 2^-133 */
  } else if (e == 255) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(m + 128), e - 134); /* (1 + m/128) * 2^(e-127) */
  }
  return sign ? -v : v;
}

void orc_decode_f16(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_half_to_double(in[i]);
}

void orc_decode_bf16(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_double(in[i]);
}

void orc_decode_f32(const float* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = (double)in[i];
}

/* ---- the base-3 codec -------------------------------------------------- */

static const double k_pow3[6] = {1.0, 3.0, 9.0, 27.0, 81.0, 243.0};

/* [P1] "What Ferrox does with it": digit n = floor(3^(n+1) u) - 3 floor(3^n u),
   u = byte / 256.  Every quantity is exact in double. */
int orc_peel_digit(uint8_t byte, int n) {
  double u = (double)byte / 256.0;
  return (int)(floor(k_pow3[n + 1] * u) - 3.0 * floor(k_pow3[n] * u));
}

/* Encode rule of the tiny PTQ1_0 matvec workload: digit = trit + 1,
   v = sum_i d_i 3^(4-i) over the byte's five positions (positions past the
   block's 128 weights carry digit 1), byte = ceil(256 v / 243). */
int orc_pack(const int8_t* trits, uint8_t* wq, int64_t N, int64_t K) {
  if (K % ORC_WEIGHTS_PER_BLOCK != 0 || N < 0) return -1;
  int64_t nb = K / ORC_WEIGHTS_PER_BLOCK;
  for (int64_t i = 0; i < N * K; ++i)
    if (trits[i] < -1 || trits[i] > 1) return -1;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const int8_t* t = trits + n * K + b * ORC_WEIGHTS_PER_BLOCK;
      uint8_t* out = wq + (n * nb + b) * ORC_BYTES_PER_BLOCK;
      for (int j = 0; j < ORC_BYTES_PER_BLOCK; ++j) {
        int v = 0;
        for (int i = 0; i < ORC_TRITS_PER_BYTE; ++i) {
          int pos = ORC_TRITS_PER_BYTE * j + i;
          int d = pos < ORC_WEIGHTS_PER_BLOCK ? t[pos] + 1 : 1;
          v = 3 * v + d; /* Horner form of sum_i d_i 3^(4-i) */
        }
        out[j] = (uint8_t)((256 * v + 242) / 243); /* integer ceil */
      }
    }
  }
  return 0;
}

int orc_unpack(const uint8_t* wq, int8_t* trits, int64_t N, int64_t K) {
  if (K % ORC_WEIGHTS_PER_BLOCK != 0 || N < 0) return -1;
  int64_t nb = K / ORC_WEIGHTS_PER_BLOCK;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* in = wq + (n * nb + b) * ORC_BYTES_PER_BLOCK;
      int8_t* t = trits + n * K + b * ORC_WEIGHTS_PER_BLOCK;
      for (int pos = 0; pos < ORC_WEIGHTS_PER_BLOCK; ++pos) {
        int j = pos / ORC_TRITS_PER_BYTE;
        int i = pos % ORC_TRITS_PER_BYTE;
        t[pos] = (int8_t)(orc_peel_digit(in[j], i) - 1);
      }
    }
  }
  return 0;
}

/* ---- PQ2_0: two bits per trit ------------------------------------------ */

/* [P2] "Why I Am Building Another Inference Engine", "Level 2: The short
   answer": each ternary weight in 2 bits plus one 16-bit scale per 128
   weights.  Readings: code = trit + 1; weight 4j + i of a block sits in
   byte j, bits 2i and 2i + 1; a block is 32 bytes; the decode is
   trit = code - 1 for all four codes (an encoder never writes code 3). */
int orc_pq2_pack(const int8_t* trits, uint8_t* wq, int64_t N, int64_t K) {
  if (K % ORC_WEIGHTS_PER_BLOCK != 0 || N < 0) return -1;
  for (int64_t i = 0; i < N * K; ++i)
    if (trits[i] < -1 || trits[i] > 1) return -1;
  for (int64_t i = 0; i < N * K / ORC_PQ2_PER_BYTE; ++i) {
    int v = 0;
    for (int k = 0; k < ORC_PQ2_PER_BYTE; ++k)
      v |= (trits[ORC_PQ2_PER_BYTE * i + k] + 1) << (2 * k);
    wq[i] = (uint8_t)v;
  }
  return 0;
}

int orc_pq2_unpack(const uint8_t* wq, int8_t* trits, int64_t N, int64_t K) {
  if (K % ORC_WEIGHTS_PER_BLOCK != 0 || N < 0) return -1;
  for (int64_t i = 0; i < N * K; ++i)
    trits[i] = (int8_t)(((wq[i / ORC_PQ2_PER_BYTE] >> (2 * (i % ORC_PQ2_PER_BYTE))) & 3) - 1);
  return 0;
}

/* ---- the signed Walsh-Hadamard rotation -------------------------------- */

static int popcount_u32(unsigned v) {
  int c = 0;
  while (v) {
    c += (int)(v & 1u);
    v >>= 1;
  }
  return c;
}

void orc_fwht_def(const double* x, const int8_t* signs, double* y, int64_t M,
                  int64_t K) {
  int64_t nblk = K / ORC_ROT;
#pragma omp parallel for schedule(static)
  for (int64_t mb = 0; mb < M * nblk; ++mb) {
    int64_t m = mb / nblk, b = mb % nblk;
    const double* xb = x + m * K + b * ORC_ROT;
    const int8_t* sb = signs + b * ORC_ROT;
    double* yb = y + m * K + b * ORC_ROT;
    for (int j = 0; j < ORC_ROT; ++j) {
      double acc = 0.0;
      for (int i = 0; i < ORC_ROT; ++i) {
        double h = (popcount_u32((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
        acc += h * (double)sb[i] * xb[i];
      }
      yb[j] = acc / 32.0;
    }
  }
}

void orc_fwht_fast(const double* x, const int8_t* signs, double* y, int64_t M,
                   int64_t K) {
  int64_t nblk = K / ORC_ROT;
#pragma omp parallel for schedule(static)
  for (int64_t mb = 0; mb < M * nblk; ++mb) {
    int64_t m = mb / nblk, b = mb % nblk;
    double v[ORC_ROT];
    const double* xb = x + m * K + b * ORC_ROT;
    const int8_t* sb = signs + b * ORC_ROT;
    for (int i = 0; i < ORC_ROT; ++i) v[i] = (double)sb[i] * xb[i];
    for (int h = 1; h < ORC_ROT; h <<= 1) {
      for (int i = 0; i < ORC_ROT; i += 2 * h) {
        for (int j = i; j < i + h; ++j) {
          double a = v[j], c = v[j + h];
          v[j] = a + c;
          v[j + h] = a - c;
        }
      }
    }
    double* yb = y + m * K + b * ORC_ROT;
    for (int i = 0; i < ORC_ROT; ++i) yb[i] = v[i] / 32.0;
  }
}

/* The inverse rotation.  R = H D_s / 32 with H symmetric and H H = 1024 I,
   so R is orthonormal and R^T = D_s H / 32: per block,
   x_i = (1/32) s_i sum_j (-1)^popcount(i&j) y_j.  The definition, O(1024^2)
   per block. */
void orc_unrotate_def(const double* y, const int8_t* signs, double* x,
                      int64_t M, int64_t K) {
  int64_t nblk = K / ORC_ROT;
#pragma omp parallel for schedule(static)
  for (int64_t mb = 0; mb < M * nblk; ++mb) {
    int64_t m = mb / nblk, b = mb % nblk;
    const double* yb = y + m * K + b * ORC_ROT;
    const int8_t* sb = signs + b * ORC_ROT;
    double* xb = x + m * K + b * ORC_ROT;
    for (int i = 0; i < ORC_ROT; ++i) {
      double acc = 0.0;
      for (int j = 0; j < ORC_ROT; ++j) {
        double h = (popcount_u32((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
        acc += h * yb[j];
      }
      xb[i] = (double)sb[i] * acc / 32.0;
    }
  }
}

/* ---- embedding lookup on a rotated table -------------------------------- */

/* [P1] "What Bonsai is": the rotation folded into the stored weights is
   undone on the embedding table after each lookup.  The stored row of token
   v is R e_v, so out[m] = R^T table[ids[m]].  A row whose id lies outside
   [0, V) is all NaN. */
void orc_embed(const double* table, const int32_t* ids, const int8_t* signs,
               double* out, int64_t M, int64_t V, int64_t H) {
  for (int64_t m = 0; m < M; ++m) {
    double* om = out + m * H;
    if (ids[m] < 0 || ids[m] >= V) {
      for (int64_t k = 0; k < H; ++k) om[k] = NAN;
      continue;
    }
    orc_unrotate_def(table + (int64_t)ids[m] * H, signs, om, 1, H);
  }
}

/* The same with a PTQ1_0 table: row v is t[v,k] * s[v, k/128], its trits
   peeled from wq.  Returns 0, or -1 on a bad shape or allocation failure. */
int orc_embed_ptq1(const uint8_t* wq, const uint16_t* scales,
                   const int32_t* ids, const int8_t* signs, double* out,
                   int64_t M, int64_t V, int64_t H) {
  if (H % ORC_ROT != 0 || M < 0 || V < 0) return -1;
  int64_t nb = H / ORC_WEIGHTS_PER_BLOCK;
  int8_t* t = (int8_t*)malloc((size_t)H);
  double* row = (double*)malloc(sizeof(double) * (size_t)H);
  if (!t || !row) {
    free(t);
    free(row);
    return -1;
  }
  for (int64_t m = 0; m < M; ++m) {
    double* om = out + m * H;
    if (ids[m] < 0 || ids[m] >= V) {
      for (int64_t k = 0; k < H; ++k) om[k] = NAN;
      continue;
    }
    int64_t v = ids[m];
    orc_unpack(wq + v * nb * ORC_BYTES_PER_BLOCK, t, 1, H);
    for (int64_t k = 0; k < H; ++k)
      row[k] = (double)t[k] *
               orc_half_to_double(scales[v * nb + k / ORC_WEIGHTS_PER_BLOCK]);
    orc_unrotate_def(row, signs, om, 1, H);
  }
  free(t);
  free(row);
  return 0;
}

/* ---- the block-scaled ternary matmul ------------------------------------ */

/* One output row n for all M activation rows: decode the row's trits (PTQ1_0
   or PQ2_0), then y[m] = sum_b s_b * (sum_i t_i x_i). */
static void matmul_row(const uint8_t* wq, const uint16_t* scales,
                       const double* x, double* out, int64_t out_stride,
                       int64_t M, int64_t n, int64_t K, int8_t* trow, int pq2) {
  int64_t nb = K / ORC_WEIGHTS_PER_BLOCK;
  if (pq2)
    orc_pq2_unpack(wq + n * nb * ORC_PQ2_BYTES_PER_BLOCK, trow, 1, K);
  else
    orc_unpack(wq + n * nb * ORC_BYTES_PER_BLOCK, trow, 1, K);
  for (int64_t m = 0; m < M; ++m) {
    const double* xm = x + m * K;
    double y = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
      double s = orc_half_to_double(scales[n * nb + b]);
      double dot = 0.0;
      for (int i = 0; i < ORC_WEIGHTS_PER_BLOCK; ++i) {
        int64_t k = b * ORC_WEIGHTS_PER_BLOCK + i;
        dot += (double)trow[k] * xm[k];
      }
      y += s * dot;
    }
    out[m * out_stride] = y;
  }
}

static void matmul_fmt(const uint8_t* wq, const uint16_t* scales,
                       const double* x, double* y, int64_t M, int64_t N,
                       int64_t K, int pq2) {
#pragma omp parallel
  {
    int8_t* trow = (int8_t*)malloc((size_t)K);
#pragma omp for schedule(static)
    for (int64_t n = 0; n < N; ++n)
      matmul_row(wq, scales, x, y + n, N, M, n, K, trow, pq2);
    free(trow);
  }
}

static void matmul_rows_fmt(const uint8_t* wq, const uint16_t* scales,
                            const double* x, double* y, int64_t M, int64_t K,
                            const int64_t* rows, int64_t nrows, int pq2) {
#pragma omp parallel
  {
    int8_t* trow = (int8_t*)malloc((size_t)K);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < nrows; ++r)
      matmul_row(wq, scales, x, y + r, nrows, M, rows[r], K, trow, pq2);
    free(trow);
  }
}

void orc_matmul(const uint8_t* wq, const uint16_t* scales, const double* x,
                double* y, int64_t M, int64_t N, int64_t K) {
  matmul_fmt(wq, scales, x, y, M, N, K, 0);
}

void orc_matmul_rows(const uint8_t* wq, const uint16_t* scales,
                     const double* x, double* y, int64_t M, int64_t N,
                     int64_t K, const int64_t* rows, int64_t nrows) {
  (void)N;
  matmul_rows_fmt(wq, scales, x, y, M, K, rows, nrows, 0);
}

void orc_pq2_matmul(const uint8_t* wq, const uint16_t* scales, const double* x,
                    double* y, int64_t M, int64_t N, int64_t K) {
  matmul_fmt(wq, scales, x, y, M, N, K, 1);
}

void orc_pq2_matmul_rows(const uint8_t* wq, const uint16_t* scales,
                         const double* x, double* y, int64_t M, int64_t N,
                         int64_t K, const int64_t* rows, int64_t nrows) {
  (void)N;
  matmul_rows_fmt(wq, scales, x, y, M, K, rows, nrows, 1);
}

/* ---- SwiGLU and the feed-forward block ---------------------------------- */

void orc_swiglu(const double* g, const double* u, double* h, int64_t n) {
  for (int64_t i = 0; i < n; ++i) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

int orc_ffn(const uint8_t* wgu_q, const uint16_t* wgu_s, const uint8_t* wd_q,
            const uint16_t* wd_s, const int8_t* signs_in,
            const int8_t* signs_mid, const double* x, double* y, int64_t M,
            int64_t H, int64_t I) {
  if (H % ORC_ROT != 0 || I % ORC_ROT != 0 || M < 0) return -1;
  double* xr = (double*)malloc(sizeof(double) * (size_t)(M * H));
  double* gu = (double*)malloc(sizeof(double) * (size_t)(M * 2 * I));
  double* h = (double*)malloc(sizeof(double) * (size_t)(M * I));
  if (!xr || !gu || !h) {
    free(xr);
    free(gu);
    free(h);
    return -1;
  }
  orc_fwht_fast(x, signs_in, xr, M, H);             /* rotate */
  orc_matmul(wgu_q, wgu_s, xr, gu, M, 2 * I, H);   /* gate and up */
  for (int64_t m = 0; m < M; ++m)                   /* SwiGLU */
    orc_swiglu(gu + m * 2 * I, gu + m * 2 * I + I, h + m * I, I);
  orc_fwht_fast(h, signs_mid, h, M, I);             /* rotate */
  orc_matmul(wd_q, wd_s, h, y, M, H, I);            /* down */
  free(xr);
  free(gu);
  free(h);
  return 0;
}

/* ---- the chained feed-forward stack ----------------------------------- */

/* [P1] "Speed, and where it goes": the next step named there is to run a
   whole layer on the device, the norms and the residual adds included.
   Reading: a pre-norm residual stack, for l = 0..L-1
     xn = x / sqrt(mean(x^2) + eps) * g_l,   x = x + FFN_l(xn),
   with FFN_l the block of orc_ffn.  wgu_q[l] etc. are per-layer arrays;
   x (M x H) is updated in place.  Returns 0 or -1. */
int orc_ffn_stack(const uint8_t* const* wgu_q, const uint16_t* const* wgu_s,
                  const uint8_t* const* wd_q, const uint16_t* const* wd_s,
                  const int8_t* const* signs_in, const int8_t* const* signs_mid,
                  const double* const* norm_w, int64_t L, double eps, double* x,
                  int64_t M, int64_t H, int64_t I) {
  if (H % ORC_ROT != 0 || I % ORC_ROT != 0 || M < 0 || L < 0) return -1;
  double* xn = (double*)malloc(sizeof(double) * (size_t)(M * H));
  double* y = (double*)malloc(sizeof(double) * (size_t)(M * H));
  if (!xn || !y) {
    free(xn);
    free(y);
    return -1;
  }
  int rc = 0;
  for (int64_t l = 0; l < L && rc == 0; ++l) {
    for (int64_t m = 0; m < M; ++m) {
      const double* xm = x + m * H;
      double ss = 0.0;
      for (int64_t k = 0; k < H; ++k) ss += xm[k] * xm[k];
      const double inv = 1.0 / sqrt(ss / (double)H + eps);
      for (int64_t k = 0; k < H; ++k) xn[m * H + k] = xm[k] * inv * norm_w[l][k];
    }
    rc = orc_ffn(wgu_q[l], wgu_s[l], wd_q[l], wd_s[l], signs_in[l], signs_mid[l], xn, y, M,
                 H, I);
    for (int64_t i = 0; i < M * H && rc == 0; ++i) x[i] += y[i];
  }
  free(xn);
  free(y);
  return rc;
}


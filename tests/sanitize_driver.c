/* sanitize_driver.c -- every entry point of the CPU oracle (and of the
 * seeded input generator that feeds it) on small inputs, for a build with
 * AddressSanitizer and UndefinedBehaviorSanitizer.  Test infrastructure: it
 * checks memory and arithmetic safety of the oracle's C, not its values
 * (the pins in test_oracle_pins.py do that); a few round trips are checked
 * so that a run that silently skipped work fails too.  Exit status 0 when
 * everything ran and the round trips hold. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../oracle/ptq_oracle.h"

/* the generator's entry points (synth/gen.c) */
void syn_trits_uniform(uint64_t seed, uint64_t stream, int8_t* out, int64_t n);
void syn_trits_sparse(uint64_t seed, uint64_t stream, double p_zero, int8_t* out, int64_t n);
void syn_signs(uint64_t seed, uint64_t stream, int8_t* out, int64_t n);
void syn_normal_f64(uint64_t seed, uint64_t stream, double* out, int64_t n);
void syn_normal_f32(uint64_t seed, uint64_t stream, float* out, int64_t n);
void syn_normal_bf16(uint64_t seed, uint64_t stream, uint16_t* out, int64_t n);
void syn_abs_normal_f16(uint64_t seed, uint64_t stream, double sigma, uint16_t* out, int64_t n);
void syn_token_ids(uint64_t seed, uint64_t stream, int64_t V, int32_t* out, int64_t n);
uint16_t syn_half_bits(double v);
uint16_t syn_bf16_bits(float f);

static int failures = 0;
#define CHECK(c)                                                    \
  do {                                                              \
    if (!(c)) {                                                     \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
      ++failures;                                                   \
    }                                                               \
  } while (0)

static void* must(size_t n) {
  void* p = calloc(n ? n : 1, 1);
  if (!p) {
    fprintf(stderr, "out of memory\n");
    exit(2);
  }
  return p;
}

int main(void) {
  enum { N = 8, K = 2048, M = 3, H = 1024, I = 1024, L = 2, V = 5 };
  const int64_t nblk = K / 128;

  /* number decoding, every pattern */
  uint16_t* pat = must(65536 * sizeof(uint16_t));
  double* dec = must(65536 * sizeof(double));
  for (int i = 0; i < 65536; ++i) pat[i] = (uint16_t)i;
  orc_decode_f16(pat, dec, 65536);
  orc_decode_bf16(pat, dec, 65536);
  CHECK(orc_half_to_double(0x3c00) == 1.0 && orc_bf16_to_double(0x3f80) == 1.0);
  float f32[4] = {1.0f, -2.5f, 0.0f, 3.0e-39f};
  double f64[4];
  orc_decode_f32(f32, f64, 4);
  CHECK(f64[1] == -2.5);
  for (int b = 0; b < 256; ++b)
    for (int n = 0; n < 5; ++n) CHECK(orc_peel_digit((uint8_t)b, n) >= 0);

  /* PTQ1_0 and PQ2_0 codecs: round trips */
  int8_t* t = must(N * K);
  int8_t* t2 = must(N * K);
  uint8_t* wq = must(N * nblk * 26);
  uint8_t* wq2 = must(N * nblk * 32);
  syn_trits_uniform(1, 0, t, N * K);
  CHECK(orc_pack(t, wq, N, K) == 0);
  CHECK(orc_unpack(wq, t2, N, K) == 0);
  CHECK(memcmp(t, t2, N * K) == 0);
  syn_trits_sparse(1, 1, 0.4, t, N * K);
  CHECK(orc_pq2_pack(t, wq2, N, K) == 0);
  CHECK(orc_pq2_unpack(wq2, t2, N, K) == 0);
  CHECK(memcmp(t, t2, N * K) == 0);
  CHECK(orc_pack(t, wq, N, 100) != 0); /* K % 128 refused */

  /* rotation: definition, butterfly (also in place), inverse */
  double* x = must(M * K * sizeof(double));
  double* y = must(M * K * sizeof(double));
  double* z = must(M * K * sizeof(double));
  int8_t* s = must(K);
  syn_normal_f64(2, 0, x, M * K);
  syn_signs(2, 1, s, K);
  orc_fwht_def(x, s, y, M, K);
  orc_fwht_fast(x, s, z, M, K);
  for (int i = 0; i < M * K; ++i) CHECK(fabs(y[i] - z[i]) < 1e-9);
  orc_fwht_fast(z, s, z, M, K);
  orc_unrotate_def(y, s, z, M, K);
  for (int i = 0; i < M * K; ++i) CHECK(fabs(z[i] - x[i]) < 1e-9);

  /* matmul, all rows and listed rows, both formats */
  uint16_t* sc = must(N * nblk * sizeof(uint16_t));
  syn_abs_normal_f16(3, 0, 0.02, sc, N * nblk);
  double* out = must(M * N * sizeof(double));
  double* part = must(M * N * sizeof(double));
  const int64_t rows[3] = {0, 5, 7};
  orc_matmul(wq, sc, x, out, M, N, K);
  orc_matmul_rows(wq, sc, x, part, M, N, K, rows, 3);
  for (int m = 0; m < M; ++m)
    for (int r = 0; r < 3; ++r) CHECK(part[m * 3 + r] == out[m * N + rows[r]]);
  orc_pq2_matmul(wq2, sc, x, out, M, N, K);
  orc_pq2_matmul_rows(wq2, sc, x, part, M, N, K, rows, 3);
  for (int m = 0; m < M; ++m)
    for (int r = 0; r < 3; ++r) CHECK(part[m * 3 + r] == out[m * N + rows[r]]);

  /* embedding lookups, one id out of range */
  double* table = must(V * H * sizeof(double));
  int32_t ids[4];
  syn_normal_f64(4, 0, table, V * H);
  syn_token_ids(4, 1, V, ids, 3);
  ids[3] = V;
  int8_t* se = must(H);
  syn_signs(4, 2, se, H);
  double* emb = must(4 * H * sizeof(double));
  orc_embed(table, ids, se, emb, 4, V, H);
  CHECK(isnan(emb[3 * H]));
  int8_t* te = must(V * H);
  uint8_t* qe = must(V * (H / 128) * 26);
  uint16_t* se16 = must(V * (H / 128) * sizeof(uint16_t));
  syn_trits_uniform(4, 3, te, V * H);
  CHECK(orc_pack(te, qe, V, H) == 0);
  syn_abs_normal_f16(4, 4, 0.02, se16, V * (H / 128));
  CHECK(orc_embed_ptq1(qe, se16, ids, se, emb, 4, V, H) == 0);

  /* SwiGLU, one block, a two-layer stack */
  double g[4] = {-3.0, 0.0, 1.0, 20.0}, u[4] = {1.0, 2.0, 3.0, 4.0}, hh[4];
  orc_swiglu(g, u, hh, 4);
  CHECK(hh[1] == 0.0);
  uint8_t *gq[L], *dq[L];
  uint16_t *gs[L], *ds[L];
  int8_t *si[L], *sm[L];
  double* nw[L];
  int8_t* tg = must((size_t)2 * I * H);
  int8_t* td = must((size_t)H * I);
  for (int l = 0; l < L; ++l) {
    gq[l] = must((size_t)2 * I * (H / 128) * 26);
    dq[l] = must((size_t)H * (I / 128) * 26);
    gs[l] = must((size_t)2 * I * (H / 128) * sizeof(uint16_t));
    ds[l] = must((size_t)H * (I / 128) * sizeof(uint16_t));
    si[l] = must(H);
    sm[l] = must(I);
    nw[l] = must(H * sizeof(double));
    syn_trits_uniform(5, 16 * l, tg, (int64_t)2 * I * H);
    syn_trits_uniform(5, 16 * l + 1, td, (int64_t)H * I);
    CHECK(orc_pack(tg, gq[l], 2 * I, H) == 0);
    CHECK(orc_pack(td, dq[l], H, I) == 0);
    syn_abs_normal_f16(5, 16 * l + 2, 0.02, gs[l], (int64_t)2 * I * (H / 128));
    syn_abs_normal_f16(5, 16 * l + 3, 0.02, ds[l], (int64_t)H * (I / 128));
    syn_signs(5, 16 * l + 4, si[l], H);
    syn_signs(5, 16 * l + 5, sm[l], I);
    for (int k = 0; k < H; ++k) nw[l][k] = 1.0;
  }
  double* xs = must(M * H * sizeof(double));
  double* ys = must(M * H * sizeof(double));
  syn_normal_f64(6, 0, xs, M * H);
  CHECK(orc_ffn(gq[0], gs[0], dq[0], ds[0], si[0], sm[0], xs, ys, M, H, I) == 0);
  for (int threads = 1; threads <= 2; ++threads) {
    orc_set_threads(threads);
    CHECK(orc_get_threads() == threads);
    CHECK(orc_ffn_stack((const uint8_t* const*)gq, (const uint16_t* const*)gs,
                        (const uint8_t* const*)dq, (const uint16_t* const*)ds,
                        (const int8_t* const*)si, (const int8_t* const*)sm,
                        (const double* const*)nw, L, 1e-6, xs, M, H, I) == 0);
  }
  CHECK(orc_ffn_stack(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 1e-6, xs, M, H, I) == 0);

  /* the generator's remaining outputs */
  float xf[64];
  uint16_t xb[64];
  syn_normal_f32(7, 0, xf, 64);
  syn_normal_bf16(7, 1, xb, 64);
  CHECK(syn_half_bits(1.0) == 0x3c00 && syn_bf16_bits(1.0f) == 0x3f80);

  for (int l = 0; l < L; ++l) {
    free(gq[l]); free(dq[l]); free(gs[l]); free(ds[l]); free(si[l]); free(sm[l]); free(nw[l]);
  }
  free(pat); free(dec); free(t); free(t2); free(wq); free(wq2); free(x); free(y); free(z);
  free(s); free(sc); free(out); free(part); free(table); free(se); free(emb); free(te);
  free(qe); free(se16); free(tg); free(td); free(xs); free(ys);
  if (failures) fprintf(stderr, "%d checks failed\n", failures);
  else printf("sanitized oracle run: ok\n");
  return failures ? 1 : 0;
}

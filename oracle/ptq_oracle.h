/*
 * ptq_oracle.h -- CPU oracle for the PTQ1_0 ternary matmul and the signed
 * 1024-wide Walsh-Hadamard rotation.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this library.
 * It shares no code, header, table or helper with the CUDA library: it is
 * written from the definitions on the source pages, in plain C, in fp64.
 *
 * Sources (page title, section):
 *   [P1] "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally"
 *        - "What Bonsai is": weights in {-1,0,+1}, one 16-bit scale per 128
 *          weights, five trits per byte in base 3 (1.75 bits/weight); every
 *          weight matrix is multiplied by a 1024-wide Walsh-Hadamard
 *          butterfly with a sign pattern, so the same rotation must be
 *          applied to the activation before every matmul.
 *        - "What Ferrox does with it": trit n of a byte is
 *          floor(3^(n+1) u) - 3 floor(3^n u) with u = byte/256.
 *        - "Speed, and where it goes": the feed-forward block is rotate,
 *          gate (+ up), SwiGLU, rotate, down.
 *   [P2] "Why I Am Building Another Inference Engine"
 *        - "Level 2: The short answer": PQ2_0 stores each ternary weight in
 *          2 bits plus one 16-bit scale per 128 weights (2.125 bits/weight).
 *   The encode rule (digit = trit + 1, v = sum d_i 3^(4-i),
 *   byte = ceil(256 v / 243), last byte of a block holds 3 trits padded with
 *   digit 1) is the workload definition of the tiny PTQ1_0 matvec case.
 *
 * Readings where the pages are silent:
 *   - trit order inside a block is contiguous: byte j, digit n <-> weight
 *     5j+n, n = 0 is the most significant base-3 digit;
 *   - the rotation flips signs first, then applies the Sylvester-ordered
 *     Hadamard matrix H[i][j] = (-1)^popcount(i & j), then scales by 1/32;
 *     the sign vector has one entry per element (block b uses its own 1024);
 *   - the gate/up weight of the fused feed-forward block stacks the gate rows
 *     (0..I-1) above the up rows (I..2I-1); h = silu(gate) * up;
 *   - PQ2_0: code = trit + 1; weight 4j + i of a block is bits 2i, 2i + 1
 *     of byte j; 32 bytes per block; decode trit = code - 1 for all four
 *     codes (no encoder writes code 3);
 *   - the embedding table is stored rotated like the weights (row v holds
 *     R e_v), so a lookup returns R^T of the stored row; an id outside the
 *     table gives a row of NaN.
 *
 * Storage (the same on both sides of the parity tests):
 *   wq     : N x (K/128) x 26 bytes, row-major (row n is (K/128)*26 bytes)
 *   scales : N x (K/128) IEEE binary16 bit patterns
 *   signs  : K int8 values, each +1 or -1
 */
#ifndef PTQ_ORACLE_H
#define PTQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Threads used by the parallel loops (over independent output rows). */
void orc_set_threads(int n);
int orc_get_threads(void);

/* Exact decodes of the storage formats into double. */
double orc_half_to_double(uint16_t h);
double orc_bf16_to_double(uint16_t b);
void orc_decode_f16(const uint16_t* in, double* out, int64_t n);
void orc_decode_bf16(const uint16_t* in, double* out, int64_t n);
void orc_decode_f32(const float* in, double* out, int64_t n);

/* The peel of [P1] "What Ferrox does with it", evaluated in double.
   Returns the base-3 digit n (0..4, 0 = most significant) of `byte`. */
int orc_peel_digit(uint8_t byte, int n);

/* Encode N x K trits (int8 in {-1,0,1}) into PTQ1_0 bytes.
   Returns 0, or -1 if a trit is outside {-1,0,1} or K % 128 != 0. */
int orc_pack(const int8_t* trits, uint8_t* wq, int64_t N, int64_t K);

/* Decode PTQ1_0 bytes back into trits with orc_peel_digit.
   Returns 0, or -1 if K % 128 != 0. */
int orc_unpack(const uint8_t* wq, int8_t* trits, int64_t N, int64_t K);

/* PQ2_0 codec: N x K trits <-> N x (K/128) x 32 bytes.  Return 0, or -1 on
   a trit outside {-1,0,1} (pack) or K % 128 != 0. */
int orc_pq2_pack(const int8_t* trits, uint8_t* wq, int64_t N, int64_t K);
int orc_pq2_unpack(const uint8_t* wq, int8_t* trits, int64_t N, int64_t K);

/* Signed rotation, the definition: for every row m and 1024-block b,
   y_j = (1/32) sum_i (-1)^popcount(i&j) s_i x_i.  O(1024^2) per block.
   x and y are M x K row-major; y may not alias x. */
void orc_fwht_def(const double* x, const int8_t* signs, double* y,
                  int64_t M, int64_t K);

/* The same transform by the radix-2 butterfly (10 stages), for speed.
   y may alias x. */
void orc_fwht_fast(const double* x, const int8_t* signs, double* y,
                   int64_t M, int64_t K);

/* The inverse rotation R^T = D_s H / 32 (R is orthonormal), the definition:
   per 1024-block, x_i = (1/32) s_i sum_j (-1)^popcount(i&j) y_j.
   O(1024^2) per block; x may not alias y. */
void orc_unrotate_def(const double* y, const int8_t* signs, double* x,
                      int64_t M, int64_t K);

/* Embedding lookup on a rotated table ([P1] "What Bonsai is": the rotation
   is undone on the embedding row after each lookup):
   out[m] = R^T table[ids[m]], table V x H, out M x H.  Rows with an id
   outside [0, V) are NaN. */
void orc_embed(const double* table, const int32_t* ids, const int8_t* signs,
               double* out, int64_t M, int64_t V, int64_t H);

/* The same for a PTQ1_0 table (wq V x (H/128) x 26, scales V x H/128): the
   row is the peeled trits times their block scales.  Returns 0 or -1. */
int orc_embed_ptq1(const uint8_t* wq, const uint16_t* scales,
                   const int32_t* ids, const int8_t* signs, double* out,
                   int64_t M, int64_t V, int64_t H);

/* y[m,n] = sum_b s[n,b] * sum_{i<128} t[n,128b+i] * x[m,128b+i], where the
   trits are peeled from wq.  x is M x K, y is M x N, both row-major. */
void orc_matmul(const uint8_t* wq, const uint16_t* scales, const double* x,
                double* y, int64_t M, int64_t N, int64_t K);

/* The same, for the listed output rows only: y is M x nrows, column r holds
   output row rows[r]. */
void orc_matmul_rows(const uint8_t* wq, const uint16_t* scales,
                     const double* x, double* y, int64_t M, int64_t N,
                     int64_t K, const int64_t* rows, int64_t nrows);

/* The block-scaled ternary matmul over PQ2_0 weights (the same definition,
   trits decoded from 2-bit codes), and the same for listed rows. */
void orc_pq2_matmul(const uint8_t* wq, const uint16_t* scales, const double* x,
                    double* y, int64_t M, int64_t N, int64_t K);
void orc_pq2_matmul_rows(const uint8_t* wq, const uint16_t* scales,
                         const double* x, double* y, int64_t M, int64_t N,
                         int64_t K, const int64_t* rows, int64_t nrows);

/* h = silu(g) * u, silu(a) = a / (1 + exp(-a)). */
void orc_swiglu(const double* g, const double* u, double* h, int64_t n);

/* Feed-forward block of [P1] "Speed, and where it goes":
   xr = R_in x; [g;u] = W_gu xr; h = silu(g) * u; hr = R_mid h; y = W_d hr.
   x: M x H, y: M x H, W_gu: 2I x H (gate rows then up rows), W_d: H x I.
   Everything in double, no intermediate rounding.  Returns 0 or -1 (shape or
   allocation failure). */
int orc_ffn(const uint8_t* wgu_q, const uint16_t* wgu_s, const uint8_t* wd_q,
            const uint16_t* wd_s, const int8_t* signs_in,
            const int8_t* signs_mid, const double* x, double* y, int64_t M,
            int64_t H, int64_t I);

/* A chained stack of L feed-forward blocks, pre-norm with residual adds
   (a reading of the next step [P1] "Speed, and where it goes" names):
     xn = x / sqrt(mean(x^2) + eps) * g_l;  x = x + FFN_l(xn),  l = 0..L-1.
   Per-layer arguments are arrays of L pointers; x (M x H) is updated in
   place, in double.  Returns 0 or -1. */
int orc_ffn_stack(const uint8_t* const* wgu_q, const uint16_t* const* wgu_s,
                  const uint8_t* const* wd_q, const uint16_t* const* wd_s,
                  const int8_t* const* signs_in, const int8_t* const* signs_mid,
                  const double* const* norm_w, int64_t L, double eps, double* x,
                  int64_t M, int64_t H, int64_t I);

#ifdef __cplusplus
}
#endif

#endif /* PTQ_ORACLE_H */

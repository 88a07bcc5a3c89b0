// k_gemm_tc.cu -- prefill GEMM over PTQ1_0 weights on the 5th-generation
// tensor cores (tcgen05, accumulator in TMEM).
//
//   y[m, n] = sum_b s[n, b] * sum_{i<128} t[n, 128b + i] * x[m, 128b + i]
//
// "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally", section "What
// Ferrox does with it": prefill runs a GEMM over the same packed blocks the
// decode matvec reads; the trits are peeled as floor(3^(n+1) u) - 3 floor(3^n
// u), u = byte / 256.
//
// Operands.  A = activations (16-bit, M x K), read by the MMA straight from
// the TMA-staged tile; B = the weight tile expanded in shared memory to t * s
// in A's type (kind::f16 takes A and B of one type), so the block scale is
// folded into B and the MMA (fp32 accumulation in TMEM) needs no per-block
// epilogue.  bf16 activations give bf16 tiles t * bf16(s) -- the expansion to
// bf16 tiles the decode/prefill split calls for; the scale's rounding to
// bf16 is at most 2^-9 relative.  fp16 activations (the feed-forward block's
// rotated operands) give exact fp16 tiles.
//
// Tile: 256 (M) x 128 (N): two 128-row accumulators in TMEM (256 columns)
// share every expanded B slice, so each weight is peeled once per 256
// activation rows.  K is consumed in 64-wide slices (one 128-byte swizzle atom
// of 16-bit values) through a 2-deep ring of A and B slices.  The CTA holds
// about 98 KB of shared memory, so two CTAs share an SM: the MMAs of one
// cover the load and expansion latency of the other.  Warp roles (10 warps):
//   warp 0      TMA producer of the A slices (box 64 x 256, 128B swizzle).
//   warp 1      TMEM allocation; lane 0 issues tcgen05.mma (8 per slice).
//   warps 2-9   expansion: thread (row r, half h) peels the 64 weights of half
//               h of every 128-weight block of row r in registers (two bytes
//               per integer multiply, see expand_half), reading the packed
//               row with 16-byte loads kept two blocks ahead; every pair of
//               16-bit outputs is one permute of the per-block bytes
//               {-s, 0, +s}.  Writes use the canonical K-major 128B-swizzled
//               layout; afterwards these warps run the epilogue
//               (TMEM -> registers -> y).
// The weights do not depend on the previous kernel in the stream, so the
// expansion starts before griddepcontrol.wait; the A loads and the output
// stores wait for it.  Every mbarrier wait is bounded; a wait that runs out
// raises the device status word, the CTA drains what it has in flight
// (bounded) and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "async_util.cuh"
#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int BM = 256, BN = 128, BK = 64, UM = 128;   // UM: rows per MMA
constexpr int kBSlice = BN * BK * 2;                        // 16 KB
constexpr int kExpWarp0 = 2;  // warps 0, 1: A producer, MMA issuer; then the expansion

// Shared memory layout (offsets from a 1024-aligned base) and warps of the
// two variants.  Large M: 256-row A slices, a 2-deep ring, 98 KB, 8
// expansion warps (two CTAs per SM).  Small M (M <= 128, one accumulator,
// for shapes that run unsplit in one wave): 128-row A slices, a 6-deep ring,
// 193 KB, 16 expansion warps (one CTA per SM).  A slice then holds only
// 128 x 128 x 64 of MMA work, so the expansion must run further ahead of the
// MMAs and have more warps to hide its latencies: each of four groups of 128
// threads takes one half of every other block.
template <bool kSmall>
struct Lay {
  static constexpr int kExpThreads = kSmall ? 512 : 256;
  static constexpr int kThreads = 32 * kExpWarp0 + kExpThreads;
  static constexpr int kStages = kSmall ? 6 : 2;
  static constexpr int kASlice = (kSmall ? UM : BM) * BK * 2;  // 16 or 32 KB
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kASlice;
  static constexpr int kOffBar = kOffB + kStages * kBSlice;
  // barriers: a_full[S], b_full[S], empty[S], acc
  static constexpr int kNumBars = 3 * kStages + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kCtasPerSm = kSmall ? 1 : 2;
};
static_assert(2 * (Lay<false>::kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(Lay<true>::kSmemBytes + 1024 <= 227 * 1024, "one CTA per SM");

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return smem_addr(p); }

// Shared-memory matrix descriptor of a K-major, 128B-swizzled tile whose
// 8-row x 128-byte atoms are stacked every 1024 bytes (SBO).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);        // start address
  d |= (uint64_t)1 << 16;                       // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset
  d |= (uint64_t)1 << 46;                       // descriptor version
  d |= (uint64_t)2 << 61;                       // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 accumulator (bits 4-5), A and B format
// (bits 7-9, 10-12: 0 fp16, 1 bf16), both K-major, N = 128, M = 128.
template <bool kBf16>
__host__ __device__ constexpr uint32_t idesc() {
  return (1u << 4) | (kBf16 ? (1u << 7) | (1u << 10) : 0u) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)(UM >> 4) << 24);
}

template <bool kBf16>
__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc<kBf16>()), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Byte offset of element (r, k) (k < 64) inside a 128-row, 64-wide 16-bit tile
// in the canonical K-major 128B-swizzled layout.
__device__ __forceinline__ uint32_t sw128_off(int r, int k) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((k >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

// Expansion arithmetic.  PRMT picks each output byte from 8 source bytes; the
// per-block sources are {-s, 0, +s} as 16-bit values (bytes 0-1, 2-3, 4-5), so
// a weight with digit d = t + 1 selects bytes 2d and 2d + 1, and a pair of
// weights with digits (da, db) -- one 32-bit output word -- uses the selector
//   (2da) | (2da+1) << 4 | (2db) << 8 | (2db+1) << 12 = 34 (da + 256 db) + 0x1010.
// Digits come from the peel of "What Ferrox does with it",
//   d_n = floor(3^(n+1) u) - 3 floor(3^n u),  u = byte / 256,
// computed for two bytes at once: with byte A in bits 0-7 and byte B in bits
// 16-23 of S, S * 3^n holds 3^n A and 3^n B in its two 16-bit lanes
// (3^5 * 255 < 2^16), their floors (/256) are bytes 1 and 3, and
// F_{n+1} - 3 F_n never borrows across lanes (it is the digit, 0..2).
// digits2(S) returns D_n = dA_n | dB_n << 16 for n = 0..4.
__device__ __forceinline__ void digits2(uint32_t S, uint32_t D[5]) {
  uint32_t F = 0u;  // F_0 = floor(byte / 256) = 0
  uint32_t P = S;
#pragma unroll
  for (int n = 0; n < 5; ++n) {
    P *= 3u;                                         // 3^(n+1) byte, per lane
    const uint32_t Fn = __byte_perm(P, 0u, 0x4341);  // floor(.../256), per lane
    D[n] = Fn - 3u * F;
    F = Fn;
  }
}

// Output word for the digit pair picked from Da and Db: the pair's selector
// applied to the {-s, 0, +s} sources.
__device__ __forceinline__ uint32_t word_of(uint32_t Da, uint32_t Db, uint32_t pick, uint32_t ta,
                                            uint32_t tb) {
  const uint32_t pair = __byte_perm(Da, Db, pick);  // da | db << 8
  return __byte_perm(ta, tb, 34u * pair + 0x1010u);
}
// picks: digit of byte A (lane 0) or B (lane 1) of Da, then of Db
constexpr uint32_t kAA = 0x1140, kBB = 0x1162, kAB = 0x1160;

// Half h of one 128-weight block of one row: 64 16-bit values t * s written as
// 8 swizzled 16-byte chunks.  `win` holds the 16-byte-aligned bytes that
// contain the block, which starts at byte `o` of the window.  Bytes (2i, 2i+1)
// of the block are peeled together and give the ten weights 10i..10i+9 as five
// words: (d0,d1)A (d2,d3)A (d4A,d0B) (d1,d2)B (d3,d4)B.
template <int h, int o>
__device__ __forceinline__ void expand_half(const uint32_t win[12], uint32_t ta, uint32_t tb,
                                            uint32_t bslice, int r) {
  auto pair_of = [&](int i) -> uint32_t {  // bytes 2i, 2i+1 of the block in lanes 0, 1
    const int j0 = o + 2 * i, j1 = o + 2 * i + 1;
    const uint32_t sel = (uint32_t)(j0 & 3) | ((uint32_t)(4 + (j1 & 3)) << 8);
    return __byte_perm(win[j0 >> 2], win[j1 >> 2], sel) & 0x00FF00FFu;
  };
  uint32_t out[32];
  int n = 0;
  if constexpr (h == 0) {
#pragma unroll
    for (int i = 0; i < 6; ++i) {  // weights 0..59
      uint32_t D[5];
      digits2(pair_of(i), D);
      out[n++] = word_of(D[0], D[1], kAA, ta, tb);
      out[n++] = word_of(D[2], D[3], kAA, ta, tb);
      out[n++] = word_of(D[4], D[0], kAB, ta, tb);
      out[n++] = word_of(D[1], D[2], kBB, ta, tb);
      out[n++] = word_of(D[3], D[4], kBB, ta, tb);
    }
    uint32_t D[5];
    digits2(pair_of(6), D);  // weights 60..63
    out[n++] = word_of(D[0], D[1], kAA, ta, tb);
    out[n++] = word_of(D[2], D[3], kAA, ta, tb);
  } else {
    {
      uint32_t D[5];
      digits2(pair_of(6), D);  // weights 64..69
      out[n++] = word_of(D[4], D[0], kAB, ta, tb);
      out[n++] = word_of(D[1], D[2], kBB, ta, tb);
      out[n++] = word_of(D[3], D[4], kBB, ta, tb);
    }
#pragma unroll
    for (int i = 7; i < 12; ++i) {  // weights 70..119
      uint32_t D[5];
      digits2(pair_of(i), D);
      out[n++] = word_of(D[0], D[1], kAA, ta, tb);
      out[n++] = word_of(D[2], D[3], kAA, ta, tb);
      out[n++] = word_of(D[4], D[0], kAB, ta, tb);
      out[n++] = word_of(D[1], D[2], kBB, ta, tb);
      out[n++] = word_of(D[3], D[4], kBB, ta, tb);
    }
    uint32_t D[5];
    digits2(pair_of(12), D);  // weights 120..127; byte 25's last two digits are padding
    out[n++] = word_of(D[0], D[1], kAA, ta, tb);
    out[n++] = word_of(D[2], D[3], kAA, ta, tb);
    out[n++] = word_of(D[4], D[0], kAB, ta, tb);
    out[n++] = word_of(D[1], D[2], kBB, ta, tb);
  }
#pragma unroll
  for (int c = 0; c < 8; ++c)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(bslice + sw128_off(r, 8 * c)),
                 "r"(out[4 * c]), "r"(out[4 * c + 1]), "r"(out[4 * c + 2]), "r"(out[4 * c + 3])
                 : "memory");
}

// The packed bytes of one block of one row: the 16-byte chunks of the row
// that the block's 26 bytes touch (two or three), and the block's scale.
// Block kb of a row starts at byte 26 kb; rows are whole multiples of 208 =
// 13 * 16 bytes (K % 1024 == 0), so with q = kb % 8 the block starts at byte
// (26 q) % 16 of the chunk (26 kb) / 16 and no chunk past the block is read.
template <int q>
__device__ __forceinline__ void load_block(const uint8_t* row, const uint16_t* srow, int kb,
                                           uint32_t win[12], uint32_t& sc) {
  constexpr int o = (kBlockBytes * q) & 15;
  constexpr int nc = (o + kBlockBytes + 15) / 16;
  const uint4* p = reinterpret_cast<const uint4*>(row + ((kBlockBytes * kb) & ~15));
#pragma unroll
  for (int i = 0; i < nc; ++i) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p + i));
    win[4 * i] = v.x; win[4 * i + 1] = v.y; win[4 * i + 2] = v.z; win[4 * i + 3] = v.w;
  }
  unsigned short s;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(s) : "l"(srow + kb));
  sc = s;
}

// PQ2_0 (two bits a weight, 32 bytes a block): half h of block kb of a row is
// the 16 aligned bytes at 32 kb + 16 h -- one 16-byte load -- and weight
// 4j + i of the half is bits 2i, 2i+1 of its byte j.
__device__ __forceinline__ void load_half_pq2(const uint8_t* row, const uint16_t* srow, int kb,
                                              int h, uint32_t (&win)[4], uint32_t& sc) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(row + 32 * kb + 16 * h));
  win[0] = v.x; win[1] = v.y; win[2] = v.z; win[3] = v.w;
  unsigned short s;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(s) : "l"(srow + kb));
  sc = s;
}

// The 64 weights of a PQ2_0 half-block as 32 output words.  Nibble k of the
// half holds the codes (ca, cb) of weights 2k, 2k+1, and the pair's selector
// over the sources {-s, 0, +s, +2s} is 34 (ca + 256 cb) + 0x1010, where
// ca + 256 cb = n + 63 (n & 12) for the nibble n = ca + 4 cb.  (Code 3, which
// no encoder writes, decodes as trit + 2 like every other code: c - 1.)
__device__ __forceinline__ void expand_half_pq2(const uint32_t (&win)[4], uint32_t ta, uint32_t tb,
                                                uint32_t bslice, int r) {
  uint32_t out[32];
#pragma unroll
  for (int w = 0; w < 4; ++w)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t m = win[w] >> (4 * i);
      const uint32_t n = m & 15u;
      out[8 * w + i] = __byte_perm(ta, tb, 34u * (n + 63u * (m & 12u)) + 0x1010u);
    }
#pragma unroll
  for (int c = 0; c < 8; ++c)
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(bslice + sw128_off(r, 8 * c)),
                 "r"(out[4 * c]), "r"(out[4 * c + 1]), "r"(out[4 * c + 2]), "r"(out[4 * c + 3])
                 : "memory");
}

struct ExpCtx {
  const uint8_t* row;     // this thread's packed row
  const uint16_t* srow;   // its scales
  int g_lo, ng;           // the split's first 1024-wide group and its group count
  uint32_t bbase;         // shared address of B slice 0 (slice s at + s kBSlice)
  uint64_t* empty;        // empty[0 .. S)
  uint64_t* b_full;       // b_full[0 .. S)
  int r;
  volatile int* abort_flag;
};

// The split's j-th 1024-wide group (j < ng).
__device__ __forceinline__ int group_at(const ExpCtx& c, int j) { return c.g_lo + j; }

// Slice 2 lb + h (block lb of the split, half h) takes ring stage
// (2 lb + h) % S for the ((2 lb + h) / S)-th time: wait until the MMAs of its
// previous use have read it (bounded), and return the stage.
template <int kS, int h>
__device__ __forceinline__ int claim_stage(const ExpCtx& c, int lb, bool* ok) {
  const int i = 2 * lb + h, st = i % kS, n = i / kS;
  *ok = n == 0 || mbar_wait(c.empty + st, (uint32_t)((n - 1) & 1), c.abort_flag);
  return st;
}

// Block q of the split's j-th group (block lb = 8 j + q in the split's order):
// prefetch block lb + 3 into ring slot (q + 3) % 4 (the slot block lb - 1
// has left), wait for its B slice to be free, expand, publish.
template <bool kBf16, int kS, int h, int q>
__device__ __forceinline__ bool expand_step(const ExpCtx& c, int j, uint32_t (&win)[4][12],
                                            uint32_t (&sc)[4]) {
  const int lb = 8 * j + q;  // block index in the split's order
  if (lb + 3 < 8 * c.ng) {
    const int gn = q + 3 < 8 ? group_at(c, j) : group_at(c, j + 1);
    load_block<(q + 3) % 8>(c.row, c.srow, 8 * gn + (q + 3) % 8, win[(q + 3) % 4],
                            sc[(q + 3) % 4]);
  }
  uint32_t s16 = sc[q % 4];
  if constexpr (kBf16)  // the fp16 scale rounded to nearest-even bf16
    s16 = __bfloat16_as_ushort(
        __float2bfloat16_rn(__half2float(__ushort_as_half((unsigned short)s16))));
  // PRMT sources: bytes 0-1 = -s, 2-3 = 0, 4-5 = +s
  const uint32_t ta = (s16 ^ 0x8000u), tb = s16;
  bool ok;
  const int st = claim_stage<kS, h>(c, lb, &ok);
  if (!ok) return false;
  expand_half<h, (kBlockBytes * q) & 15>(win[q % 4], ta, tb, c.bbase + (uint32_t)(st * kBSlice),
                                         c.r);
  // every writer makes its stores visible to the tensor core's (async) proxy
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_arrive(c.b_full + st);
  return true;
}

// PQ2_0: block lb = 8 j + q of this thread's half (in the split's order),
// with the half-blocks of blocks lb + 1, lb + 2 prefetched into ring slots
// (q + 1) % 4, (q + 2) % 4.
template <bool kBf16, int kS, int h, int q>
__device__ __forceinline__ bool expand_step_pq2(const ExpCtx& c, int j, uint32_t (&win)[4][4],
                                                uint32_t (&sc)[4]) {
  const int lb = 8 * j + q;
  if (lb + 2 < 8 * c.ng) {
    const int gn = q + 2 < 8 ? group_at(c, j) : group_at(c, j + 1);
    load_half_pq2(c.row, c.srow, 8 * gn + (q + 2) % 8, h, win[(q + 2) % 4], sc[(q + 2) % 4]);
  }
  uint32_t s16 = sc[q % 4];
  float sf = __half2float(__ushort_as_half((unsigned short)s16));
  if constexpr (kBf16) {  // the fp16 scale rounded to nearest-even bf16
    s16 = __bfloat16_as_ushort(__float2bfloat16_rn(sf));
    sf = __uint_as_float(s16 << 16);
  }
  const uint32_t s2 = kBf16 ? (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(2.0f * sf))
                            : (uint32_t)__half_as_ushort(__float2half_rn(2.0f * sf));
  const uint32_t ta = (s16 ^ 0x8000u), tb = s16 | (s2 << 16);
  bool ok;
  const int st = claim_stage<kS, h>(c, lb, &ok);
  if (!ok) return false;
  expand_half_pq2(win[q % 4], ta, tb, c.bbase + (uint32_t)(st * kBSlice), c.r);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_arrive(c.b_full + st);
  return true;
}

template <bool kBf16, int kS, int h>
__device__ bool expand_all_pq2(const ExpCtx& c) {
  uint32_t win[4][4], sc[4];
  const int g0 = group_at(c, 0);
  load_half_pq2(c.row, c.srow, 8 * g0, h, win[0], sc[0]);
  load_half_pq2(c.row, c.srow, 8 * g0 + 1, h, win[1], sc[1]);
  for (int g = 0; g < c.ng; ++g) {
    if (!expand_step_pq2<kBf16, kS, h, 0>(c, g, win, sc)) return false;
    if (!expand_step_pq2<kBf16, kS, h, 1>(c, g, win, sc)) return false;
    if (!expand_step_pq2<kBf16, kS, h, 2>(c, g, win, sc)) return false;
    if (!expand_step_pq2<kBf16, kS, h, 3>(c, g, win, sc)) return false;
    if (!expand_step_pq2<kBf16, kS, h, 4>(c, g, win, sc)) return false;
    if (!expand_step_pq2<kBf16, kS, h, 5>(c, g, win, sc)) return false;
    if (!expand_step_pq2<kBf16, kS, h, 6>(c, g, win, sc)) return false;
    if (!expand_step_pq2<kBf16, kS, h, 7>(c, g, win, sc)) return false;
  }
  return true;
}

// The small variant's expansion: half h of the blocks of parity p (blocks
// 8 g + q, q = p, p + 2, p + 4, p + 6), each thread two of its own blocks
// ahead in a 4-slot register ring (own block kb in slot q / 2).
template <bool kBf16, int kS, int h, int q>
__device__ __forceinline__ bool expand_step_par(const ExpCtx& c, int j, uint32_t (&win)[4][12],
                                                uint32_t (&sc)[4]) {
  const int lb = 8 * j + q;
  if (lb + 4 < 8 * c.ng) {
    const int gn = q + 4 < 8 ? group_at(c, j) : group_at(c, j + 1);
    load_block<(q + 4) % 8>(c.row, c.srow, 8 * gn + (q + 4) % 8, win[((q >> 1) + 2) % 4],
                            sc[((q >> 1) + 2) % 4]);
  }
  uint32_t s16 = sc[q >> 1];
  if constexpr (kBf16)  // the fp16 scale rounded to nearest-even bf16
    s16 = __bfloat16_as_ushort(
        __float2bfloat16_rn(__half2float(__ushort_as_half((unsigned short)s16))));
  const uint32_t ta = (s16 ^ 0x8000u), tb = s16;
  bool ok;
  const int st = claim_stage<kS, h>(c, lb, &ok);
  if (!ok) return false;
  expand_half<h, (kBlockBytes * q) & 15>(win[q >> 1], ta, tb, c.bbase + (uint32_t)(st * kBSlice),
                                         c.r);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_arrive(c.b_full + st);
  return true;
}

template <bool kBf16, int kS, int h, int p>
__device__ bool expand_par(const ExpCtx& c) {
  uint32_t win[4][12], sc[4];
  const int g0 = group_at(c, 0);
  load_block<p>(c.row, c.srow, 8 * g0 + p, win[0], sc[0]);  // a split holds >= 8 blocks
  load_block<p + 2>(c.row, c.srow, 8 * g0 + p + 2, win[1], sc[1]);
  for (int g = 0; g < c.ng; ++g) {
    if (!expand_step_par<kBf16, kS, h, p>(c, g, win, sc)) return false;
    if (!expand_step_par<kBf16, kS, h, p + 2>(c, g, win, sc)) return false;
    if (!expand_step_par<kBf16, kS, h, p + 4>(c, g, win, sc)) return false;
    if (!expand_step_par<kBf16, kS, h, p + 6>(c, g, win, sc)) return false;
  }
  return true;
}

template <bool kBf16, int kS, int h>
__device__ bool expand_all(const ExpCtx& c) {
  uint32_t win[4][12], sc[4];
  const int g0 = group_at(c, 0);
  load_block<0>(c.row, c.srow, 8 * g0, win[0], sc[0]);
  load_block<1>(c.row, c.srow, 8 * g0 + 1, win[1], sc[1]);  // a split holds >= 8 blocks
  load_block<2>(c.row, c.srow, 8 * g0 + 2, win[2], sc[2]);
  for (int g = 0; g < c.ng; ++g) {
    if (!expand_step<kBf16, kS, h, 0>(c, g, win, sc)) return false;
    if (!expand_step<kBf16, kS, h, 1>(c, g, win, sc)) return false;
    if (!expand_step<kBf16, kS, h, 2>(c, g, win, sc)) return false;
    if (!expand_step<kBf16, kS, h, 3>(c, g, win, sc)) return false;
    if (!expand_step<kBf16, kS, h, 4>(c, g, win, sc)) return false;
    if (!expand_step<kBf16, kS, h, 5>(c, g, win, sc)) return false;
    if (!expand_step<kBf16, kS, h, 6>(c, g, win, sc)) return false;
    if (!expand_step<kBf16, kS, h, 7>(c, g, win, sc)) return false;
  }
  return true;
}

// 16 consecutive fp32 accumulator columns of this warp's 32 TMEM lanes
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

// blockIdx.z = split of K: with G = q S + r 1024-wide groups, splits
// 0..r-1 take q + 1 consecutive groups and the rest q, so the longer splits
// are the lower CTA indices and start in the first round of CTAs placed on
// the SMs; when S > 1 split z writes fp32 partial sums to y + z M N
// (kOutF32).
// kSwiGLU: the weight is a fused gate+up of N = 2I rows (gate rows 0..I-1,
// then up rows), and y is h = silu(g) * u, M x I fp32, with
// silu(a) = a / (1 + e^-a) (the feed-forward block of "Speed, and where it
// goes").  Tile x then covers gate rows [64 x, 64 x + 64) in its first 64
// columns and the matching up rows in the other 64, so the epilogue holds
// both factors of each output; no split.
// kPQ2: the weights are PQ2_0 (2-bit codes, 32 bytes a block).
// kSmall: M <= 128 (one 128-row accumulator), the deep ring of Lay<true>.
template <bool kBf16, bool kOutF32, bool kSwiGLU = false, bool kPQ2 = false, bool kSmall = false>
__global__ void __launch_bounds__(Lay<kSmall>::kThreads, Lay<kSmall>::kCtasPerSm)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const uint8_t* __restrict__ wq,
                   const uint16_t* __restrict__ scales, void* __restrict__ y, int M, int N, int K,
                   int splits, int* status) {
  static_assert(!kSwiGLU || kOutF32, "h is fp32");
  // No static shared variables: the dynamic window starts at offset 0, so the
  // declared 1024-byte alignment holds, and every access below stays a
  // shared-memory instruction (an address laundered through an integer
  // would turn them into generic ones).
  extern __shared__ __align__(1024) unsigned char smem[];
  using Y = Lay<kSmall>;
  constexpr int kStages = Y::kStages, kASlice = Y::kASlice;
  constexpr int kOffA = Y::kOffA, kOffB = Y::kOffB, kOffMisc = Y::kOffMisc;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Y::kOffBar);
  uint64_t* a_full = bars;
  uint64_t* b_full = bars + kStages;
  uint64_t* empty = bars + 2 * kStages;
  uint64_t* acc_full = bars + 3 * kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * (kSwiGLU ? BN / 2 : BN);
  const int I = N / 2;  // kSwiGLU: gate rows, up rows, and the columns of h
  const int nblk = K / kBlockWeights;
  const int G = K / kRot, z = blockIdx.z;
  const int gq = G / splits, gr = G % splits;
  const int g_lo = z * gq + (z < gr ? z : gr), g_hi = g_lo + gq + (z < gr ? 1 : 0);
  const int kb0 = g_lo * (kRot / BK), kb1 = g_hi * (kRot / BK);  // this split's 64-wide slices
  const int nk = kb1 - kb0;
  // the second 128-row half only when it holds rows (never in the small variant)
  const int nmh = !kSmall && M - m0 > UM ? 2 : 1;
  if (kOutF32 && splits > 1) y = static_cast<float*>(y) + (size_t)z * M * N;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&b_full[s], BN);  // the 128 threads (one per row) that expand a slice
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // TMEM: two 128-column fp32 accumulators x 128 lanes
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(2 * BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  int a_issued = 0;
  if (warp == 0) {
    // ---- TMA producer of A --------------------------------------------------------
    if (lane == 0) {
      pdl_wait();  // A may come from the previous kernel
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kStages, round = kb / kStages;
        if (round > 0) ok = mbar_wait(&empty[s], (round - 1) & 1, abort_flag);
        if (!ok) break;
        // M <= 128: the A box is 128 rows (no zero fill for the empty half)
        mbar_expect_tx(&a_full[s], (kSmall || M <= UM) ? UM * BK * 2 : kASlice);
        tma_2d(smem_u32(smem + kOffA + s * kASlice), &map_a, (kb0 + kb) * BK, m0, &a_full[s]);
        ++a_issued;
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ------------------------------------------------------------------
    if (lane == 0) {
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kStages, round = kb / kStages;
        ok = mbar_wait(&a_full[s], round & 1, abort_flag) &&
             mbar_wait(&b_full[s], round & 1, abort_flag);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a_addr = smem_u32(smem + kOffA + s * kASlice);
        const uint32_t b_addr = smem_u32(smem + kOffB + s * kBSlice);
        for (int mh = 0; mh < nmh; ++mh)
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // K = 16 per MMA: 32 bytes along the atom
            umma_f16<kBf16>(tmem + mh * BN, sw128_desc(a_addr + mh * (UM * 128) + 32 * kk),
                            sw128_desc(b_addr + 32 * kk), (kb | kk) != 0);
        umma_commit(&empty[s]);  // frees the slice once these MMAs have read it
      }
      umma_commit(acc_full);     // all MMAs issued by this thread
    }
  } else {
    // ---- B expansion: thread (row r, half h); slice 2 kb + h uses stage (2 kb + h) % S
    // h, p: warp-uniform; p (small variant) picks the blocks of one parity
    const int t = threadIdx.x - 32 * kExpWarp0, r = t & (BN - 1), h = (t >> 7) & 1, p = t >> 8;
    int n;
    if constexpr (kSwiGLU) {  // columns 0-63: gate rows n0.., 64-127: up rows I + n0..
      const int i = n0 + (r & (BN / 2 - 1));
      n = (r < BN / 2 ? 0 : I) + (i < I ? i : I - 1);  // past I: a valid row, never stored
    } else {
      n = n0 + r < N ? n0 + r : N - 1;  // rows past N expand a valid row; never stored
    }
    ExpCtx c;
    c.row = wq + (size_t)n * nblk * (kPQ2 ? 32 : kBlockBytes);
    c.srow = scales + (size_t)n * nblk;
    c.g_lo = g_lo;
    c.ng = g_hi - g_lo;
    c.bbase = smem_u32(smem + kOffB);
    c.empty = empty;
    c.b_full = b_full;
    c.r = r;
    c.abort_flag = abort_flag;
    static_assert(!(kPQ2 && kSmall), "the small variant expands PTQ1_0 blocks");
    if constexpr (kPQ2)
      ok = h == 0 ? expand_all_pq2<kBf16, kStages, 0>(c) : expand_all_pq2<kBf16, kStages, 1>(c);
    else if constexpr (kSmall)
      ok = h == 0 ? (p == 0 ? expand_par<kBf16, kStages, 0, 0>(c) : expand_par<kBf16, kStages, 0, 1>(c))
                  : (p == 0 ? expand_par<kBf16, kStages, 1, 0>(c) : expand_par<kBf16, kStages, 1, 1>(c));
    else
      ok = h == 0 ? expand_all<kBf16, kStages, 0>(c) : expand_all<kBf16, kStages, 1>(c);
  }
  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) atomicOr(status, kDevTimeout);
  }

  // ---- epilogue: warps 2-9; warp w reads TMEM lanes 32 (w % 4) .. + 31 of
  // accumulator (w - 2) / 4 -------------------------------------------------------------
  if (warp >= kExpWarp0 && warp < kExpWarp0 + 8) {  // small variant: the other warps idle
    const bool done = !*abort_flag && mbar_wait(acc_full, 0, abort_flag);
    if (done) {
      pdl_wait();  // the previous kernel may still read y
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int q = warp & 3, mh = (warp - kExpWarp0) >> 2;
      const int row = m0 + mh * UM + 32 * q + lane;
      if constexpr (kSwiGLU) {
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(mh * BN);
#pragma unroll 1
        for (int c0 = 0; c0 < BN / 2; c0 += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(taddr + (uint32_t)c0, g);
          tmem_ld16(taddr + (uint32_t)(BN / 2 + c0), u);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          if (row < M) {
            float* out = static_cast<float*>(y) + (size_t)row * I + n0 + c0;
            float hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a = __uint_as_float(g[i]);
              hv[i] = a / (1.0f + expf(-a)) * __uint_as_float(u[i]);
            }
            if (n0 + c0 + 16 <= I && (I & 3) == 0) {
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(out + i) = make_float4(hv[i], hv[i + 1], hv[i + 2], hv[i + 3]);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (n0 + c0 + i < I) out[i] = hv[i];
            }
          }
        }
      } else
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
            "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, "
            "%26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
              "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
              "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]),
              "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
              "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
              "=r"(v[30]), "=r"(v[31])
            : "r"(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(mh * BN + c0)));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (row < M) {
          const int ncol = n0 + c0;
          if constexpr (kOutF32) {
            float* out = static_cast<float*>(y) + (size_t)row * N + ncol;
            if (ncol + 32 <= N && (N & 3) == 0) {
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(out + i) =
                    make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (ncol + i < N) out[i] = __uint_as_float(v[i]);
            }
          } else {
            uint16_t* out = static_cast<uint16_t*>(y) + (size_t)row * N + ncol;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[2 * i]))) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[2 * i + 1])))
                       << 16);
            if (ncol + 32 <= N && (N & 7) == 0) {
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<uint4*>(out + 2 * i) =
                    make_uint4(pk[i], pk[i + 1], pk[i + 2], pk[i + 3]);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (ncol + i < N) out[i] = (uint16_t)(pk[i >> 1] >> (16 * (i & 1)));
            }
          }
        }
      }
    }
  }
  if (*abort_flag && warp == 1 && lane == 0) {
    // let the MMAs already issued finish before TMEM is released (bounded;
    // acc_full was committed after the issuing loop, aborted or not)
    static_cast<void>(mbar_wait(acc_full, 0, nullptr));
  }
  if (*abort_flag && warp == 0 && lane == 0) {
    // let this CTA's copies in flight land before its shared memory goes away
    for (int kb = (a_issued > kStages ? a_issued - kStages : 0); kb < a_issued; ++kb)
      static_cast<void>(mbar_wait(&a_full[kb % kStages], (kb / kStages) & 1, nullptr));
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  pdl_release();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * BN)
                 : "memory");
  }
}

// y[i] = sum over splits z = 0..S-1 of part[z][i], in that order, stored as
// bf16 (kOutF32 false) or fp32.
template <bool kOutF32>
__global__ void __launch_bounds__(256) gemm_split_reduce_kernel(const float* __restrict__ part,
                                                                void* __restrict__ y, size_t MN,
                                                                int S) {
  pdl_release();
  pdl_wait();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= MN) return;
  float acc = 0.0f;
  for (int z = 0; z < S; ++z) acc += __ldcg(part + (size_t)z * MN + i);
  if constexpr (kOutF32)
    static_cast<float*>(y)[i] = acc;
  else
    static_cast<uint16_t*>(y)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
}

// ---- host side -------------------------------------------------------------------------
// The TMA map of A (M x K, 16-bit): boxes of 64 x 256 rows, or 64 x 128 when
// M <= 128 -- then only the lower accumulator has rows, and the upper 128
// rows of the box would only be zero fill.
static cudaError_t encode_a(CUtensorMap* ma, const void* x, int64_t M, int64_t K) {
  return encode_tma_2d(ma, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, K, M, K * 2, BK, M <= UM ? UM : BM,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool kBf16, bool kOutF32, bool kSwiGLU, bool kPQ2, bool kSmall>
cudaError_t launch_v(const CUtensorMap& ma, const uint8_t* wq, const uint16_t* scales, void* y,
                     int M, int N, int K, int splits, int* status, cudaStream_t st) {
  auto kern = gemm_tc_kernel<kBf16, kOutF32, kSwiGLU, kPQ2, kSmall>;
  constexpr int kSmemBytes = Lay<kSmall>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const int cols = kSwiGLU ? BN / 2 : BN;  // output columns per tile
  const int ncols = kSwiGLU ? N / 2 : N;
  const dim3 grid((unsigned)((ncols + cols - 1) / cols), (unsigned)((M + BM - 1) / BM),
                  (unsigned)splits);
  return launch_pdl(kern, grid, dim3(Lay<kSmall>::kThreads), (size_t)kSmemBytes, st, ma, wq,
                    scales, y, M, N,
                    K, splits, status);
}

constexpr int64_t kGpuSms = 152;

// The small-M variant (one accumulator, deep ring, one CTA per SM) serves
// M <= 128 when the tiles fill between half and all of the SMs: unsplit, in
// one wave.  Fewer tiles are split along K over two CTAs per SM, more run
// two per SM in the large variant.
static bool small_variant(int64_t M, int64_t N) {
  const int64_t tiles = (N + BN - 1) / BN;
  return M <= UM && 2 * tiles > kGpuSms && tiles <= kGpuSms;
}

template <bool kBf16, bool kOutF32, bool kSwiGLU = false, bool kPQ2 = false>
cudaError_t launch_t(const CUtensorMap& ma, const uint8_t* wq, const uint16_t* scales, void* y,
                     int M, int N, int K, int splits, int* status, cudaStream_t st) {
  if constexpr (!kPQ2)  // (the PQ2_0 expansion has no parity-strided form)
    if (splits == 1 && small_variant(M, N))
      return launch_v<kBf16, kOutF32, kSwiGLU, kPQ2, true>(ma, wq, scales, y, M, N, K, splits,
                                                           status, st);
  return launch_v<kBf16, kOutF32, kSwiGLU, kPQ2, false>(ma, wq, scales, y, M, N, K, splits,
                                                        status, st);
}

}  // namespace

// Number of K splits for an M x N x K product.  Splitting pays only when most
// SMs of a 152-SM part would otherwise idle (fewer tiles than half the SMs:
// measured, 136 tiles of M=128 ran 40 us unsplit and 54 us in two splits);
// then enough splits to fill two CTAs per SM, at most one per 1024-wide group
// and at most kMaxSplits.  (The feed-forward down projection at M=256, 40
// tiles, ran its 64 layers in 10.47 ms with 7 splits against 10.11 ms with
// 6, although the GEMM alone took 72 against 76 us.)  A function of the
// shape alone, so the workspace query and the launch agree.
int gemm_tc_splits(int64_t M, int64_t N, int64_t K) {
  constexpr int64_t kSms = kGpuSms, kMaxSplits = 6;
  if (K % kRot != 0 || M <= 0 || N <= 0) return 1;
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  if (2 * tiles > kSms) return 1;
  int64_t s = 2 * kSms / tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  if (s > K / kRot) s = K / kRot;
  return s < 2 ? 1 : (int)s;
}

size_t gemm_tc_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int s = gemm_tc_splits(M, N, K);
  return s > 1 ? (size_t)s * (size_t)M * (size_t)N * 4 : 0;
}

// Tensor-core GEMM for K % 1024 == 0 (cudaErrorNotSupported otherwise).
// ws/ws_bytes: scratch for split-K partial sums; with less than
// gemm_tc_workspace_bytes the product runs with as many splits as fit.
cudaError_t launch_gemm_tc(const uint8_t* wq, const uint16_t* scales, const void* x, Act x_t,
                           void* y, Act y_t, int64_t M, int64_t N, int64_t K, void* ws,
                           size_t ws_bytes, cudaStream_t st) {
  if (K % kRot != 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX ||
      (M + BM - 1) / BM > 65535)
    return cudaErrorNotSupported;
  cudaError_t e;
  CUtensorMap ma;
  if ((e = encode_a(&ma, x, M, K)) != cudaSuccess) return e;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevice;
  const int m = (int)M, n = (int)N, k = (int)K;
  const bool bf = x_t == Act::BF16, f32 = y_t == Act::F32;
  int splits = gemm_tc_splits(M, N, K);
  const size_t per = (size_t)M * (size_t)N * 4;
  if (splits > 1 && (ws == nullptr || ws_bytes / per < 2)) splits = 1;
  if (splits > 1 && ws_bytes / per < (size_t)splits) splits = (int)(ws_bytes / per);
  if (splits > 1) {  // fp32 partials, then the fixed-order sum
    e = bf ? launch_t<true, true>(ma, wq, scales, ws, m, n, k, splits, status, st)
           : launch_t<false, true>(ma, wq, scales, ws, m, n, k, splits, status, st);
    if (e != cudaSuccess) return e;
    const size_t mn = (size_t)M * (size_t)N;
    const dim3 grid((unsigned)((mn + 255) / 256));
    return f32 ? launch_pdl(gemm_split_reduce_kernel<true>, grid, dim3(256), 0, st,
                            (const float*)ws, y, mn, splits)
               : launch_pdl(gemm_split_reduce_kernel<false>, grid, dim3(256), 0, st,
                            (const float*)ws, y, mn, splits);
  }
  if (bf && f32) return launch_t<true, true>(ma, wq, scales, y, m, n, k, 1, status, st);
  if (bf) return launch_t<true, false>(ma, wq, scales, y, m, n, k, 1, status, st);
  if (f32) return launch_t<false, true>(ma, wq, scales, y, m, n, k, 1, status, st);
  return launch_t<false, false>(ma, wq, scales, y, m, n, k, 1, status, st);
}

// The GEMM over PQ2_0 weights: x bf16, y bf16 (K % 1024 == 0).
cudaError_t launch_gemm_tc_pq2(const uint8_t* wq, const uint16_t* scales, const void* x, void* y,
                               int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes,
                               cudaStream_t st) {
  if (K % kRot != 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX ||
      (M + BM - 1) / BM > 65535)
    return cudaErrorNotSupported;
  cudaError_t e;
  CUtensorMap ma;
  if ((e = encode_a(&ma, x, M, K)) != cudaSuccess) return e;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevice;
  const int m = (int)M, n = (int)N, k = (int)K;
  int splits = gemm_tc_splits(M, N, K);
  const size_t per = (size_t)M * (size_t)N * 4;
  if (splits > 1 && (ws == nullptr || ws_bytes / per < 2)) splits = 1;
  if (splits > 1 && ws_bytes / per < (size_t)splits) splits = (int)(ws_bytes / per);
  if (splits > 1) {
    e = launch_t<true, true, false, true>(ma, wq, scales, ws, m, n, k, splits, status, st);
    if (e != cudaSuccess) return e;
    const size_t mn = (size_t)M * (size_t)N;
    return launch_pdl(gemm_split_reduce_kernel<false>, dim3((unsigned)((mn + 255) / 256)),
                      dim3(256), 0, st, (const float*)ws, y, mn, splits);
  }
  return launch_t<true, false, false, true>(ma, wq, scales, y, m, n, k, 1, status, st);
}

cudaError_t launch_gemm_tc_swiglu(const uint8_t* wq, const uint16_t* scales, const void* x,
                                  Act x_t, float* h, int64_t M, int64_t I, int64_t K,
                                  cudaStream_t st) {
  const int64_t N = 2 * I;
  if (K % kRot != 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX ||
      (M + BM - 1) / BM > 65535 || gemm_tc_splits(M, N, K) != 1)
    return cudaErrorNotSupported;
  cudaError_t e;
  CUtensorMap ma;
  if ((e = encode_a(&ma, x, M, K)) != cudaSuccess) return e;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevice;
  const int m = (int)M, n = (int)N, k = (int)K;
  return x_t == Act::BF16 ? launch_t<true, true, true>(ma, wq, scales, h, m, n, k, 1, status, st)
                          : launch_t<false, true, true>(ma, wq, scales, h, m, n, k, 1, status, st);
}

}  // namespace ptq

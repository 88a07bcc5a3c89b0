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
// Tile: 256 (M) x 128 (N): two 128-row accumulators in TMEM share every
// expanded B slice, so each weight is peeled once per 256 activation rows.
// K is consumed in 64-wide slices (one 128-byte swizzle atom of 16-bit
// values), kStages slices in flight.  Warp roles (10 warps):
//   warp 0      TMA producer: A slices (box 64 x 256, 128B swizzle) and, per
//               1024-wide group, the packed trits (box 208 B x 128 rows) and
//               scales (box 8 x 128) into a 2-deep group ring, one group ahead.
//   warp 1      TMEM allocation; lane 0 issues tcgen05.mma (8 per slice).
//   warps 2-9   expansion: thread (row r, half h) peels the 64 weights of half
//               h of each 128-weight block of row r.  A table built per CTA
//               maps each byte value to byte-permute selectors, so every pair
//               of 16-bit outputs is one permute of the per-block bytes
//               {-s, 0, +s}.  Writes use the canonical K-major 128B-swizzled
//               layout; afterwards these warps run the epilogue
//               (TMEM -> registers -> y).
// Every mbarrier wait is bounded; a wait that runs out raises the device
// status word, the CTA drains what it has in flight (bounded) and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int BM = 256, BN = 128, BK = 64, UM = 128;   // UM: rows per MMA
constexpr int kStages = 3;
constexpr int kASlice = BM * BK * 2;                        // 32 KB
constexpr int kBSlice = BN * BK * 2;                        // 16 KB
constexpr int kQsBytes = BN * kGroupBytes;                  // 26,624
constexpr int kScBytes = BN * kGroupBlocks * 2;             // 2,048
constexpr int kGroupBuf = kQsBytes + kScBytes;              // 28,672 = 28 * 1024
constexpr int kLutBytes = 2 * 256 * 16;                     // even / odd selector tables
constexpr int kThreads = 10 * 32;
constexpr int kExpWarp0 = 2, kExpThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 22;

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kASlice;
constexpr int kOffQ = kOffB + kStages * kBSlice;
constexpr int kOffLut = kOffQ + 2 * kGroupBuf;
constexpr int kOffBar = kOffLut + kLutBytes;
// barriers: a_full[S], b_full[S], empty[S], q_full[2], q_empty[2], acc
constexpr int kNumBars = 3 * kStages + 4 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;            // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bounded wait for phase `parity`.  Returns false when the limit ran out or
// (when `abort` is given) another role has already aborted the CTA.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if (abort && (i & 1023) == 1023 && *abort) return false;
  }
  return false;
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

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

// Byte offset of element (r, k) (k < 64) inside a 128-row, 64-wide fp16 tile
// in the canonical K-major 128B-swizzled layout.
__device__ __forceinline__ uint32_t sw128_off(int r, int k) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((k >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

// Selector tables.  PRMT picks each output byte from 8 source bytes; the
// per-block sources are {-s, 0, +s} as fp16 (bytes 0-1, 2-3, 4-5), so digit
// d = t + 1 of a weight selects bytes 2d and 2d + 1.  For a byte value v with
// digits d0..d4 (weights 5j .. 5j+4): an even-positioned byte (5j even) is
// emitted as pairs (d0,d1), (d2,d3) and a low half d4; an odd-positioned
// byte as a high half d0 and pairs (d1,d2), (d3,d4).  Entry = 4 words:
// {pair selector, pair selector, half selector, 0}; the straddling pair is
// the OR of the two half selectors.
__device__ __forceinline__ uint32_t sel_pair(uint32_t da, uint32_t db) {
  return (2 * da) | ((2 * da + 1) << 4) | ((2 * db) << 8) | ((2 * db + 1) << 12);
}

__device__ void build_luts(uint4* lut) {
  for (int i = threadIdx.x; i < 512; i += blockDim.x) {
    const uint32_t v = i & 255;
    uint32_t d[5], fprev = 0;
#pragma unroll
    for (int n = 0; n < 5; ++n) {  // digit n = floor(3^(n+1) v/256) - 3 floor(3^n v/256)
      const uint32_t p = n == 0 ? 3u : n == 1 ? 9u : n == 2 ? 27u : n == 3 ? 81u : 243u;
      const uint32_t fnext = (v * p) >> 8;
      d[n] = fnext - 3u * fprev;
      fprev = fnext;
    }
    lut[i] = i < 256 ? make_uint4(sel_pair(d[0], d[1]), sel_pair(d[2], d[3]),
                                  (2 * d[4]) | ((2 * d[4] + 1) << 4), 0u)
                     : make_uint4(sel_pair(d[1], d[2]), sel_pair(d[3], d[4]),
                                  ((2 * d[0]) | ((2 * d[0] + 1) << 4)) << 8, 0u);
  }
}

// Half h of one 128-weight block of one row: 64 fp16 values t * s written as
// 8 swizzled 16-byte chunks.  `win` holds the 16-byte-aligned 48 bytes that
// contain the block, which starts at byte `o` of the window.
template <int h, int o>
__device__ __forceinline__ void expand_half(const uint32_t win[12], uint32_t ta, uint32_t tb,
                                            const unsigned char* lut, unsigned char* bslice,
                                            int r) {
  auto byte_of = [&](int j) -> uint32_t {
    return __byte_perm(win[(o + j) >> 2], 0u, 0x4440u | ((o + j) & 3));
  };
  auto even = [&](int j) { return *reinterpret_cast<const uint4*>(lut + byte_of(j) * 16); };
  auto odd = [&](int j) { return *reinterpret_cast<const uint4*>(lut + 4096 + byte_of(j) * 16); };
  auto P = [&](uint32_t sel) { return __byte_perm(ta, tb, sel); };
  uint32_t out[32];
  int n = 0;
  if constexpr (h == 0) {
#pragma unroll
    for (int j = 0; j < 12; j += 2) {  // bytes 0..11: weights 0..59
      const uint4 e = even(j), q = odd(j + 1);
      out[n++] = P(e.x);
      out[n++] = P(e.y);
      out[n++] = P(e.z | q.z);
      out[n++] = P(q.x);
      out[n++] = P(q.y);
    }
    const uint4 e = even(12);  // weights 60..63
    out[n++] = P(e.x);
    out[n++] = P(e.y);
  } else {
    {
      const uint4 e = even(12), q = odd(13);  // weights 64..69
      out[n++] = P(e.z | q.z);
      out[n++] = P(q.x);
      out[n++] = P(q.y);
    }
#pragma unroll
    for (int j = 14; j < 24; j += 2) {  // bytes 14..23: weights 70..119
      const uint4 e = even(j), q = odd(j + 1);
      out[n++] = P(e.x);
      out[n++] = P(e.y);
      out[n++] = P(e.z | q.z);
      out[n++] = P(q.x);
      out[n++] = P(q.y);
    }
    const uint4 e = even(24), q = odd(25);  // weights 120..127 (byte 25 holds 3)
    out[n++] = P(e.x);
    out[n++] = P(e.y);
    out[n++] = P(e.z | q.z);
    out[n++] = P(q.x);
  }
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(bslice + sw128_off(r, 8 * c)) =
        make_uint4(out[4 * c], out[4 * c + 1], out[4 * c + 2], out[4 * c + 3]);
}

// The 8 blocks of one staged group for this thread's row and half, as fp16
// or (kBf16) bf16 values t * s.
template <bool kBf16, int h, int bb = 0>
__device__ __forceinline__ bool expand_group(const unsigned char* qrow, const uint16_t* srow,
                                             const unsigned char* lut, unsigned char* smem,
                                             uint64_t* empty, uint64_t* b_full, int g, int r,
                                             volatile int* abort_flag) {
  if constexpr (bb < kGroupBlocks) {
    constexpr int base16 = (kBlockBytes * bb) & ~15, o = (kBlockBytes * bb) & 15;
    uint32_t win[12];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint4 v = *reinterpret_cast<const uint4*>(qrow + base16 + 16 * i);
      win[4 * i] = v.x; win[4 * i + 1] = v.y; win[4 * i + 2] = v.z; win[4 * i + 3] = v.w;
    }
    uint32_t s16 = srow[bb];
    if constexpr (kBf16)  // the fp16 scale rounded to nearest-even bf16
      s16 = __bfloat16_as_ushort(__float2bfloat16_rn(__half2float(__ushort_as_half((unsigned short)s16))));
    // PRMT sources: bytes 0-1 = -s, 2-3 = 0, 4-5 = +s
    const uint32_t ta = (s16 ^ 0x8000u), tb = s16;
    const int kb = g * 16 + bb * 2 + h;
    const int s = kb % kStages, round = kb / kStages;
    if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1, abort_flag)) return false;
    expand_half<h, o>(win, ta, tb, lut, smem + kOffB + s * kBSlice, r);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive(&b_full[s]);
    return expand_group<kBf16, h, bb + 1>(qrow, srow, lut, smem, empty, b_full, g, r, abort_flag);
  }
  return true;
}

template <bool kBf16, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_s, void* __restrict__ y, int M, int N,
                   int K, int* status) {
  // No static shared variables: the dynamic window starts at offset 0, so the
  // declared 1024-byte alignment holds, and every access below stays a
  // shared-memory instruction (an address laundered through an integer
  // would turn them into generic ones).
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* a_full = bars;
  uint64_t* b_full = bars + kStages;
  uint64_t* empty = bars + 2 * kStages;
  uint64_t* q_full = bars + 3 * kStages;
  uint64_t* q_empty = q_full + 2;
  uint64_t* acc_full = q_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
  const unsigned char* lut = smem + kOffLut;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nk = K / BK;            // 64-wide slices
  const int ng = K / kRot;          // 1024-wide groups

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&b_full[s], kExpThreads / 2);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], kExpThreads);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  build_luts(reinterpret_cast<uint4*>(smem + kOffLut));
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
  pdl_wait();  // A may come from the previous kernel

  bool ok = true;
  int a_issued = 0;
  if (warp == 0) {
    // ---- TMA producer ----------------------------------------------------------
    if (lane == 0) {
      // packed weights run one 1024-wide group ahead of the A slices
      auto issue_group = [&](int g) {
        const int qb = g & 1;
        if (g >= 2 && !mbar_wait(&q_empty[qb], ((g >> 1) - 1) & 1, abort_flag)) return false;
        const uint32_t qdst = smem_u32(smem + kOffQ + qb * kGroupBuf);
        mbar_expect_tx(&q_full[qb], kGroupBuf);
        tma_2d(qdst, &map_q, g * kGroupBytes, n0, &q_full[qb]);
        tma_2d(qdst + kQsBytes, &map_s, g * kGroupBlocks, n0, &q_full[qb]);
        return true;
      };
      ok = issue_group(0) && (ng < 2 || issue_group(1));
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kStages, round = kb / kStages;
        if (kb % 16 == 0 && kb > 0 && kb / 16 + 1 < ng) ok = issue_group(kb / 16 + 1);
        if (!ok) break;
        if (round > 0) ok = mbar_wait(&empty[s], (round - 1) & 1, abort_flag);
        if (!ok) break;
        mbar_expect_tx(&a_full[s], kASlice);
        tma_2d(smem_u32(smem + kOffA + s * kASlice), &map_a, kb * BK, m0, &a_full[s]);
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
#pragma unroll
        for (int mh = 0; mh < 2; ++mh)
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // K = 16 per MMA: 32 bytes along the atom
            umma_f16<kBf16>(tmem + mh * BN, sw128_desc(a_addr + mh * (UM * 128) + 32 * kk),
                            sw128_desc(b_addr + 32 * kk), (kb | kk) != 0);
        umma_commit(&empty[s]);  // frees the slice once these MMAs have read it
      }
      umma_commit(acc_full);     // all MMAs issued by this thread
    }
  } else {
    // ---- B expansion: thread (row r, half h) ---------------------------------------
    const int t = threadIdx.x - 32 * kExpWarp0, r = t & (BN - 1), h = t >> 7;  // h: warp-uniform
    for (int g = 0; g < ng && ok; ++g) {
      const int qb = g & 1;
      ok = mbar_wait(&q_full[qb], (g >> 1) & 1, abort_flag);
      if (!ok) break;
      const unsigned char* qrow = smem + kOffQ + qb * kGroupBuf + r * kGroupBytes;
      const uint16_t* srow =
          reinterpret_cast<const uint16_t*>(smem + kOffQ + qb * kGroupBuf + kQsBytes) + r * 8;
      ok = h == 0 ? expand_group<kBf16, 0>(qrow, srow, lut, smem, empty, b_full, g, r, abort_flag)
                  : expand_group<kBf16, 1>(qrow, srow, lut, smem, empty, b_full, g, r, abort_flag);
      if (ok) mbar_arrive(&q_empty[qb]);
    }
  }
  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) atomicOr(status, kDevTimeout);
  }

  // ---- epilogue: warps 2-9; warp w reads TMEM lanes 32 (w % 4) .. + 31 of
  // accumulator (w - 2) / 4 -------------------------------------------------------------
  if (warp >= kExpWarp0) {
    const bool done = !*abort_flag && mbar_wait(acc_full, 0, abort_flag);
    if (done) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int q = warp & 3, mh = (warp - kExpWarp0) >> 2;
      const int row = m0 + mh * UM + 32 * q + lane;
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
              for (int i = 0; i < 32 && ncol + i < N; ++i) out[i] = __uint_as_float(v[i]);
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
              for (int i = 0; i < 32 && ncol + i < N; ++i)
                out[i] = (uint16_t)(pk[i >> 1] >> (16 * (i & 1)));
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

// ---- host side -------------------------------------------------------------------------
template <bool kBf16, bool kOutF32>
cudaError_t launch_t(const CUtensorMap& ma, const CUtensorMap& mq, const CUtensorMap& ms, void* y,
                     int M, int N, int K, int* status, cudaStream_t st) {
  auto kern = gemm_tc_kernel<kBf16, kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
  return launch_pdl(kern, grid, dim3(kThreads), (size_t)kSmemBytes, st, ma, mq, ms, y, M, N, K,
                    status);
}

}  // namespace

// Tensor-core GEMM for K % 1024 == 0 (cudaErrorNotSupported otherwise).
cudaError_t launch_gemm_tc(const uint8_t* wq, const uint16_t* scales, const void* x, Act x_t,
                           void* y, Act y_t, int64_t M, int64_t N, int64_t K, cudaStream_t st) {
  if (K % kRot != 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX ||
      (M + BM - 1) / BM > 65535)
    return cudaErrorNotSupported;
  cudaError_t e;
  const int64_t nblk = K / kBlockWeights, row_bytes = nblk * kBlockBytes;
  CUtensorMap ma, mq, ms;
  if ((e = encode_tma_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, K, M, K * 2, BK, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)  // box 64 x 256
    return e;
  if ((e = encode_tma_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, row_bytes, N, row_bytes,
                         kGroupBytes, BN, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  if ((e = encode_tma_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, nblk, N, nblk * 2,
                         kGroupBlocks, BN, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevice;
  const int m = (int)M, n = (int)N, k = (int)K;
  const bool bf = x_t == Act::BF16, f32 = y_t == Act::F32;
  if (bf && f32) return launch_t<true, true>(ma, mq, ms, y, m, n, k, status, st);
  if (bf) return launch_t<true, false>(ma, mq, ms, y, m, n, k, status, st);
  if (f32) return launch_t<false, true>(ma, mq, ms, y, m, n, k, status, st);
  return launch_t<false, false>(ma, mq, ms, y, m, n, k, status, st);
}

}  // namespace ptq

// k_gemv_tc.cu -- decode GEMV over PTQ1_0 weights at M = 1, with the
// multiply-adds on the tensor cores.
//
//   y[n] = sum_b s[n, b] * sum_{i<128} t[n, 128b + i] * x[128b + i]
//
// Why: the peel of "A 27B model in 5.5 GB: Bonsai ternary on Ferrox,
// locally" (section "What Ferrox does with it": digit n of a byte is
// floor(3^(n+1) u) - 3 floor(3^n u), u = byte/256) costs three or more SIMT
// instructions per weight, while a GB300 must consume a weight every ~1.3
// lane-instructions to keep up with HBM (the page notes the decode is
// arithmetic-bound even on an M2 Pro).  Here the CUDA cores only extract the
// floors, two per instruction pair, and the contraction runs on mma.sync.
//
// Arithmetic.  With 3^n u = f_n + phi_n (f_n its floor, phi_n its fraction),
// the digit is d_n = floor(3 phi_n) = 3 phi_n - phi_{n+1}, so a byte
// contributes
//   sum_{n<5} d_n x_n = 3 phi_0 x_0 + sum_{j=1..4} phi_j (3 x_j - x_{j-1})
//                       - phi_5 x_4,          phi_0 = u = byte / 256,
// and sum_i t_i x_i = sum d x - E_x (E_x = block sum of x).  The fractions
// keep every partial sum the size of the result (the floor form
// sum f_j (x_{j-1} - 3 x_j) cancels about 400-fold, more than the tensor
// core's truncating fp32 accumulation tolerates).  A 32-bit integer
// multiply of (b_A | b_B << 16) by 3^j leaves (3^j b mod 256) = 256 phi_j
// in the LOW byte of each 16-bit lane (3^5 * 255 < 2^16); one byte permute
// moves the two into the low bytes of two fp16 values with zero high bytes,
// the exact fp16 subnormals phi * 2^-16.  The spread register itself is the
// j = 0 operand (b * 2^-24 = u * 2^-16).  These are the A operand of an
// m16n8k16 f16 MMA (16 weight rows x 16 terms).  The B operand holds the
// activation coefficients (3 x_0; 3 x_j - x_{j-1}; -x_4) as two fp16 limbs
// (hi + lo) of c * 2^S_b, with S_b a power of two per block chosen from the
// block's largest |x|; hi + lo carries 22 bits of c.  The accumulator is
// fp32, and  dot_b = 2^(16 - S_b) * (D_hi + D_lo) - E_x.
//
// Layout of the work.  A "slab" is 16 weight rows, a "group" 1024 weights (8
// blocks = 208 bytes per row).  For one (slab, group) unit a warp holds rows
// g and g+8 in the lanes of quad g (g = lane / 4); lane t = lane % 4 of the
// quad owns blocks 2t and 2t+1 of the group (bytes 52t..52t+51: 13 aligned
// words).  In each k-tile the 16 terms are four from each lane's current
// block; B puts lane t's coefficients in columns 2t (hi) and 2t+1 (lo) only,
// so D[r][2t], D[r][2t+1] hold exactly lane t's block for row r -- the
// registers that lane already owns -- and the block scale is applied in
// fp32 after the block's 39 k-tiles (154 terms + 2 padding).  Per term the
// CUDA cores spend about 0.85 instructions.
//
// Launch.  Programmatic dependent launch: the barrier set-up and the first
// weight loads run while the previous kernel (the rotation that produces x)
// is still finishing; griddepcontrol.wait precedes every read of x.
//
// Data movement.  Each warp streams its own units: lane 0 issues 2-D TMA
// loads (16 rows x 208 bytes of trits, 16 rows x 8 scales) into a private
// ring of shared-memory stages that completes on an mbarrier.  The
// coefficient table is built once per CTA (persistent grid, one CTA per SM).
// Per-unit partial sums go to shared memory and are reduced per slab in a
// fixed order, so results are bitwise reproducible.  Every mbarrier wait is
// bounded; a wait that runs out raises the device status word and the CTA
// stops issuing work.
#include <cuda.h>
#include <cuda_fp16.h>
#include <mutex>

#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int kStages = 2;                 // TMA stages per warp
constexpr int kSlabRows = 16;
constexpr int kTileQs = kSlabRows * kGroupBytes;          // 3328 bytes
constexpr int kTileSc = kSlabRows * kGroupBlocks * 2;     // 256 bytes
constexpr int kStageBytes = kTileQs + kTileSc;            // 3584 = 28 * 128
constexpr int kPairs = 78;                 // term pairs per block (77 + 1 zero pad)
constexpr int kKt = kPairs / 2;            // k-tiles per block
constexpr int kBlkTab = kKt * 16 + 8;      // bytes of B fragments per block (+ bank pad)
constexpr uint32_t kWaitLimit = 1u << 22;  // try_wait polls before giving up

// ---- the pair-slot table: one definition drives both the A producer and
// the coefficient builder.  Per block parity p (0: block starts at word 0 of
// the lane's 13-word window, 1: at byte 26) there are 78 slots in k order:
// s < 72: regular spread r = s / 6 at power j = s % 6 (bytes a, b of the
// block); s = 72..75: the pair (24, 25) at j = 0..3 (byte 25 holds three
// trits, so j = 4, 5 carry zero coefficients and are left out); s = 76:
// byte 24 at j = 4 and j = 5; s = 77: padding (A = 0, B = 0).
struct Slot {
  int src;   // index into the 28 spread registers of the window (-1: padding)
  int a, b;  // block-relative byte of term A and term B
  int ja, jb;
};

__host__ __device__ constexpr Slot slot_of(int p, int s) {
  // Regular spreads of each parity, as (spread index, byte a, byte b):
  //   even: window words 0..5 -> spreads 2i (bytes 4i, 4i+2), 2i+1 (4i+1, 4i+3)
  //   odd : spread 14 -> (0, 1); words 7..11 -> spreads 15 + 2(i-7) and
  //         16 + 2(i-7) (bytes 4i-26, 4i-24 / 4i-25, 4i-23); spread 25 -> (22, 23)
  if (s < 72) {
    const int r = s / 6, j = s % 6;
    if (p == 0) {
      const int i = r / 2;
      return (r % 2 == 0) ? Slot{r, 4 * i, 4 * i + 2, j, j} : Slot{r, 4 * i + 1, 4 * i + 3, j, j};
    }
    if (r == 0) return Slot{14, 0, 1, j, j};
    if (r == 11) return Slot{25, 22, 23, j, j};
    const int q = r - 1, i = 7 + q / 2;
    return (q % 2 == 0) ? Slot{15 + q, 4 * i - 26, 4 * i - 24, j, j}
                        : Slot{15 + q, 4 * i - 25, 4 * i - 23, j, j};
  }
  if (s < 76) return Slot{p == 0 ? 12 : 26, 24, 25, s - 72, s - 72};
  if (s == 76) return Slot{p == 0 ? 13 : 27, 24, 24, 4, 5};
  return Slot{-1, 0, 0, 0, 0};
}

// Multiplier of slot s: the scalar 3^j for a two-byte spread (each 16-bit
// lane is multiplied on its own, 3^5 * 255 < 2^16, no carry between lanes);
// 81 | 243 << 16 for the single byte 24, whose lanes become 81 b and 243 b.
__host__ __device__ constexpr uint32_t mult_of(int p, int s) {
  return s == 76 ? (81u | (243u << 16))
                 : (slot_of(p, s).ja == 1 ? 3u : slot_of(p, s).ja == 2 ? 9u
                    : slot_of(p, s).ja == 3 ? 27u : slot_of(p, s).ja == 4 ? 81u : 243u);
}

// ---- small PTX helpers ---------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bounded wait for phase `parity`; false if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
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
  }
  return false;
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_f16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// A operand of slot s for one row: two fp16 subnormals (256 phi) * 2^-24.
// S holds the 14 spreads of the block (index = src - 14 p).
template <int p, int s>
__device__ __forceinline__ uint32_t a_slot(const uint32_t S[14]) {
  constexpr Slot sl = slot_of(p, s);
  if constexpr (sl.src < 0) return 0u;                              // padding
  else if constexpr (sl.ja == 0) return S[sl.src - 14 * p];         // phi_0 = u: the bytes
  else return __byte_perm(S[sl.src - 14 * p] * mult_of(p, s), 0u, 0x4240u);  // 256 phi_j
}

// The 14 spread registers of one block (see slot_of; index = src - 14 p)
// from the 7 words that hold it: words 0..6 of the window for p = 0
// (word 6 carries bytes 24, 25), words 6..12 for p = 1 (word 6 carries the
// block's bytes 0, 1).
template <int p>
__device__ __forceinline__ void spreads(const uint32_t w[7], uint32_t S[14]) {
  if constexpr (p == 0) {
#pragma unroll
    for (int i = 0; i < 6; ++i) {
      S[2 * i] = __byte_perm(w[i], 0, 0x4240);
      S[2 * i + 1] = __byte_perm(w[i], 0, 0x4341);
    }
    S[12] = __byte_perm(w[6], 0, 0x4140);
    S[13] = __byte_perm(w[6], 0, 0x4440);
  } else {
    S[0] = __byte_perm(w[0], 0, 0x4342);
#pragma unroll
    for (int i = 1; i < 6; ++i) {
      S[2 * i - 1] = __byte_perm(w[i], 0, 0x4240);
      S[2 * i] = __byte_perm(w[i], 0, 0x4341);
    }
    S[11] = __byte_perm(w[6], 0, 0x4140);
    S[12] = __byte_perm(w[6], 0, 0x4342);
    S[13] = __byte_perm(w[6], 0, 0x4442);
  }
}

// The 39 k-tiles of one block: A from the lane's spreads, B from the table.
// Two accumulator chains (even and odd k-tiles) halve the MMA dependency
// chain; the caller adds them.
template <int p, int kt = 0>
__device__ __forceinline__ void block_mma(float d[2][4], const uint32_t S0[14],
                                          const uint32_t S1[14], const uint2* bt) {
  if constexpr (kt < kKt) {
    const uint2 bv = bt[kt * 2];
    mma_f16(d[kt & 1], a_slot<p, 2 * kt>(S0), a_slot<p, 2 * kt>(S1), a_slot<p, 2 * kt + 1>(S0),
            a_slot<p, 2 * kt + 1>(S1), bv.x, bv.y);
    block_mma<p, kt + 1>(d, S0, S1, bt);
  }
}

struct Params {
  int N, K, G, nblk, slabs;
};

// x value k of the block held by the warp as one float4 per lane (0 past 127)
__device__ __forceinline__ float x_at(const float4& v, int k) {
  const int src = (k < kBlockWeights ? k : 0) >> 2;
  const float a = __shfl_sync(0xffffffffu, v.x, src), b = __shfl_sync(0xffffffffu, v.y, src);
  const float c = __shfl_sync(0xffffffffu, v.z, src), d = __shfl_sync(0xffffffffu, v.w, src);
  const float r = (k & 3) == 0 ? a : (k & 3) == 1 ? b : (k & 3) == 2 ? c : d;
  return k < kBlockWeights ? r : 0.0f;
}

// coefficient of term (byte, j): 3 x_0 (j = 0), 3 x_j - x_{j-1} (j = 1..4),
// -x_4 (j = 5), where x_n is x[5 byte + n] of the block
__device__ __forceinline__ float coef_at(const float4& v, int byte, int j) {
  const int k = 5 * byte;
  const float hi = x_at(v, k + (j < 5 ? j : 4));
  const float lo = x_at(v, k + (j > 0 ? j - 1 : 0));
  return j == 0 ? 3.0f * hi : j == 5 ? -hi : fmaf(3.0f, hi, -lo);
}

template <int kWarps>
__global__ void __launch_bounds__(kWarps * 32, 1)
    gemv_m1_tc_kernel(const __grid_constant__ CUtensorMap map_qs,
                      const __grid_constant__ CUtensorMap map_sc, const float* __restrict__ x,
                      float* __restrict__ y, Params P, int* status) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;

  // this CTA's slabs and units
  const int s0 = (int)((long long)blockIdx.x * P.slabs / gridDim.x);
  const int s1 = (int)((long long)(blockIdx.x + 1) * P.slabs / gridDim.x);
  const int units = (s1 - s0) * P.G;

  // shared memory carve-up
  unsigned char* stages = smem;                                              // per warp ring
  unsigned char* btab = stages + (size_t)kWarps * kStages * kStageBytes;     // B fragments
  // btab holds nblk blocks of B fragments plus one all-zero block that the
  // lanes holding no B of a k-tile read instead (no predication)
  float* etab = reinterpret_cast<float*>(btab + (size_t)(P.nblk + 1) * kBlkTab);  // E_x, scale
  float* part = etab + 2 * P.nblk;                                          // units x 16
  uint64_t* bars = reinterpret_cast<uint64_t*>(part + (size_t)units * kSlabRows);
  uint64_t* mybar = bars + warp * kStages;
  int& s_abort = *reinterpret_cast<int*>(bars + kWarps * kStages);
  unsigned char* mystage = stages + (size_t)warp * kStages * kStageBytes;

  if (threadIdx.x == 0) s_abort = 0;
  int issued = 0;  // units this warp has put in flight (lane 0's count)
  if (lane == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&mybar[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  auto issue = [&](int u, int stage) {  // lane 0 only
    const int slab = s0 + u / P.G, grp = u % P.G;
    unsigned char* dst = mystage + stage * kStageBytes;
    mbar_expect_tx(&mybar[stage], kStageBytes);
    tma_2d(dst, &map_qs, grp * kGroupBytes, slab * kSlabRows, &mybar[stage]);
    tma_2d(dst + kTileQs, &map_sc, grp * kGroupBlocks, slab * kSlabRows, &mybar[stage]);
  };
  // the first kStages units of this warp are in flight while the table is built
  if (lane == 0)
    for (int k = 0; k < kStages; ++k) {
      const int u = warp + k * kWarps;
      if (u < units) {
        issue(u, k);
        ++issued;
      }
    }

  // ---- coefficient table (once per CTA) ----------------------------------------
  for (int i = threadIdx.x; i < kBlkTab / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(btab + (size_t)P.nblk * kBlkTab)[i] = 0u;
  // x may be written by the previous kernel in the stream: everything above
  // (barrier set-up, weight prefetch) ran before it finished.
  pdl_wait();
  // One warp per block: one 16-byte load per lane, then shuffles.  2^S_b from
  // the block's largest |x| (|c| <= 4 max|x|, kept below 2^15).  The next
  // block's load is issued before this one is processed.
  const float4* x4 = reinterpret_cast<const float4*>(x);
  float4 v_next = warp < P.nblk ? x4[(size_t)warp * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int b = warp; b < P.nblk; b += kWarps) {
    const float4 v = v_next;
    if (b + kWarps < P.nblk) v_next = x4[(size_t)(b + kWarps) * 32 + lane];
    float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    float sx = (v.x + v.y) + (v.z + v.w);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      sx += __shfl_xor_sync(0xffffffffu, sx, o);
    }
    int e = 0;
    frexpf(4.0f * m, &e);                   // 4m < 2^e
    const int S = m > 0.0f ? 15 - e : 0;    // c * 2^S < 2^15
    const float up = ldexpf(1.0f, S);
    if (lane == 0) {
      etab[2 * b] = sx;                       // E_x
      etab[2 * b + 1] = ldexpf(1.0f, 16 - S); // undoes 2^S and the 2^-16 of A
    }
    const int p = b & 1;
#pragma unroll
    for (int it = 0; it < (kPairs + 31) / 32; ++it) {
      const int s = lane + 32 * it;
      const Slot sl = slot_of(p, s < kPairs ? s : 0);
      const float ca = coef_at(v, sl.a, sl.ja) * up, cb = coef_at(v, sl.b, sl.jb) * up;
      if (s >= kPairs) continue;
      const bool pad = sl.src < 0;
      const __half ha = __float2half_rn(pad ? 0.0f : ca), hb = __float2half_rn(pad ? 0.0f : cb);
      const __half la = __float2half_rn(pad ? 0.0f : ca - __half2float(ha));
      const __half lb = __float2half_rn(pad ? 0.0f : cb - __half2float(hb));
      // entry [b][kt][limb] = {slot 2kt: A, B; slot 2kt+1: A, B}, 8 bytes
      __half* en = reinterpret_cast<__half*>(btab + (size_t)b * kBlkTab) + (s >> 1) * 8 + (s & 1) * 2;
      en[0] = ha; en[1] = hb;   // limb 0
      en[4] = la; en[5] = lb;   // limb 1
    }
  }
  __syncthreads();
  pdl_release();  // the next kernel may start its own prologue

  // ---- main loop: this warp's units -----------------------------------------------
  const bool b_lane = (g >> 1) == t;  // holds non-zero B: column g in {2t, 2t+1}
  const int limb = g & 1;
  const uint2* zero_b = reinterpret_cast<const uint2*>(btab + (size_t)P.nblk * kBlkTab);
  int k = 0;
  for (int u = warp; u < units; u += kWarps, ++k) {
    const int stage = k % kStages;
    if (!mbar_wait(&mybar[stage], (k / kStages) & 1)) {
      if (lane == 0) atomicOr(status, kDevTimeout);
      s_abort = 1;
      break;
    }
    const int grp = u % P.G;
    const unsigned char* tile = mystage + stage * kStageBytes;
    const unsigned char* row0 = tile + g * kGroupBytes + 52 * t;
    const unsigned char* row1 = tile + (g + 8) * kGroupBytes + 52 * t;
    const uint32_t sc0 = *reinterpret_cast<const uint32_t*>(tile + kTileQs + g * 16 + 4 * t);
    const uint32_t sc1 = *reinterpret_cast<const uint32_t*>(tile + kTileQs + (g + 8) * 16 + 4 * t);
    float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      uint32_t S0[14], S1[14];
      {
        uint32_t w0[7], w1[7];
#pragma unroll
        for (int i = 0; i < 7; ++i) {
          w0[i] = reinterpret_cast<const uint32_t*>(row0)[6 * p + i];
          w1[i] = reinterpret_cast<const uint32_t*>(row1)[6 * p + i];
        }
        if (p == 0) {
          spreads<0>(w0, S0);
          spreads<0>(w1, S1);
        } else {
          spreads<1>(w0, S0);
          spreads<1>(w1, S1);
        }
      }
      const int gb = grp * kGroupBlocks + 2 * t + p;          // this lane's block
      const int gbB = grp * kGroupBlocks + 2 * (g >> 1) + p;  // block whose B this lane holds
      const uint2* bt =
          b_lane ? reinterpret_cast<const uint2*>(btab + (size_t)gbB * kBlkTab) + limb : zero_b;
      float dd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if (p == 0)
        block_mma<0>(dd, S0, S1, bt);
      else
        block_mma<1>(dd, S0, S1, bt);
      const float d[4] = {dd[0][0] + dd[1][0], dd[0][1] + dd[1][1], dd[0][2] + dd[1][2],
                          dd[0][3] + dd[1][3]};
      const float inv = etab[2 * gb + 1], E = etab[2 * gb];
      const float s_0 = __half2float(__ushort_as_half((unsigned short)(sc0 >> (16 * p))));
      const float s_1 = __half2float(__ushort_as_half((unsigned short)(sc1 >> (16 * p))));
      y0 = fmaf(s_0, fmaf(d[0] + d[1], inv, -E), y0);
      y1 = fmaf(s_1, fmaf(d[2] + d[3], inv, -E), y1);
    }
    __syncwarp();  // every lane has consumed the stage
    if (lane == 0 && u + kStages * kWarps < units) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(u + kStages * kWarps, stage);  // refill this stage
      ++issued;
    }
    y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
    y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
    y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
    if (t == 0) {
      part[u * kSlabRows + g] = y0;
      part[u * kSlabRows + g + 8] = y1;
    }
  }
  __syncthreads();
  if (s_abort) {
    // let this warp's copies still in flight land (bounded) before the CTA exits
    if (lane == 0)
      for (int kk = k; kk < issued; ++kk) (void)mbar_wait(&mybar[kk % kStages], (kk / kStages) & 1);
    return;
  }
  // fixed-order reduction over the groups of each slab
  for (int r = threadIdx.x; r < (s1 - s0) * kSlabRows; r += blockDim.x) {
    const int sl = r / kSlabRows, row = (s0 + sl) * kSlabRows + r % kSlabRows;
    if (row >= P.N) continue;
    float acc = 0.0f;
    for (int gp = 0; gp < P.G; ++gp) acc += part[(sl * P.G + gp) * kSlabRows + r % kSlabRows];
    y[row] = acc;
  }
}

// ---- host side ---------------------------------------------------------------------
int g_sms[64];

}  // namespace

size_t gemv_m1_tc_smem(int64_t N, int64_t K, int grid, int warps) {
  const int64_t nblk = K / kBlockWeights, G = K / kRot;
  const int64_t slabs = (N + kSlabRows - 1) / kSlabRows;
  const int64_t max_units = ((slabs + grid - 1) / grid) * G;
  return (size_t)warps * kStages * kStageBytes + (size_t)(nblk + 1) * kBlkTab + 8 * nblk +
         (size_t)max_units * kSlabRows * 4 + warps * kStages * 8 + 16;
}

// Returns cudaErrorNotSupported when the shape does not fit this kernel (the
// caller then uses the SIMT kernel).  20 warps per CTA when the shared memory
// allows it, else 16.
cudaError_t launch_gemv_m1_tc(const uint8_t* wq, const uint16_t* scales, const float* x, float* y,
                              int64_t N, int64_t K, cudaStream_t st) {
  if (K % kRot != 0 || N > INT32_MAX / 2 || K > (1 << 24)) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (g_sms[dev] == 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemv_m1_tc_kernel<20>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gemv_m1_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               227 * 1024);
    if (e != cudaSuccess) return e;
    g_sms[dev] = sms;
  }
  const int slabs = (int)((N + kSlabRows - 1) / kSlabRows);
  const int grid = slabs < g_sms[dev] ? slabs : g_sms[dev];
  int warps = 20;
  size_t smem = gemv_m1_tc_smem(N, K, grid, warps);
  if (smem > 227 * 1024) {
    warps = 16;
    smem = gemv_m1_tc_smem(N, K, grid, warps);
  }
  if (smem > 227 * 1024) return cudaErrorNotSupported;
  const int64_t nblk = K / kBlockWeights, row_bytes = nblk * kBlockBytes;
  CUtensorMap mq, ms;
  if ((e = encode_tma_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, row_bytes, N, row_bytes,
                         kGroupBytes, kSlabRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  if ((e = encode_tma_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, nblk, N, nblk * 2,
                         kGroupBlocks, kSlabRows, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevice;
  Params P{(int)N, (int)K, (int)(K / kRot), (int)nblk, slabs};
  if (warps == 20)
    return launch_pdl(gemv_m1_tc_kernel<20>, dim3(grid), dim3(20 * 32), smem, st, mq, ms, x, y, P,
                      status);
  return launch_pdl(gemv_m1_tc_kernel<16>, dim3(grid), dim3(16 * 32), smem, st, mq, ms, x, y, P,
                    status);
}

}  // namespace ptq

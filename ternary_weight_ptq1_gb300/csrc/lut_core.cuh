// lut_core.cuh -- the pieces of the table-lookup decode GEMV that more than
// one kernel uses: the shared-memory layout of the lane tables and of the
// weight ring, the signed rotation of one 1024-block, the table build, and
// the per-lane lookup of a word with its block scales.  Included by the
// stand-alone GEMV (k_gemv_lut.cu) and by the persistent decode stack
// (k_stack_decode.cu); every definition has internal linkage.
//
// The method is described in k_gemv_lut.cu: a PTQ1_0 byte's contribution
// sum_{i<5} t_i x_{5q+i} depends only on the byte and the five activations at
// its position ("A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally",
// section "What Bonsai is"), so it is tabulated for all 256 byte values.
#pragma once

#include <cuda_fp16.h>

#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kChunkWords = 32;            // one word per lane
constexpr int kXFloats = 2 * kRot;         // a chunk touches at most 6 blocks = 768
                                           // weights, inside at most two 1024-blocks
constexpr uint32_t kTab = 0x10000u;        // the tables' offset in the shared window
constexpr uint32_t kTabEnd = 0x30000u;     // 4 positions x 32 lanes x 256 x 4 B

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// The tables' shared address for a CTA whose dynamic shared memory starts at
// `raw`: kTab into its shared window.  The window starts at 0, or, for the
// CTA of rank r in a cluster, at r x 16 MB; either way the low 16 bits of the
// table addresses are free for the byte a lookup puts in bits 8-15.
__device__ __forceinline__ uint32_t table_base(uint32_t raw) { return (raw & 0xFFFF0000u) + kTab; }

__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds_f32x4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// Per-lane constants of the main loop.
struct Lanes {
  uint32_t lb0, lb1, lb2, lb3;  // table address bytes of positions 0..3
  uint32_t ssel;                // byte selector that puts s[bA], s[bB] low/high
  uint32_t red;                 // this warp's reduction buffer
  uint32_t wrow, srow;          // words per row of trits and of scales
};

template <int R>
__device__ __forceinline__ void build_entries(const float (&A)[9], const float (&B)[27],
                                              uint32_t dst) {
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    constexpr int e0 = 64 * R;
    const int e = e0 + i;
    const int v = (243 * e) >> 8;  // the five digits the peel reads from byte e
    sts_f32(dst + 256u * (uint32_t)e, A[v / 27] + B[v % 27]);
  }
}

// Entries e = 64 R .. 64 R + 63 of one PQ2_0 table: a byte holds four 2-bit
// codes, weights 4q..4q+3 from the low bits up, so T[e] = Lo[e & 15] +
// Hi[e >> 4] with Lo / Hi the sums over the low / high two codes.
template <int R>
__device__ __forceinline__ void build_entries_pq2(const float (&Lo)[16], const float (&Hi)[16],
                                                  uint32_t dst) {
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    constexpr int e0 = 64 * R;
    const int e = e0 + i;
    sts_f32(dst + 256u * (uint32_t)e, Lo[e & 15] + Hi[e >> 4]);
  }
}

// The signed rotation of one 1024-block of x by the 256 threads of 8 warps
// (g8: thread index within them), written to xs_blk (1024 floats):
//   xs_blk[j] = (1/32) sum_i (-1)^popcount(i & j) s[i] x[i]
// ("What Bonsai is": a 1024-wide butterfly with a sign pattern; sign first,
// then the Sylvester-ordered Hadamard butterfly).  load(g8) returns elements
// 4 g8 .. 4 g8 + 3 of the block.  Bits 0-1 of the index are done in
// registers, bits 2-6 across the lanes of a warp, bits 7-9 in registers after
// a transpose through `exch` (1024 floats).  The caller synchronises the 8
// warps around it with bar(); `bar` is that barrier.
template <typename Load, typename Bar>
__device__ __forceinline__ void rotate_block(Load load, const int8_t* __restrict__ s,
                                             uint32_t exch, uint32_t xs_blk, int g8, Bar bar) {
  const int lane = g8 & 31;
  const float4 xv = load(g8);
  const uint32_t sv = reinterpret_cast<const uint32_t*>(s)[g8];
  float v[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if ((int8_t)(sv >> (8 * i)) < 0) v[i] = -v[i];
  // bits 0, 1
  float a = v[0] + v[1], b = v[0] - v[1], c = v[2] + v[3], d = v[2] - v[3];
  v[0] = a + c; v[1] = b + d; v[2] = a - c; v[3] = b - d;
  // bits 2..6: the lane bits
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool up = lane & m;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], m);
      v[i] = up ? o - v[i] : v[i] + o;
    }
  }
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(exch + 16u * (uint32_t)g8),
               "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3])
               : "memory");
  bar();
  if (g8 < 128) {  // bits 7..9: elements g8 + 128 k, k = 0..7
    float w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = lds_f32(exch + 4u * (uint32_t)(g8 + 128 * k));
#pragma unroll
    for (int m = 1; m < 8; m <<= 1)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (!(k & m)) {
          const float p = w[k], q = w[k + m];
          w[k] = p + q;
          w[k + m] = p - q;
        }
#pragma unroll
    for (int k = 0; k < 8; ++k) sts_f32(xs_blk + 4u * (uint32_t)(g8 + 128 * k), w[k] * 0.03125f);
  }
}

// The lane tables of a chunk (words ws.. of every row) from the activations
// staged at `xs` (xs[0] is weight index xbase).  Warp w builds quarter w / 4
// of the entries of position w % 4 of every lane's word; lanes past the
// chunk (`live` false) get all-zero tables.  All threads of the CTA take part.
// kPQ2: the weights are PQ2_0 (32 bytes per block, four 2-bit codes a byte).
template <bool kPQ2 = false>
__device__ __forceinline__ void build_tables(int ws, bool live, uint32_t xs, int xbase,
                                             uint32_t tab) {
  constexpr int kBB = kPQ2 ? 32 : kBlockBytes;  // bytes per block
  const int L = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if constexpr (kPQ2) {
    const int j = warp & 3;
    const int Pj = 4 * (ws + L) + j;
    const int b = Pj / kBB, q = Pj % kBB;
    float xv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      xv[i] = live ? lds_f32(xs + 4u * (uint32_t)(b * kBlockWeights + 4 * q + i - xbase)) : 0.0f;
    float Lo[16], Hi[16];
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      // code c contributes (c - 1) x; code 3 (never written) gives 2 x
      const float c0 = (float)((n & 3) - 1), c1 = (float)(((n >> 2) & 3) - 1);
      Lo[n] = fmaf(c1, xv[1], c0 * xv[0]);
      Hi[n] = fmaf(c1, xv[3], c0 * xv[2]);
    }
    const uint32_t dst = tab + 0x10000u * (uint32_t)(j >> 1) + 128u * (uint32_t)(j & 1) + 4u * L;
    switch (warp >> 2) {
      case 0: build_entries_pq2<0>(Lo, Hi, dst); break;
      case 1: build_entries_pq2<1>(Lo, Hi, dst); break;
      case 2: build_entries_pq2<2>(Lo, Hi, dst); break;
      default: build_entries_pq2<3>(Lo, Hi, dst); break;
    }
  } else {
    // warp -> (position j of every lane's word, quarter R of the entries)
    const int j = warp & 3;
    const int Pj = 4 * (ws + L) + j;
    const int b = Pj / kBlockBytes, q = Pj % kBlockBytes;
    float xv[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      const bool in = live && 5 * q + i < kBlockWeights;  // byte 25 holds three trits
      xv[i] = in ? lds_f32(xs + 4u * (uint32_t)(b * kBlockWeights + 5 * q + i - xbase)) : 0.0f;
    }
    float A[9], B[27];
#pragma unroll
    for (int a = 0; a < 9; ++a) {
      // digits d0 = a / 3, d1 = a % 3 contribute (d - 1) x
      const int d0 = a / 3 - 1, d1 = a % 3 - 1;
      const float t0 = d0 > 0 ? xv[0] : (d0 < 0 ? -xv[0] : 0.0f);
      A[a] = d1 > 0 ? t0 + xv[1] : (d1 < 0 ? t0 - xv[1] : t0);
    }
#pragma unroll
    for (int bb = 0; bb < 27; ++bb) {
      const int d2 = bb / 9 - 1, d3 = (bb / 3) % 3 - 1, d4 = bb % 3 - 1;
      float t = d2 > 0 ? xv[2] : (d2 < 0 ? -xv[2] : 0.0f);
      t = d3 > 0 ? t + xv[3] : (d3 < 0 ? t - xv[3] : t);
      B[bb] = d4 > 0 ? t + xv[4] : (d4 < 0 ? t - xv[4] : t);
    }
    const uint32_t dst = tab + 0x10000u * (uint32_t)(j >> 1) + 128u * (uint32_t)(j & 1) + 4u * L;
    switch (warp >> 2) {
      case 0: build_entries<0>(A, B, dst); break;
      case 1: build_entries<1>(A, B, dst); break;
      case 2: build_entries<2>(A, B, dst); break;
      default: build_entries<3>(A, B, dst); break;
    }
  }
}

// The rotation blocks a chunk (words [ws, we) of every row) touches: the
// first is f0, the last f1 (one or two of them).
template <bool kPQ2 = false>
__device__ __forceinline__ void chunk_rot_blocks(int ws, int we, int* f0, int* f1) {
  constexpr int kBB = kPQ2 ? 32 : kBlockBytes;
  const int bx0 = (4 * ws) / kBB, bx1 = (4 * we - 1) / kBB;
  *f0 = bx0 * kBlockWeights / kRot;
  *f1 = (bx1 * kBlockWeights + kBlockWeights - 1) / kRot;
}

// The activations a chunk (words [ws, we) of every row) touches, rotated
// first when `signs` is given, staged at `xs`; then the lane tables.  All
// threads of the CTA take part; `exch` is 8 KB of scratch for the rotation.
template <bool kPQ2 = false>
__device__ __forceinline__ void stage_tables(const float* __restrict__ x,
                                             const int8_t* __restrict__ signs, int ws, int we,
                                             bool live, uint32_t exch, uint32_t xs,
                                             uint32_t tab) {
  constexpr int kBB = kPQ2 ? 32 : kBlockBytes;  // bytes per block
  const int warp = threadIdx.x >> 5;
  int xbase;  // weight index of xs[0]
  if (signs == nullptr) {
    const int bx0 = (4 * ws) / kBB, bx1 = (4 * we - 1) / kBB;
    xbase = bx0 * kBlockWeights;
    const int nx = (bx1 - bx0 + 1) * kBlockWeights;  // <= 6 * 128
    for (int i = threadIdx.x; i < nx; i += kThreads)
      sts_f32(xs + 4u * (uint32_t)i, x[(size_t)xbase + i]);
  } else {
    // the rotation blocks that hold this chunk's weights: one or two, one per
    // half of the CTA
    int f0, f1;
    chunk_rot_blocks<kPQ2>(ws, we, &f0, &f1);
    xbase = f0 * kRot;
    const int half = warp >> 3, g8 = threadIdx.x & 255;
    auto bar = [half]() {
      asm volatile("bar.sync %0, 256;" ::"r"(1 + half) : "memory");
    };
    if (f0 + half <= f1) {
      const size_t off = (size_t)(f0 + half) * kRot;
      const float4* xb = reinterpret_cast<const float4*>(x + off);
      rotate_block([xb](int i) { return xb[i]; }, signs + off, exch + (uint32_t)(half * kRot * 4),
                   xs + (uint32_t)(half * kRot * 4), g8, bar);
    }
  }
  __syncthreads();
  build_tables<kPQ2>(ws, live, xs, xbase, tab);
}

constexpr int kBoxRows = 16;                          // rows per box = per batch
constexpr int kBoxScaleWords = 8;                     // scale words per row in a box
constexpr int kSlotTrits = kBoxRows * kChunkWords * 4;     // 2048
constexpr int kSlotBytes = kSlotTrits + kBoxRows * kBoxScaleWords * 4;  // 2560
constexpr int kSlotsPerWarp = 2;
constexpr int kSlots = kWarps * kSlotsPerWarp;       // 32
constexpr int kLowSlots = 18;                        // below the tables; the rest above them
constexpr int kExchBytes = 2 * kRot * 4;             // rotation scratch (two blocks)
constexpr int kBarOff = kExchBytes + kXFloats * 4;   // after the exchange and x
constexpr int kRingOff = (kBarOff + kSlots * 8 + 127) / 128 * 128;
constexpr size_t kSmemTma = 227 * 1024;               // the whole window
static_assert(kTabEnd + (kSlots - kLowSlots) * kSlotBytes <= kSmemTma, "upper ring fits");

__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ float lane_value(uint32_t w, uint32_t sw, const Lanes& ln) {
  const uint32_t a0 = __byte_perm(w, ln.lb0, 0x7604), a1 = __byte_perm(w, ln.lb1, 0x7614);
  const uint32_t a2 = __byte_perm(w, ln.lb2, 0x7624), a3 = __byte_perm(w, ln.lb3, 0x7634);
  const uint32_t s2 = __byte_perm(sw, 0u, ln.ssel);
  const float t0 = lds_f32(a0), t1 = lds_f32(a1), t2 = lds_f32(a2), t3 = lds_f32(a3);
  const float sA = __half2float(__ushort_as_half((unsigned short)(s2 & 0xffffu)));
  const float sB = __half2float(__ushort_as_half((unsigned short)(s2 >> 16)));
  return fmaf(t2 + t3, sB, (t0 + t1) * sA);
}

// lo/hi: this lane's values of two rows; the lane keeps the one its bit m
// selects and adds the partner lane's copy of it
__device__ __forceinline__ float fold(float lo, float hi, bool up, int m) {
  const float keep = up ? hi : lo, send = up ? lo : hi;
  return keep + __shfl_xor_sync(0xffffffffu, send, m);
}

}  // namespace
}  // namespace ptq

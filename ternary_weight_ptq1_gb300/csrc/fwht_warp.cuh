// fwht_warp.cuh -- the 1024-point Sylvester-ordered Hadamard butterfly of one
// warp, shared by the forward rotation and the embedding lookup's inverse.
//
// Layout.  Lane l holds the elements 128 j + 4 l + c (j = 0..7, c = 0..3) as
// value 4 j + c of its 32, kept as 16 pairs: value 2 k + e is v[k].x (e = 0)
// or v[k].y (e = 1).  Index bits 0-1 (c) and 7-9 (j) are in registers, bits
// 2-6 are the lane.  H is a tensor product over the index bits, so the
// stages can run in any order: the five register bits first; then a
// transpose through shared memory (row 8 c + j of 32 floats, padded to 36 so
// that both access patterns are free of bank conflicts) gives lane l the 32
// elements 128 j' + 4 t + c' (t = 0..31) with (c', j') = (l / 8, l % 8),
// whose index bits 2-6 are now in registers; their five stages follow, and
// the transpose back restores the layout.  The result is H v, unnormalised:
// y_k = sum_i (-1)^popcount(i & k) v_i.  No shuffles: of an element's ten
// butterfly adds, eight are halves of packed fp32x2 instructions, and it
// crosses shared memory four times.
#pragma once

#include <stdint.h>

namespace ptq {

constexpr int kRowPad = 36;
constexpr int kWarpBuf = 32 * kRowPad;  // floats of shared memory per warp

// Butterflies over the five register index bits of 16 pairs.  Bit 0 pairs
// the halves of each v[k] (scalar adds); bits 1-4 pair whole v[k] and
// v[k | m], two butterflies per packed fp32x2 add and one packed fused
// multiply-add (d * -1 + a is a - d, rounded once, as a subtraction is).
__device__ __forceinline__ void reg_hadamard_32(float2 (&v)[16]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float a = v[k].x, d = v[k].y;
    v[k] = make_float2(a + d, a - d);
  }
  const float2 neg1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int m = 1; m < 16; m <<= 1)
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      if (k & m) continue;
      const float2 a = v[k], d = v[k | m];
      v[k] = __fadd2_rn(a, d);
      v[k | m] = __ffma2_rn(d, neg1, a);
    }
}

// H over the 1024 elements the warp holds, in place (layout above).  `buf`
// is the warp's kWarpBuf floats; it is free again when this returns.
__device__ __forceinline__ void warp_hadamard_1024(float2 (&v)[16], float* buf, int lane) {
  // index bits 0, 1 (c) and 7, 8, 9 (j)
  reg_hadamard_32(v);
  // transpose: element (j, c, lane) to row 8 c + j, column lane
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    buf[(8 * 0 + j) * kRowPad + lane] = v[2 * j].x;
    buf[(8 * 1 + j) * kRowPad + lane] = v[2 * j].y;
    buf[(8 * 2 + j) * kRowPad + lane] = v[2 * j + 1].x;
    buf[(8 * 3 + j) * kRowPad + lane] = v[2 * j + 1].y;
  }
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float4 q = *reinterpret_cast<const float4*>(buf + lane * kRowPad + 4 * k);
    v[2 * k] = make_float2(q.x, q.y);
    v[2 * k + 1] = make_float2(q.z, q.w);
  }
  // index bits 2..6 (t, now the register index)
  reg_hadamard_32(v);
  __syncwarp();  // every lane has read its row before any is overwritten
#pragma unroll
  for (int k = 0; k < 8; ++k)
    *reinterpret_cast<float4*>(buf + lane * kRowPad + 4 * k) =
        make_float4(v[2 * k].x, v[2 * k].y, v[2 * k + 1].x, v[2 * k + 1].y);
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[2 * j] = make_float2(buf[(8 * 0 + j) * kRowPad + lane], buf[(8 * 1 + j) * kRowPad + lane]);
    v[2 * j + 1] =
        make_float2(buf[(8 * 2 + j) * kRowPad + lane], buf[(8 * 3 + j) * kRowPad + lane]);
  }
  __syncwarp();  // the buffer is free for the warp's next block
}

// The sign bits of sign bytes c = 2 h and 2 h + 1 of `sg` at bits 15 and 31,
// the sign positions of a 16-bit pair.
__device__ __forceinline__ uint32_t pair_sign_mask(uint32_t sg, int h) {
  return __byte_perm(sg, 0u, h ? 0x3424u : 0x1404u) & 0x80008000u;
}

// The sign bit of sign byte c of `sg` at bit 31, the sign position of an fp32.
__device__ __forceinline__ uint32_t f32_sign_mask(uint32_t sg, int c) {
  return (sg << (24 - 8 * c)) & 0x80000000u;
}

}  // namespace ptq

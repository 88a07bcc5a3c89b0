// fwht_warp.cuh -- the 1024-point Sylvester-ordered Hadamard butterfly of one
// warp, shared by the forward rotation and the embedding lookup's inverse.
//
// Lane l holds elements 128 j + 4 l + c (j = 0..7, c = 0..3) in v[j][c]:
// index bits 0-1 (c) and 7-9 (j) live in registers, bits 2-6 are the lane id.
// H is a tensor product over the index bits, so the stage order is free; the
// ten stages are the five in-register ones and five xor-shuffles.  The result
// is H v, unnormalised: y_k = sum_i (-1)^popcount(i & k) v_i.
#pragma once

namespace ptq {

__device__ __forceinline__ void warp_hadamard_1024(float (&v)[8][4], int lane) {
  // index bits 0 and 1 (c)
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float a0 = v[j][0] + v[j][1], a1 = v[j][0] - v[j][1];
    float a2 = v[j][2] + v[j][3], a3 = v[j][2] - v[j][3];
    v[j][0] = a0 + a2; v[j][2] = a0 - a2;
    v[j][1] = a1 + a3; v[j][3] = a1 - a3;
  }
  // index bits 7, 8, 9 (j)
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j & h) continue;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float a = v[j][c], d = v[j + h][c];
        v[j][c] = a + d;
        v[j + h][c] = a - d;
      }
    }
  }
  // index bits 2..6 (lane): the partner lane holds the other element of the pair
#pragma unroll
  for (int mask = 1; mask < 32; mask <<= 1) {
    const float sgn = (lane & mask) ? -1.0f : 1.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float p = __shfl_xor_sync(0xffffffffu, v[j][c], mask);
        v[j][c] = fmaf(sgn, v[j][c], p);  // low: v + p, high: p - v
      }
    }
  }
}

}  // namespace ptq

// k_embed.cu -- token-embedding lookup on a rotated table.
//
// "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally", section "What
// Bonsai is": the rotation folded into the stored weights is undone on the
// embedding table after each lookup.  Row v of the table holds R e_v with
// R = H D_s / 32 (the signed rotation the activations get); R is orthonormal,
// so the lookup returns e_v = R^T row = D_s H row / 32: the Hadamard
// butterfly first, then the signs and 1/32 -- the reverse order of the
// forward rotation.
//
// A (token m, 1024-block b) pair goes to one CTA of 256 threads, 4 values
// each, which keeps the dependent chain short (a decode step has only
// H / 1024 pairs); with many pairs, to one warp instead, laid out over the
// lanes as warp_hadamard_1024 (fwht_warp.cuh) wants it.  The
// table is dense (fp32 or bf16 rows, read with 16- or 8-byte vector loads) or
// PTQ1_0: a thread's four weights 4l..4l+3 of a 128-weight block sit in one
// or two of its 26 bytes, and each is the pages' peel (section "What Ferrox
// does with it": digit n of byte e is floor(3^(n+1) u) - 3 floor(3^n u),
// u = e / 256, exact in fp32) minus one, times the block's fp16 scale.
// Arithmetic is fp32; a bf16 output is rounded to nearest-even once, at the
// end.  An id outside [0, V) gives quiet NaN and reads nothing from the table.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fwht_warp.cuh"
#include "ptq_internal.cuh"

namespace ptq {
namespace {

enum class Tab { F32, BF16, PTQ1 };

// Digit n of byte e by the pages' peel, exact in fp32: u = e / 256 and p = 3^n,
// so 3 p u <= 243 * 255 / 256 needs no rounding.
__device__ __forceinline__ float peel(uint32_t e, float p) {
  const float u = (float)e * (1.0f / 256.0f);
  return floorf(3.0f * p * u) - 3.0f * floorf(p * u);
}

__device__ __forceinline__ float pow3(int n) {
  return n == 0 ? 1.0f : n == 1 ? 3.0f : n == 2 ? 9.0f : n == 3 ? 27.0f : 81.0f;
}

// The four values at weights 4l..4l+3 of 128-weight block j of 1024-group g
// of table row `id` (dense: elements 128 j + 4 l + c of that group).  For
// PTQ1_0 the group's 8 blocks are 208 contiguous bytes starting at
// 208 (id bpr + g) and its 8 scales 16 contiguous bytes.
template <Tab kT>
__device__ __forceinline__ void load4(const void* __restrict__ table,
                                      const uint16_t* __restrict__ scales, int64_t row_group,
                                      int j, int l, float (&v)[4]) {
  if constexpr (kT == Tab::F32) {
    const float4 r = *reinterpret_cast<const float4*>(static_cast<const float*>(table) +
                                                      row_group * kRot + 128 * j + 4 * l);
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  } else if constexpr (kT == Tab::BF16) {
    const uint2 r = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(table) +
                                                    row_group * kRot + 128 * j + 4 * l);
    v[0] = __uint_as_float(r.x << 16);
    v[1] = __uint_as_float(r.x & 0xffff0000u);
    v[2] = __uint_as_float(r.y << 16);
    v[3] = __uint_as_float(r.y & 0xffff0000u);
  } else {
    const uint8_t* blk = static_cast<const uint8_t*>(table) + row_group * kGroupBytes + j * kBlockBytes;
    const float s = __half2float(__ushort_as_half(scales[row_group * kGroupBlocks + j]));
    const int w0 = 4 * l, q0 = w0 / 5, q1 = (w0 + 3) / 5;  // the one or two bytes
    const uint32_t e0 = blk[q0], e1 = blk[q1];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int w = w0 + c;
      v[c] = (peel(w / 5 == q0 ? e0 : e1, pow3(w % 5)) - 1.0f) * s;
    }
  }
}

template <Act kOut>
__device__ __forceinline__ void store4(void* out, int64_t e, const float (&o)[4]) {
  if constexpr (kOut == Act::BF16) {
    uint2 r;
    r.x = __bfloat16_as_ushort(__float2bfloat16_rn(o[0])) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o[1])) << 16);
    r.y = __bfloat16_as_ushort(__float2bfloat16_rn(o[2])) |
          ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(o[3])) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + e) = r;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + e) = make_float4(o[0], o[1], o[2], o[3]);
  }
}

template <Act kOut>
__device__ __forceinline__ void store1(void* out, int64_t e, float o) {
  if constexpr (kOut == Act::BF16)
    static_cast<uint16_t*>(out)[e] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
  else
    static_cast<float*>(out)[e] = o;
}

constexpr float kQNaN = __builtin_nanf("");

// Many (token, block) pairs: one warp each, 32 values a lane in the layout
// of warp_hadamard_1024, which does the butterfly around two transposes
// through the warp's kWarpBuf floats of shared memory.
//
// A PTQ1_0 group (208 bytes and 8 scales, 16 bytes) is read by lanes 0..13
// with one 16-byte load each and staged in shared memory; each lane then
// takes its two bytes per block from there.  A byte's five digits come from
// a 256-entry table of codes (digit n in bits 2n, 2n + 1) that the CTA
// builds once with the pages' peel, so a weight costs a shift-and-mask, a
// conversion and d * s - s.
constexpr int kEmbedWarps = 8;
constexpr int kStageBytes = kGroupBytes + 16;  // a group's trits and its 8 scales
constexpr size_t kEmbedSmem =
    (size_t)kEmbedWarps * kWarpBuf * 4 + 256 * 4 + (size_t)kEmbedWarps * kStageBytes;

template <Act kOut>
__device__ __forceinline__ void store_pair4(void* out, int64_t e, float2 a, float2 b,
                                            uint32_t sg) {
  const float2 s = make_float2(1.0f / 32.0f, 1.0f / 32.0f);
  a = __fmul2_rn(a, s);
  b = __fmul2_rn(b, s);
  if constexpr (kOut == Act::BF16) {  // rounding is symmetric: flip after it
    const __nv_bfloat162 ha = __floats2bfloat162_rn(a.x, a.y), hb = __floats2bfloat162_rn(b.x, b.y);
    uint2 r;
    r.x = *reinterpret_cast<const uint32_t*>(&ha) ^ pair_sign_mask(sg, 0);
    r.y = *reinterpret_cast<const uint32_t*>(&hb) ^ pair_sign_mask(sg, 1);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + e) = r;
  } else {
    float4 r;
    r.x = __uint_as_float(__float_as_uint(a.x) ^ f32_sign_mask(sg, 0));
    r.y = __uint_as_float(__float_as_uint(a.y) ^ f32_sign_mask(sg, 1));
    r.z = __uint_as_float(__float_as_uint(b.x) ^ f32_sign_mask(sg, 2));
    r.w = __uint_as_float(__float_as_uint(b.y) ^ f32_sign_mask(sg, 3));
    *reinterpret_cast<float4*>(static_cast<float*>(out) + e) = r;
  }
}

template <Tab kT, Act kOut>
__global__ void __launch_bounds__(32 * kEmbedWarps) embed_warp_kernel(
    const void* __restrict__ table, const uint16_t* __restrict__ scales, const int32_t* ids,
    const int8_t* __restrict__ signs, void* out, int64_t total_blocks, int64_t blocks_per_row,
    int64_t V) {
  extern __shared__ __align__(16) unsigned char esmem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* buf = reinterpret_cast<float*>(esmem) + warp * kWarpBuf;
  uint32_t* code = reinterpret_cast<uint32_t*>(esmem + kEmbedWarps * kWarpBuf * 4);
  unsigned char* stage = esmem + kEmbedWarps * kWarpBuf * 4 + 256 * 4 + warp * kStageBytes;
  const int64_t H = blocks_per_row * kRot;
  const int64_t nwarps = (int64_t)gridDim.x * kEmbedWarps;
  pdl_release();
  if constexpr (kT == Tab::PTQ1) {
    for (int e = threadIdx.x; e < 256; e += blockDim.x) {
      uint32_t c = 0;
#pragma unroll
      for (int n = 0; n < 5; ++n) c |= (uint32_t)peel((uint32_t)e, pow3(n)) << (2 * n);
      code[e] = c;
    }
    __syncthreads();
  }
  // PTQ1_0: this lane's weights 4 l .. 4 l + 3 of each block sit in bytes
  // q0 and q1 (q1 = q0 or q0 + 1); weight c is digit dn[c] of byte q0 or q1
  const int q0 = (4 * lane) / 5, q1 = (4 * lane + 3) / 5;
  pdl_wait();  // the ids may come from the previous kernel (a sampler)
  for (int64_t wb = (int64_t)blockIdx.x * kEmbedWarps + warp; wb < total_blocks; wb += nwarps) {
    const int64_t m = wb / blocks_per_row, b = wb % blocks_per_row;
    const int32_t id = ids[m];
    const bool ok = id >= 0 && (int64_t)id < V;  // the same for the whole warp
    if (!ok) {
      const float4 nan4 = make_float4(kQNaN, kQNaN, kQNaN, kQNaN);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t e = m * H + b * kRot + 128 * j + 4 * lane;
        const float o[4] = {nan4.x, nan4.y, nan4.z, nan4.w};
        store4<kOut>(out, e, o);
      }
      continue;
    }
    const int64_t rg = (int64_t)id * blocks_per_row + b;  // the table row's group
    float2 v[16];
    if constexpr (kT == Tab::PTQ1) {
      if (lane < 14) {  // 13 x 16 bytes of trits, then the 8 scales
        const uint4 q = lane < 13 ? reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(table) +
                                                                   rg * kGroupBytes)[lane]
                                  : *reinterpret_cast<const uint4*>(scales + rg * kGroupBlocks);
        *reinterpret_cast<uint4*>(stage + 16 * lane) = q;
      }
      __syncwarp();
      const uint4 sraw = *reinterpret_cast<const uint4*>(stage + kGroupBytes);
      const uint32_t sw[4] = {sraw.x, sraw.y, sraw.z, sraw.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float s = __half2float(__ushort_as_half((unsigned short)(sw[j / 2] >> (16 * (j & 1)))));
        const uint32_t c0 = code[stage[kBlockBytes * j + q0]];
        const uint32_t c1 = code[stage[kBlockBytes * j + q1]];
        float t[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int w = 4 * lane + c;
          const uint32_t d = ((w / 5 == q0 ? c0 : c1) >> (2 * (w % 5))) & 3u;
          t[c] = fmaf((float)d, s, -s);  // (d - 1) s, exact
        }
        v[2 * j] = make_float2(t[0], t[1]);
        v[2 * j + 1] = make_float2(t[2], t[3]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float t[4];
        load4<kT>(table, scales, rg, j, lane, t);
        v[2 * j] = make_float2(t[0], t[1]);
        v[2 * j + 1] = make_float2(t[2], t[3]);
      }
    }
    warp_hadamard_1024(v, buf, lane);  // its barriers also free the stage
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t k = b * kRot + 128 * j + 4 * lane;  // index within the row
      const uint32_t sg = *reinterpret_cast<const uint32_t*>(signs + k);
      store_pair4<kOut>(out, m * H + k, v[2 * j], v[2 * j + 1], sg);
    }
  }
}

// Few pairs (a decode step): one CTA of 256 threads each, 4 values a thread.
// Thread (warp j, lane l) holds elements 128 j + 4 l + c: index bits 0-1 in
// registers, bits 2-6 across the lanes; bits 7-9 (the warp) are done after a
// transpose through shared memory, by 128 threads holding elements t + 128 k.
// The output signs are requested before the id: they do not depend on it,
// and a decode step's chain of few pairs is short.
template <Tab kT, Act kOut>
__global__ void __launch_bounds__(256) embed_cta_kernel(const void* __restrict__ table,
                                                        const uint16_t* __restrict__ scales,
                                                        const int32_t* ids,
                                                        const int8_t* __restrict__ signs,
                                                        void* out, int64_t total_blocks,
                                                        int64_t blocks_per_row, int64_t V) {
  __shared__ float4 exch[kRot / 4];
  const int t = threadIdx.x, lane = t & 31, j = t >> 5;
  const int64_t H = blocks_per_row * kRot;
  pdl_release();
  pdl_wait();
  for (int64_t wb = blockIdx.x; wb < total_blocks; wb += gridDim.x) {
    const int64_t m = wb / blocks_per_row, b = wb % blocks_per_row;
    // the output signs do not depend on the id
    int8_t sg[8];
    if (t < 128) {
#pragma unroll
      for (int k = 0; k < 8; ++k) sg[k] = signs[b * kRot + t + 128 * k];
    }
    const int32_t id = ids[m];
    const bool ok = id >= 0 && (int64_t)id < V;  // the same for the whole CTA
    if (!ok) {
      for (int i = t; i < kRot; i += 256) store1<kOut>(out, m * H + b * kRot + i, kQNaN);
      continue;
    }
    float v[4];
    load4<kT>(table, scales, (int64_t)id * blocks_per_row + b, j, lane, v);
    {  // bits 0, 1
      const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
      v[0] = a0 + a2; v[2] = a0 - a2; v[1] = a1 + a3; v[3] = a1 - a3;
    }
#pragma unroll
    for (int mask = 1; mask < 32; mask <<= 1) {  // bits 2..6
      const float sgn = (lane & mask) ? -1.0f : 1.0f;
#pragma unroll
      for (int c = 0; c < 4; ++c) v[c] = fmaf(sgn, v[c], __shfl_xor_sync(0xffffffffu, v[c], mask));
    }
    __syncthreads();  // the previous pair's readers are done with exch
    exch[t] = make_float4(v[0], v[1], v[2], v[3]);
    __syncthreads();
    if (t < 128) {  // bits 7..9: elements t + 128 k
      const float* ex = reinterpret_cast<const float*>(exch);
      float w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = ex[t + 128 * k];
#pragma unroll
      for (int h = 1; h < 8; h <<= 1)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (!(k & h)) {
            const float p = w[k], q = w[k + h];
            w[k] = p + q;
            w[k + h] = p - q;
          }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t i = b * kRot + t + 128 * k;
        const float f = w[k] * (1.0f / 32.0f);
        const int8_t sk = sg[k];
        store1<kOut>(out, m * H + i, sk < 0 ? -f : f);
      }
    }
  }
}

template <Tab kT, Act kOut>
cudaError_t launch_embed_t(const void* table, const uint16_t* scales, const int32_t* ids,
                           const int8_t* signs, void* out, int64_t M, int64_t V, int64_t H,
                           cudaStream_t st) {
  const int64_t bpr = H / kRot, total = M * bpr;
  constexpr int64_t kSms = 152;
  // Measured on a GB300 (V = 131072, H = 5120) with the earlier shuffle
  // butterfly: a CTA per pair was faster up to M = 256 (1280 pairs) for
  // dense tables and at every M for PTQ1_0 ones.
  if (total < 16 * kSms) {
    const int64_t grid = total;
    return launch_pdl(embed_cta_kernel<kT, kOut>, dim3((unsigned)grid), dim3(256), 0, st,
                      table, scales, ids, signs, out, total, bpr, V);
  }
  int64_t grid = (total + kEmbedWarps - 1) / kEmbedWarps;
  if (grid > kSms * 64) grid = kSms * 64;
  return launch_pdl(embed_warp_kernel<kT, kOut>, dim3((unsigned)grid), dim3(32 * kEmbedWarps),
                    kEmbedSmem, st, table, scales, ids, signs, out, total, bpr, V);
}

}  // namespace

cudaError_t launch_embed(const void* table, Act table_t, const int32_t* ids, const int8_t* signs,
                         void* out, Act out_t, int64_t M, int64_t V, int64_t H, cudaStream_t st) {
  if (table_t == Act::F32 && out_t == Act::F32)
    return launch_embed_t<Tab::F32, Act::F32>(table, nullptr, ids, signs, out, M, V, H, st);
  if (table_t == Act::BF16 && out_t == Act::BF16)
    return launch_embed_t<Tab::BF16, Act::BF16>(table, nullptr, ids, signs, out, M, V, H, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_embed_ptq1(const uint8_t* wq, const uint16_t* scales, const int32_t* ids,
                              const int8_t* signs, void* out, Act out_t, int64_t M, int64_t V,
                              int64_t H, cudaStream_t st) {
  if (out_t == Act::F32)
    return launch_embed_t<Tab::PTQ1, Act::F32>(wq, scales, ids, signs, out, M, V, H, st);
  if (out_t == Act::BF16)
    return launch_embed_t<Tab::PTQ1, Act::BF16>(wq, scales, ids, signs, out, M, V, H, st);
  return cudaErrorInvalidValue;
}

}  // namespace ptq

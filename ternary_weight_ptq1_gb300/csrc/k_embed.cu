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
// One warp owns one (token m, 1024-block b) pair, laid out over the lanes as
// warp_hadamard_1024 (fwht_warp.cuh) wants it.  The table is dense (fp32 or
// bf16 rows, read with 16- or 8-byte vector loads) or PTQ1_0: a lane's four
// weights 4l..4l+3 of a 128-weight block sit in one or two of its 26 bytes,
// and each is the pages' peel (section "What Ferrox does with it": digit n
// of byte e is floor(3^(n+1) u) - 3 floor(3^n u), u = e / 256, exact in fp32)
// minus one, times the block's fp16 scale.  Arithmetic is fp32; a bf16 output
// is rounded to nearest-even once, at the end.  An id outside [0, V) makes
// the warp write quiet NaN and read nothing from the table.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fwht_warp.cuh"
#include "ptq_internal.cuh"

namespace ptq {
namespace {

enum class Tab { F32, BF16, PTQ1 };

// Weight w (0..127) of a PTQ1_0 block whose 26 bytes start at `blk`.
__device__ __forceinline__ float ptq1_trit(const uint8_t* blk, int w) {
  const int q = w / 5, n = w % 5;
  const float u = (float)blk[q] * (1.0f / 256.0f);
  const float p = n == 0 ? 1.0f : n == 1 ? 3.0f : n == 2 ? 9.0f : n == 3 ? 27.0f : 81.0f;  // 3^n
  return floorf(3.0f * p * u) - 3.0f * floorf(p * u) - 1.0f;
}

template <Tab kT, Act kOut>
__global__ void __launch_bounds__(256) embed_kernel(const void* __restrict__ table,
                                                    const uint16_t* __restrict__ scales,
                                                    const int32_t* ids,
                                                    const int8_t* __restrict__ signs, void* out,
                                                    int64_t total_blocks, int64_t blocks_per_row,
                                                    int64_t V) {
  const int lane = threadIdx.x & 31;
  const int64_t H = blocks_per_row * kRot;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  pdl_release();
  pdl_wait();  // the ids may come from the previous kernel (a sampler)
  for (int64_t wb = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); wb < total_blocks;
       wb += nwarps) {
    const int64_t m = wb / blocks_per_row, b = wb % blocks_per_row;
    const int32_t id = ids[m];
    const bool ok = id >= 0 && (int64_t)id < V;  // the same for the whole warp
    float v[8][4] = {};
    if (ok) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t e = (int64_t)id * H + b * kRot + 128 * j + 4 * lane;
        if constexpr (kT == Tab::F32) {
          const float4 r = *reinterpret_cast<const float4*>(static_cast<const float*>(table) + e);
          v[j][0] = r.x; v[j][1] = r.y; v[j][2] = r.z; v[j][3] = r.w;
        } else if constexpr (kT == Tab::BF16) {
          const uint2 r = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(table) + e);
          v[j][0] = __uint_as_float(r.x << 16);
          v[j][1] = __uint_as_float(r.x & 0xffff0000u);
          v[j][2] = __uint_as_float(r.y << 16);
          v[j][3] = __uint_as_float(r.y & 0xffff0000u);
        } else {
          const int64_t blk = (int64_t)id * (H / kBlockWeights) + b * kGroupBlocks + j;
          const uint8_t* bytes = static_cast<const uint8_t*>(table) + blk * kBlockBytes;
          const float s = __half2float(__ushort_as_half(scales[blk]));
#pragma unroll
          for (int c = 0; c < 4; ++c) v[j][c] = ptq1_trit(bytes, 4 * lane + c) * s;
        }
      }
      warp_hadamard_1024(v, lane);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t k = b * kRot + 128 * j + 4 * lane;  // index within the row
      const uint32_t sg = *reinterpret_cast<const uint32_t*>(signs + k);
      float o[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float f = v[j][c] * (1.0f / 32.0f);
        o[c] = ok ? ((int8_t)(sg >> (8 * c)) < 0 ? -f : f) : __uint_as_float(0x7fc00000u);
      }
      const int64_t e = m * H + k;
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
  }
}

template <Tab kT, Act kOut>
cudaError_t launch_embed_t(const void* table, const uint16_t* scales, const int32_t* ids,
                           const int8_t* signs, void* out, int64_t M, int64_t V, int64_t H,
                           cudaStream_t st) {
  const int64_t bpr = H / kRot, total = M * bpr;
  const int warps = 8;
  int64_t grid = (total + warps - 1) / warps;
  if (grid > 152 * 64) grid = 152 * 64;
  return launch_pdl(embed_kernel<kT, kOut>, dim3((unsigned)grid), dim3(32 * warps), 0, st, table,
                    scales, ids, signs, out, total, bpr, V);
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

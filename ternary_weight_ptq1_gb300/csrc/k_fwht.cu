// k_fwht.cu -- signed 1024-wide Walsh-Hadamard rotation of activations.
//
// "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally", section "What
// Bonsai is": the stored weights carry a 1024-wide butterfly with a sign
// pattern, so every activation is flipped by the signs, pushed through the
// Sylvester-ordered Hadamard butterfly and scaled by 1/32 (orthonormal).
//
// One warp owns one 1024-element block, laid out over the lanes as
// warp_hadamard_1024 (fwht_warp.cuh) wants it.  Loads and stores are 16-byte
// (fp32) or 8-byte (16-bit types) vectors, 512 (256) contiguous bytes per warp
// instruction.  Arithmetic is fp32 (16-bit outputs are rounded
// to nearest-even once, at the end); y may alias x because a warp reads its
// whole block before it writes any of it (in-place needs equal element
// sizes, which the callers guarantee).  Launched with programmatic
// dependent launch: it lets its consumer start at once and waits for its
// own producer before reading x.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fwht_warp.cuh"
#include "ptq_internal.cuh"

namespace ptq {
namespace {

// 16-bit storage: decode to fp32 exactly, encode with round-to-nearest-even.
template <Act T>
__device__ __forceinline__ float from16(uint32_t bits) {
  if constexpr (T == Act::BF16) return __uint_as_float(bits << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

template <Act T>
__device__ __forceinline__ uint32_t to16(float f) {
  if constexpr (T == Act::BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  else return __half_as_ushort(__float2half_rn(f));
}

// fp16 rounds |v| >= 65520 (the largest finite value 65504 plus half its
// last-place step) to infinity.
__device__ __forceinline__ bool beyond_f16(float v) {
  const float a = fabsf(v);
  return a >= 65520.0f && a <= 3.402823466e38f;
}

template <Act kIn, Act kOut>
__global__ void __launch_bounds__(256) fwht1024_kernel(const void* x, void* y,
                                                       const int8_t* __restrict__ signs,
                                                       int64_t total_blocks, int64_t blocks_per_row,
                                                       int* status) {
  const int lane = threadIdx.x & 31;
  bool over = false;  // kOut == F16: a finite value stored as infinity
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  pdl_release();  // the consumer's prologue (its weight prefetch) may start now
  pdl_wait();     // x may come from the previous kernel
  for (int64_t wb = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); wb < total_blocks;
       wb += nwarps) {
    const int64_t b = wb % blocks_per_row;
    const int64_t base = wb * kRot;  // rows are contiguous: row m, block b -> wb * 1024
    float v[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t e = base + 128 * j + 4 * lane;
      const uint32_t sg = *reinterpret_cast<const uint32_t*>(signs + b * kRot + 128 * j + 4 * lane);
      float a[4];
      if constexpr (kIn != Act::F32) {
        const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + e);
        a[0] = from16<kIn>(raw.x & 0xffffu);
        a[1] = from16<kIn>(raw.x >> 16);
        a[2] = from16<kIn>(raw.y & 0xffffu);
        a[3] = from16<kIn>(raw.y >> 16);
      } else {
        const float4 raw = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + e);
        a[0] = raw.x; a[1] = raw.y; a[2] = raw.z; a[3] = raw.w;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int s = static_cast<int8_t>((sg >> (8 * c)) & 0xffu);
        v[j][c] = s < 0 ? -a[c] : a[c];
      }
    }
    warp_hadamard_1024(v, lane);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t e = base + 128 * j + 4 * lane;
      const float s = 1.0f / 32.0f;
      if constexpr (kOut == Act::F16) {
#pragma unroll
        for (int c = 0; c < 4; ++c) over |= beyond_f16(v[j][c] * s);
      }
      if constexpr (kOut != Act::F32) {
        uint2 out;
        out.x = to16<kOut>(v[j][0] * s) | (to16<kOut>(v[j][1] * s) << 16);
        out.y = to16<kOut>(v[j][2] * s) | (to16<kOut>(v[j][3] * s) << 16);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + e) = out;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(y) + e) =
            make_float4(v[j][0] * s, v[j][1] * s, v[j][2] * s, v[j][3] * s);
      }
    }
  }
  if constexpr (kOut == Act::F16) {
    if (__any_sync(0xffffffffu, over) && lane == 0) atomicOr(status, kDevRange);
  }
}

}  // namespace

cudaError_t launch_fwht(const void* x, Act in, void* y, Act out, const int8_t* signs,
                        int64_t M, int64_t K, cudaStream_t st) {
  const int64_t bpr = K / kRot;
  const int64_t total = M * bpr;
  const int warps = 8;
  int64_t grid = (total + warps - 1) / warps;
  if (grid > 152 * 64) grid = 152 * 64;
  const dim3 g((unsigned)grid), b(32 * warps);
  int* status = nullptr;
  if (out == Act::F16 && (status = device_status_ptr()) == nullptr) return cudaErrorInvalidDevice;
  if (in == Act::F32 && out == Act::F32)
    return launch_pdl(fwht1024_kernel<Act::F32, Act::F32>, g, b, 0, st, x, y, signs, total, bpr,
                      status);
  if (in == Act::BF16 && out == Act::BF16)
    return launch_pdl(fwht1024_kernel<Act::BF16, Act::BF16>, g, b, 0, st, x, y, signs, total, bpr,
                      status);
  if (in == Act::BF16 && out == Act::F16)
    return launch_pdl(fwht1024_kernel<Act::BF16, Act::F16>, g, b, 0, st, x, y, signs, total, bpr,
                      status);
  if (in == Act::F32 && out == Act::F16)
    return launch_pdl(fwht1024_kernel<Act::F32, Act::F16>, g, b, 0, st, x, y, signs, total, bpr,
                      status);
  return cudaErrorInvalidValue;
}

}  // namespace ptq

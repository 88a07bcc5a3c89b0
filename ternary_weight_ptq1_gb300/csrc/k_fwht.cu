// k_fwht.cu -- signed 1024-wide Walsh-Hadamard rotation of activations.
//
// "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally", section "What
// Bonsai is": the stored weights carry a 1024-wide butterfly with a sign
// pattern, so every activation is flipped by the signs, pushed through the
// Sylvester-ordered Hadamard butterfly and scaled by 1/32 (orthonormal).
//
// One warp owns one 1024-element block at a time (see fwht1024_kernel for
// the layout).  Loads and stores are 16-byte (fp32) or 8-byte (16-bit types)
// vectors, 512 (256) contiguous bytes per warp instruction.  Arithmetic is fp32 (16-bit outputs are rounded
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

// Two values rounded to nearest-even into one 16-bit pair (x low, y high).
template <Act T>
__device__ __forceinline__ uint32_t pack16(float2 f) {
  if constexpr (T == Act::BF16) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// fp16 rounds |v| >= 65520 (the largest finite value 65504 plus half its
// last-place step) to infinity.
__device__ __forceinline__ bool beyond_f16(float v) {
  const float a = fabsf(v);
  return a >= 65520.0f && a <= 3.402823466e38f;
}

// One warp owns one 1024-element block at a time, in the layout of
// warp_hadamard_1024 (fwht_warp.cuh): lane l holds the elements
// 128 j + 4 l + c, loaded and stored as 16-byte (8-byte) vectors.  Each
// element costs its load, its store, the conversions (16-bit values are
// sign-flipped and rounded two at a time) and the butterfly.
template <Act kIn, Act kOut>
__global__ void __launch_bounds__(256) fwht1024_kernel(const void* x, void* y,
                                                       const int8_t* __restrict__ signs,
                                                       int64_t total_blocks, int64_t blocks_per_row,
                                                       int* status) {
  extern __shared__ float sbuf[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* buf = sbuf + warp * kWarpBuf;
  bool over = false;  // kOut == F16: a finite value stored as infinity
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  pdl_release();  // the consumer's prologue (its weight prefetch) may start now
  pdl_wait();     // x may come from the previous kernel
  for (int64_t wb = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp; wb < total_blocks;
       wb += nwarps) {
    const int64_t b = wb % blocks_per_row;
    const int64_t base = wb * kRot;  // rows are contiguous: row m, block b -> wb * 1024
    float2 v[16];  // value 4 j + c in v[2 j + c / 2], half c % 2
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t e = base + 128 * j + 4 * lane;
      const uint32_t sg = *reinterpret_cast<const uint32_t*>(signs + b * kRot + 128 * j + 4 * lane);
      if constexpr (kIn != Act::F32) {
        // the sign bits flip the 16-bit values before they widen
        uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(x) + e);
        raw.x ^= pair_sign_mask(sg, 0);
        raw.y ^= pair_sign_mask(sg, 1);
        v[2 * j] = make_float2(from16<kIn>(raw.x & 0xffffu), from16<kIn>(raw.x >> 16));
        v[2 * j + 1] = make_float2(from16<kIn>(raw.y & 0xffffu), from16<kIn>(raw.y >> 16));
      } else {
        const float4 raw = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + e);
        float a[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int c = 0; c < 4; ++c)  // the sign bit of sign byte c flips the element
          a[c] = __uint_as_float(__float_as_uint(a[c]) ^ f32_sign_mask(sg, c));
        v[2 * j] = make_float2(a[0], a[1]);
        v[2 * j + 1] = make_float2(a[2], a[3]);
      }
    }
    warp_hadamard_1024(v, buf, lane);
    const float2 s = make_float2(1.0f / 32.0f, 1.0f / 32.0f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t e = base + 128 * j + 4 * lane;
      const float2 o01 = __fmul2_rn(v[2 * j], s), o23 = __fmul2_rn(v[2 * j + 1], s);
      if constexpr (kOut == Act::F16)
        over |= beyond_f16(o01.x) | beyond_f16(o01.y) | beyond_f16(o23.x) | beyond_f16(o23.y);
      if constexpr (kOut != Act::F32) {
        uint2 out;
        out.x = pack16<kOut>(o01);
        out.y = pack16<kOut>(o23);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + e) = out;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(y) + e) = make_float4(o01.x, o01.y, o23.x, o23.y);
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
  const size_t smem = (size_t)warps * kWarpBuf * sizeof(float);  // 36 KB
  int* status = nullptr;
  if (out == Act::F16 && (status = device_status_ptr()) == nullptr) return cudaErrorInvalidDevice;
  if (in == Act::F32 && out == Act::F32)
    return launch_pdl(fwht1024_kernel<Act::F32, Act::F32>, g, b, smem, st, x, y, signs, total, bpr,
                      status);
  if (in == Act::BF16 && out == Act::BF16)
    return launch_pdl(fwht1024_kernel<Act::BF16, Act::BF16>, g, b, smem, st, x, y, signs, total, bpr,
                      status);
  if (in == Act::BF16 && out == Act::F16)
    return launch_pdl(fwht1024_kernel<Act::BF16, Act::F16>, g, b, smem, st, x, y, signs, total, bpr,
                      status);
  if (in == Act::F32 && out == Act::F16)
    return launch_pdl(fwht1024_kernel<Act::F32, Act::F16>, g, b, smem, st, x, y, signs, total, bpr,
                      status);
  return cudaErrorInvalidValue;
}

}  // namespace ptq

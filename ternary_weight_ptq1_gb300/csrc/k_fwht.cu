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

// Butterflies over the register index bits of v[8][4] (index 4 j + c): the
// pairs that differ in bit `bit` of that index, unnormalised.
template <int kBit>
__device__ __forceinline__ void reg_stage(float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (i & (1 << kBit)) continue;
    const float a = v[i], d = v[i | (1 << kBit)];
    v[i] = a + d;
    v[i | (1 << kBit)] = a - d;
  }
}

__device__ __forceinline__ void reg_hadamard_32(float (&v)[32]) {
  reg_stage<0>(v);
  reg_stage<1>(v);
  reg_stage<2>(v);
  reg_stage<3>(v);
  reg_stage<4>(v);
}

// One warp owns one 1024-element block at a time.  Lane l first holds the
// elements 128 j + 4 l + c (j = 0..7, c = 0..3) in u[4 j + c]: index bits 0-1
// (c) and 7-9 (j) are in registers, bits 2-6 are the lane.  H is a tensor
// product over the index bits, so the stages can run in any order: the five
// register bits first; then a transpose through shared memory (row R = 8 c +
// j of 32 floats, padded to 36 so that both access patterns are free of bank
// conflicts) gives lane l the 32 elements 128 j' + 4 t + c' (t = 0..31) with
// (c', j') = (l / 8, l % 8), whose index bits 2-6 are now in registers; their
// five stages follow, and the transpose back gives the natural layout for
// 16-byte (8-byte) global stores.  No shuffles: each element costs 10 FADDs,
// 2.5 shared-memory instructions, its load, its store and the conversions.
constexpr int kRowPad = 36;
constexpr int kWarpBuf = 32 * kRowPad;  // floats per warp

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
    float u[32];
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
      for (int c = 0; c < 4; ++c)  // the sign bit of sign byte c flips the element
        u[4 * j + c] = __uint_as_float(__float_as_uint(a[c]) ^ ((sg << (24 - 8 * c)) & 0x80000000u));
    }
    // index bits 0, 1 (c) and 7, 8, 9 (j)
    reg_hadamard_32(u);
    // transpose: element (j, c, lane) to row 8 c + j, column lane
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) buf[(8 * c + j) * kRowPad + lane] = u[4 * j + c];
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 q = *reinterpret_cast<const float4*>(buf + lane * kRowPad + 4 * k);
      u[4 * k] = q.x; u[4 * k + 1] = q.y; u[4 * k + 2] = q.z; u[4 * k + 3] = q.w;
    }
    // index bits 2..6 (t, now the register index)
    reg_hadamard_32(u);
    __syncwarp();  // every lane has read its row before any is overwritten
#pragma unroll
    for (int k = 0; k < 8; ++k)
      *reinterpret_cast<float4*>(buf + lane * kRowPad + 4 * k) =
          make_float4(u[4 * k], u[4 * k + 1], u[4 * k + 2], u[4 * k + 3]);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) u[4 * j + c] = buf[(8 * c + j) * kRowPad + lane];
    __syncwarp();  // the buffer is free for the warp's next block
    const float s = 1.0f / 32.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t e = base + 128 * j + 4 * lane;
      const float o0 = u[4 * j] * s, o1 = u[4 * j + 1] * s, o2 = u[4 * j + 2] * s,
                  o3 = u[4 * j + 3] * s;
      if constexpr (kOut == Act::F16)
        over |= beyond_f16(o0) | beyond_f16(o1) | beyond_f16(o2) | beyond_f16(o3);
      if constexpr (kOut != Act::F32) {
        uint2 out;
        out.x = to16<kOut>(o0) | (to16<kOut>(o1) << 16);
        out.y = to16<kOut>(o2) | (to16<kOut>(o3) << 16);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + e) = out;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(y) + e) = make_float4(o0, o1, o2, o3);
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

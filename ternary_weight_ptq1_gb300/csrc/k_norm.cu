// k_norm.cu -- the residual add and RMSNorm between chained feed-forward
// blocks.
//
// "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally", section "Speed,
// and where it goes", names running the whole layer on the device, norms and
// residual adds included, as the next step after the matmuls.  The stack this
// serves is pre-norm: before layer l the previous block's output y is added
// into the fp32 residual stream x, and the block's input is
//     xn = x / sqrt(mean(x^2) + eps) * g_l.
//
// One CTA owns one row (rows grid-strided).  For rows of up to 16384
// elements each thread keeps its NV 16-byte vectors of the row in registers:
// it issues every load of x and y before the first store, so a row costs
// one round trip to L2, and the gains (weights, not activations) are loaded
// before the wait on the producer.  The sum of squares is fp32: a shuffle
// tree per warp, then every warp reduces the warp sums the same way, so the
// result does not depend on timing.  xn is written from the registers, fp32
// or bf16 (round to nearest even once).  1/sqrt is IEEE division of IEEE
// sqrtf.  Longer rows take a two-pass loop that re-reads its own writes.
// Launched with programmatic dependent launch: the next block's weight
// prefetch may start at once; x and y are read only after the producer is
// done.
#include <cuda_bf16.h>

#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int kThreads = 256;

template <Act T>
__device__ __forceinline__ float4 load4(const void* p, int64_t e) {
  if constexpr (T == Act::F32) {
    return *reinterpret_cast<const float4*>(static_cast<const float*>(p) + e);
  } else {
    const uint2 r = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + e);
    return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u),
                       __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
  }
}

template <Act T>
__device__ __forceinline__ void store4(void* p, int64_t e, float4 v) {
  if constexpr (T == Act::F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p) + e) = v;
  } else {
    auto b = [](float f) { return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f)); };
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p) + e) =
        make_uint2(b(v.x) | (b(v.y) << 16), b(v.z) | (b(v.w) << 16));
  }
}

// y == nullptr: no add.  xn == nullptr: no norm (the stack's final add).
template <Act T>
__global__ void __launch_bounds__(kThreads) add_rmsnorm_kernel(float* __restrict__ x,
                                                               const void* __restrict__ y,
                                                               const float* __restrict__ g,
                                                               void* __restrict__ xn, int64_t M,
                                                               int64_t H, float eps) {
  __shared__ float warp_ss[kThreads / 32];
  pdl_release();
  pdl_wait();  // x and y come from earlier kernels
  const int64_t nv = H / 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
    float4* xr = reinterpret_cast<float4*>(x + m * H);
    float ss = 0.0f;
    for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
      float4 v = xr[i];
      if (y) {
        const float4 d = load4<T>(y, m * H + 4 * i);
        v.x += d.x;
        v.y += d.y;
        v.z += d.z;
        v.w += d.w;
        xr[i] = v;
      }
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    if (!xn) continue;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) warp_ss[warp] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += warp_ss[w];
    __syncthreads();  // warp_ss is rewritten for the next row
    const float inv = 1.0f / sqrtf(tot / (float)H + eps);
    const float4* g4 = reinterpret_cast<const float4*>(g);
    for (int64_t i = threadIdx.x; i < nv; i += kThreads) {
      const float4 v = xr[i], w = g4[i];
      store4<T>(xn, m * H + 4 * i,
                make_float4(v.x * inv * w.x, v.y * inv * w.y, v.z * inv * w.z, v.w * inv * w.w));
    }
  }
}

// Sum of v over the CTA (blockDim.x a multiple of 32, at most 1024), the
// same in every thread; red holds 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  __syncthreads();  // red is rewritten by the next call
  return t;
}

// Rows of at most NV * blockDim.x vectors, held in registers.
template <Act T, int NV>
__global__ void __launch_bounds__(1024) add_rmsnorm_reg_kernel(float* __restrict__ x,
                                                               const void* __restrict__ y,
                                                               const float* __restrict__ g,
                                                               void* __restrict__ xn, int64_t M,
                                                               int64_t H, float eps) {
  __shared__ float red[32];
  const int64_t nv = H / 4;
  float4 w[NV];
  if (xn) {
    const float4* g4 = reinterpret_cast<const float4*>(g);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
      w[j] = i < nv ? g4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  pdl_release();
  pdl_wait();  // x and y come from earlier kernels
  for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
    float4* xr = reinterpret_cast<float4*>(x + m * H);
    float4 v[NV], d[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
      v[j] = i < nv ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      d[j] = (y && i < nv) ? load4<T>(y, m * H + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
      if (y) {
        v[j].x += d[j].x;
        v[j].y += d[j].y;
        v[j].z += d[j].z;
        v[j].w += d[j].w;
        if (i < nv) xr[i] = v[j];
      }
      ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
    if (!xn) continue;
    const float inv = 1.0f / sqrtf(block_sum(ss, red) / (float)H + eps);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int64_t i = threadIdx.x + (int64_t)j * blockDim.x;
      if (i < nv)
        store4<T>(xn, m * H + 4 * i,
                  make_float4(v[j].x * inv * w[j].x, v[j].y * inv * w[j].y, v[j].z * inv * w[j].z,
                              v[j].w * inv * w[j].w));
    }
  }
}

template <Act T>
cudaError_t launch_for(float* x, const void* y, const float* g, void* xn, int64_t M, int64_t H,
                       float eps, cudaStream_t st) {
  const int64_t nv = H / 4;
  const int64_t grid = M < 152 * 8 ? M : 152 * 8;
  if (nv > 4 * 1024)
    return launch_pdl(add_rmsnorm_kernel<T>, dim3((unsigned)grid), dim3(kThreads), 0, st, x, y, g,
                      xn, M, H, eps);
  // the fewest vectors per thread that 1024 threads allow, then the fewest
  // warps that hold the row
  const int per = nv <= 1024 ? 1 : nv <= 2048 ? 2 : 4;
  const int64_t threads = ((nv + per - 1) / per + 31) / 32 * 32;
  const dim3 gr((unsigned)grid), b((unsigned)threads);
  switch (per) {
    case 1: return launch_pdl(add_rmsnorm_reg_kernel<T, 1>, gr, b, 0, st, x, y, g, xn, M, H, eps);
    case 2: return launch_pdl(add_rmsnorm_reg_kernel<T, 2>, gr, b, 0, st, x, y, g, xn, M, H, eps);
    default: return launch_pdl(add_rmsnorm_reg_kernel<T, 4>, gr, b, 0, st, x, y, g, xn, M, H, eps);
  }
}

}  // namespace

cudaError_t launch_add_rmsnorm(float* x, const void* y, const float* g, void* xn, Act t,
                               int64_t M, int64_t H, float eps, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  if (t == Act::F32) return launch_for<Act::F32>(x, y, g, xn, M, H, eps, st);
  if (t == Act::BF16) return launch_for<Act::BF16>(x, y, g, xn, M, H, eps, st);
  return cudaErrorInvalidValue;
}

}  // namespace ptq

// k_gemm.cu -- prefill GEMM over PTQ1_0 weights, 16-bit activations.
//
//   y[m, n] = bf16( sum_b s[n, b] * sum_{i<128} t[n, 128b + i] * x[m, 128b + i] )
//
// Tiled SIMT kernel: a 64 x 64 output tile per CTA, one 128-weight block per
// K step.  The packed block is peeled into shared memory with the fp32 peel
// of "What Ferrox does with it"; the block's dot products accumulate in fp32
// and are scaled by the block's fp16 scale in fp32 before they join the
// running sum, so the scale is applied exactly.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int BM = 64, BN = 64, BK = kBlockWeights;

template <Act kX, bool kOutF32>
__global__ void __launch_bounds__(256) gemm_ptq1_bf16_simt(const uint8_t* __restrict__ wq,
                                                           const uint16_t* __restrict__ scales,
                                                           const uint16_t* __restrict__ x,
                                                           void* __restrict__ y, int M, int N,
                                                           int K) {
  __shared__ __align__(16) float xs[BK][BM + 4];
  __shared__ __align__(16) float ws[BK][BN + 4];
  __shared__ float sc[BN];
  const int tid = threadIdx.x;
  const int tm = (tid / 16) * 4, tn = (tid % 16) * 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nblk = K / BK;
  float acc[4][4] = {};
  for (int b = 0; b < nblk; ++b) {
    for (int i = tid; i < BM * BK; i += 256) {
      const int r = i / BK, k = i % BK;
      const int m = m0 + r;
      const uint16_t bits = m < M ? x[(size_t)m * K + (size_t)b * BK + k] : 0;
      xs[k][r] = kX == Act::BF16 ? __uint_as_float((uint32_t)bits << 16)
                                 : __half2float(__ushort_as_half(bits));
    }
    for (int i = tid; i < BN * kBlockBytes; i += 256) {
      const int r = i / kBlockBytes, j = i % kBlockBytes;
      const int n = n0 + r;
      const uint8_t byte = n < N ? wq[((size_t)n * nblk + b) * kBlockBytes + j] : 0;
      const float u = (float)byte * (1.0f / 256.0f);
      float fprev = 0.0f, p3 = 1.0f;
      for (int d = 0; d < 5; ++d) {
        p3 *= 3.0f;
        const float fnext = floorf(p3 * u);
        if (5 * j + d < BK) ws[5 * j + d][r] = n < N ? fnext - 3.0f * fprev - 1.0f : 0.0f;
        fprev = fnext;
      }
    }
    for (int i = tid; i < BN; i += 256) {
      const int n = n0 + i;
      sc[i] = n < N ? __half2float(__ushort_as_half(scales[(size_t)n * nblk + b])) : 0.0f;
    }
    __syncthreads();
    float blk[4][4] = {};
#pragma unroll 4
    for (int k = 0; k < BK; ++k) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[k][tm]);
      const float4 w = *reinterpret_cast<const float4*>(&ws[k][tn]);
      const float av[4] = {a.x, a.y, a.z, a.w}, wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) blk[i][j] = fmaf(av[i], wv[j], blk[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(sc[tn + j], blk[i][j], acc[i][j]);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + tm + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tn + j;
      if (n >= N) continue;
      if constexpr (kOutF32)
        static_cast<float*>(y)[(size_t)m * N + n] = acc[i][j];
      else
        static_cast<uint16_t*>(y)[(size_t)m * N + n] =
            __bfloat16_as_ushort(__float2bfloat16_rn(acc[i][j]));
    }
  }
}

}  // namespace

cudaError_t launch_gemm(const uint8_t* wq, const uint16_t* scales, const void* xv, Act x_t,
                        void* y, Act y_t, int64_t M, int64_t N, int64_t K, void* ws,
                        size_t ws_bytes, cudaStream_t st) {
  const cudaError_t tc = launch_gemm_tc(wq, scales, xv, x_t, y, y_t, M, N, K, ws, ws_bytes, st);
  if (tc != cudaErrorNotSupported) return tc;  // K % 1024 != 0 falls through to SIMT
  const uint16_t* x = static_cast<const uint16_t*>(xv);
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return cudaErrorInvalidValue;
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
  if (grid.y > 65535) return cudaErrorInvalidValue;
  const int m = (int)M, n = (int)N, k = (int)K;
  if (x_t == Act::BF16 && y_t == Act::BF16)
    gemm_ptq1_bf16_simt<Act::BF16, false><<<grid, 256, 0, st>>>(wq, scales, x, y, m, n, k);
  else if (x_t == Act::BF16 && y_t == Act::F32)
    gemm_ptq1_bf16_simt<Act::BF16, true><<<grid, 256, 0, st>>>(wq, scales, x, y, m, n, k);
  else if (x_t == Act::F16 && y_t == Act::BF16)
    gemm_ptq1_bf16_simt<Act::F16, false><<<grid, 256, 0, st>>>(wq, scales, x, y, m, n, k);
  else if (x_t == Act::F16 && y_t == Act::F32)
    gemm_ptq1_bf16_simt<Act::F16, true><<<grid, 256, 0, st>>>(wq, scales, x, y, m, n, k);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace ptq

// k_swiglu.cu -- h = silu(gate) * up between the two matmuls of the
// feed-forward block ("A 27B model in 5.5 GB: Bonsai ternary on Ferrox,
// locally", section "Speed, and where it goes": gate, SwiGLU, down).
// gu is M x 2I fp32 with the gate half first; h is M x I fp32.  fp32
// arithmetic with CUDA's expf.

#include "ptq_internal.cuh"

namespace ptq {
namespace {

__global__ void __launch_bounds__(256) swiglu_f32(const float* __restrict__ gu,
                                                  float* __restrict__ h, int64_t M, int64_t I) {
  pdl_release();
  pdl_wait();  // gu comes from the previous kernel
  for (int64_t m = blockIdx.y; m < M; m += gridDim.y) {
    const float* g = gu + m * 2 * I;
    const float* u = g + I;
    float* o = h + m * I;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < I;
         c += (int64_t)gridDim.x * blockDim.x)
      o[c] = g[c] / (1.0f + expf(-g[c])) * u[c];
  }
}

}  // namespace

// Used when the gate/up GEMM cannot take SwiGLU into its epilogue (a product
// split along K, or the SIMT fallback).  Rows go to the grid's y dimension,
// columns to x.
cudaError_t launch_swiglu(const float* gu, float* h, int64_t M, int64_t I, cudaStream_t st) {
  int64_t gx = (I + 255) / 256, gy = M;
  if (gx > 64) gx = 64;
  if (gy > 65535) gy = 65535;
  return launch_pdl(swiglu_f32, dim3((unsigned)gx, (unsigned)gy), dim3(256), 0, st, gu, h, M, I);
}

}  // namespace ptq

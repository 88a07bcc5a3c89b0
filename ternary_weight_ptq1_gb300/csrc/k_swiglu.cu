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
  const int64_t total = M * I;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t m = i / I, c = i - m * I;
    const float g = gu[m * 2 * I + c];
    h[i] = g / (1.0f + expf(-g)) * gu[m * 2 * I + I + c];
  }
}

}  // namespace

cudaError_t launch_swiglu(const float* gu, float* h, int64_t M, int64_t I, cudaStream_t st) {
  int64_t grid = (M * I + 255) / 256;
  if (grid > 152 * 32) grid = 152 * 32;
  swiglu_f32<<<(unsigned)grid, 256, 0, st>>>(gu, h, M, I);
  return cudaGetLastError();
}

}  // namespace ptq

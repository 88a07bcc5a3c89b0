// k_unpack.cu -- device decode of PTQ1_0 bytes into int8 trits.
//
// The peel of "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally",
// section "What Ferrox does with it": digit n of a byte is
// floor(3^(n+1) u) - 3 floor(3^n u) with u = byte / 256, evaluated on the
// fp32 pipe (every product 3^k * byte has at most 16 significant bits, so it
// is exact).  Trit = digit - 1.  Byte 25 of a block carries weights 125..127.
#include "ptq_internal.cuh"

namespace ptq {
namespace {

__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t* __restrict__ wq,
                                                     int8_t* __restrict__ trits,
                                                     int64_t total_bytes, int64_t K) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_bytes; i += stride) {
    const int64_t blk = i / kBlockBytes;  // global block index n * (K/128) + b
    const int j = static_cast<int>(i - blk * kBlockBytes);
    int8_t* out = trits + blk * kBlockWeights + 5 * j;  // rows of K trits are contiguous
    const float u = static_cast<float>(wq[i]) * (1.0f / 256.0f);
    float f_prev = 0.0f;  // floor(3^0 u) = 0 since u < 1
    float p3 = 1.0f;
#pragma unroll
    for (int n = 0; n < 5; ++n) {
      p3 *= 3.0f;
      const float f_next = floorf(p3 * u);
      if (5 * j + n < kBlockWeights) out[n] = static_cast<int8_t>(f_next - 3.0f * f_prev - 1.0f);
      f_prev = f_next;
    }
  }
  (void)K;
}

// PQ2_0 ("Why I Am Building Another Inference Engine", section "Level 2: The
// short answer": two bits per ternary weight): weight 4j + i of a row is bits
// 2i, 2i+1 of byte j, trit = code - 1.
__global__ void __launch_bounds__(256) unpack_pq2_kernel(const uint8_t* __restrict__ wq,
                                                         int8_t* __restrict__ trits,
                                                         int64_t total_bytes) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_bytes; i += stride) {
    const uint32_t b = wq[i];
    const uint32_t c = (b & 3u) | ((b & 0x0cu) << 6) | ((b & 0x30u) << 12) | ((b & 0xc0u) << 18);
    const uint32_t t = __vsub4(c, 0x01010101u);  // code - 1 in each byte, no borrow between them
    *reinterpret_cast<uint32_t*>(trits + 4 * i) = t;
  }
}

}  // namespace

cudaError_t launch_unpack_pq2(const uint8_t* wq, int8_t* trits, int64_t N, int64_t K,
                              cudaStream_t st) {
  const int64_t total = N * K / 4;
  int64_t grid = (total + 255) / 256;
  if (grid > 152 * 32) grid = 152 * 32;
  if (grid < 1) return cudaSuccess;
  unpack_pq2_kernel<<<(unsigned)grid, 256, 0, st>>>(wq, trits, total);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* wq, int8_t* trits, int64_t N, int64_t K,
                          cudaStream_t st) {
  const int64_t total = N * (K / kBlockWeights) * kBlockBytes;
  int64_t grid = (total + 255) / 256;
  if (grid > 152 * 32) grid = 152 * 32;
  unpack_kernel<<<(unsigned)grid, 256, 0, st>>>(wq, trits, total, K);
  return cudaGetLastError();
}

}  // namespace ptq

// k_gemv.cu -- decode GEMV over PTQ1_0 weights, 1 <= M <= 8, fp32.
//
//   y[m, n] = sum_b s[n, b] * sum_{i<128} t[n, 128b + i] * x[m, 128b + i]
//
// The trit peel is the one of "A 27B model in 5.5 GB: Bonsai ternary on
// Ferrox, locally", section "What Ferrox does with it": with u = byte/256,
// digit n = f_{n+1} - 3 f_n where f_j = floor(3^j u), evaluated on the fp32
// pipe.  Summed against activations the digits telescope:
//
//   sum_{n<5} d_n x_n = sum_{j=1..4} f_j (x_{j-1} - 3 x_j) + f_5 x_4,
//
// so each byte costs five floors and five FMAs against activation-side
// coefficients c_j that are computed once per call and shared by every row.
// The trit offset (t = d - 1) is the block sum of x, also activation-side:
// sum_i t_i x_i = sum_j f_j c_j - E_b with E_b = sum_{i in b} x_i.
//
// One floor is one fused multiply-add rounded toward minus infinity: with
// T = 2^23 + byte (built by a byte permute), fma_rd(T, 3^j/256,
// 2^15 (256 - 3^j)) is exactly 2^23 + floor(3^j byte/256); subtracting 2^23
// is exact.
//
// Work split: a CTA owns 32 rows (lane = row) and its warps split the row's
// 1024-wide groups (8 blocks = 208 bytes = 13 x 16 B, loaded with 16-byte
// vector loads; each block of each row is read exactly once).  Each warp
// issues the loads of its first group before the CTA builds the coefficient
// table, so the weight stream overlaps the table build.  Coefficients live in
// shared memory; all lanes of a warp read the same coefficient (broadcast).
// Partial sums are reduced across warps in a fixed order, so results are
// bitwise reproducible.
#include <cuda_fp16.h>

#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int kCoef = kGroupBytes * 5;       // 1040 coefficients per group
constexpr int kGroupStride = kCoef + 8;      // + E_b for the 8 blocks
constexpr int kSmemBudget = 200 * 1024;      // bytes: x staging + tables

__device__ __forceinline__ float floor_pow3(float tb, int j) {
  // tb = 2^23 + byte; returns floor(3^j byte / 256) (exact)
  const float mul = (j == 1 ? 3.f : j == 2 ? 9.f : j == 3 ? 27.f : j == 4 ? 81.f : 243.f) *
                    (1.0f / 256.0f);
  const float add = 32768.0f * (256.f - (j == 1 ? 3.f : j == 2 ? 9.f : j == 3 ? 27.f
                                          : j == 4 ? 81.f : 243.f));
  return __fmaf_rd(tb, mul, add) - 8388608.0f;
}

// Builds the coefficient tables of groups [g0, g0 + gp) for all M tokens.
// x is first staged in shared memory (xs: M x gp x 1024) with 16-byte loads.
// Table layout per (m, group slot): quad q = p / 4 of byte positions,
// coefficient jf (0..4 for f_1..f_5), lane e = p % 4: [q * 20 + jf * 4 + e];
// then E_b, the block sums of x, at [1040 + b], reduced with warp shuffles.
template <int M>
__device__ void build_table(float* tab, float* xs, const float* __restrict__ x, int K, int g0,
                            int gp) {
  const int per_x = gp * kRot;
  for (int i = threadIdx.x; i < M * per_x / 4; i += blockDim.x) {
    const int m = (4 * i) / per_x, r = 4 * i - m * per_x;
    reinterpret_cast<float4*>(xs)[i] =
        __ldg(reinterpret_cast<const float4*>(x + (size_t)m * K + (size_t)g0 * kRot + r));
  }
  __syncthreads();
  const int per = gp * kGroupStride;
  for (int i = threadIdx.x; i < M * gp * kCoef; i += blockDim.x) {
    const int mg = i / kCoef, slot = i - mg * kCoef;  // mg = m * gp + gs
    const int q = slot / 20, jf = (slot % 20) / 4, e = slot % 4;
    const int p = 4 * q + e;
    const int bl = p / kBlockBytes, jj = p % kBlockBytes;
    const float* xb = xs + mg * kRot + bl * kBlockWeights;
    auto xv = [&](int n) { return 5 * jj + n < kBlockWeights ? xb[5 * jj + n] : 0.0f; };
    tab[mg * kGroupStride + slot] = jf < 4 ? fmaf(-3.0f, xv(jf + 1), xv(jf)) : xv(4);
  }
  const int lane = threadIdx.x & 31;
  for (int wb = threadIdx.x >> 5; wb < M * gp * kGroupBlocks; wb += blockDim.x >> 5) {
    const int mg = wb / kGroupBlocks, b = wb % kGroupBlocks;
    const float4 v = reinterpret_cast<const float4*>(xs + mg * kRot + b * kBlockWeights)[lane];
    float sum = (v.x + v.y) + (v.z + v.w);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) tab[mg * kGroupStride + kCoef + b] = sum;
  }
  (void)per;
}

// 16-byte read-only load issued where it is written: a volatile asm keeps
// the compiler from sinking it to its first use, so all loads of a group are
// in flight together instead of paying one memory latency each.
__device__ __forceinline__ void ld16(const void* p, uint32_t& a, uint32_t& b, uint32_t& c,
                                     uint32_t& d) {
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "l"(p));
}

// One lane = one row: the 208 bytes of group g (13 x 16 B) and its 8 scales.
__device__ __forceinline__ void load_group(const uint8_t* __restrict__ wq,
                                           const uint16_t* __restrict__ scales, int row, int g,
                                           int row_bytes, int nblk, uint32_t w[52],
                                           uint32_t sw[4]) {
  const uint8_t* src = wq + (size_t)row * row_bytes + (size_t)g * kGroupBytes;
#pragma unroll
  for (int i = 0; i < 13; ++i) ld16(src + 16 * i, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  ld16(scales + (size_t)row * nblk + 8 * g, sw[0], sw[1], sw[2], sw[3]);
}

template <int M>
__device__ __forceinline__ void compute_group(const uint32_t w[52], const uint32_t sw[4],
                                              const float* tab, int per, float acc[M]) {
  float blk[M][2];
#pragma unroll
  for (int m = 0; m < M; ++m) blk[m][0] = blk[m][1] = 0.0f;

#pragma unroll
  for (int q = 0; q < 52; ++q) {
    float f[4][5];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int p = 4 * q + e;
      const float tb = __uint_as_float(__byte_perm(w[p >> 2], 0x4B000000u, 0x7440u | (p & 3)));
      const bool tail = (p % kBlockBytes) == kBlockBytes - 1;
#pragma unroll
      for (int jf = 0; jf < 5; ++jf) f[e][jf] = (tail && jf >= 3) ? 0.0f : floor_pow3(tb, jf + 1);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float4* t4 = reinterpret_cast<const float4*>(tab + m * per) + q * 5;
#pragma unroll
      for (int jf = 0; jf < 5; ++jf) {
        const float4 c = t4[jf];
        const float cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int p = 4 * q + e;
          const bool tail = (p % kBlockBytes) == kBlockBytes - 1;
          if (tail && jf >= 3) continue;  // pad digits of byte 25
          const int bl = p / kBlockBytes;
          blk[m][bl & 1] = fmaf(f[e][jf], cv[e], blk[m][bl & 1]);
        }
      }
    }
    // close every block whose last byte lies in this quad
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int p = 4 * q + e;
      if ((p % kBlockBytes) != kBlockBytes - 1) continue;
      const int bl = p / kBlockBytes;
      const uint32_t hbits = (sw[bl >> 1] >> (16 * (bl & 1))) & 0xffffu;
      const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(hbits)));
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float eb = tab[m * per + kCoef + bl];
        acc[m] = fmaf(s, blk[m][bl & 1] - eb, acc[m]);
        blk[m][bl & 1] = 0.0f;
      }
    }
  }
}

template <int M>
__global__ void __launch_bounds__(256) gemv_ptq1_f32_kernel(const uint8_t* __restrict__ wq,
                                                            const uint16_t* __restrict__ scales,
                                                            const float* __restrict__ x,
                                                            float* __restrict__ y, int N, int K,
                                                            int groups_per_pass) {
  extern __shared__ __align__(16) float smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int row = blockIdx.x * 32 + lane;
  const int G = K / kRot, nblk = K / kBlockWeights, row_bytes = nblk * kBlockBytes;
  float* tab = smem;                                          // M x gp x 1048
  float* xs = smem + M * groups_per_pass * kGroupStride;      // M x gp x 1024
  float acc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) acc[m] = 0.0f;
  uint32_t w[52], sw[4];

  for (int g0 = 0; g0 < G; g0 += groups_per_pass) {
    const int gp = min(groups_per_pass, G - g0);
    const int per = gp * kGroupStride;
    int gs = warp;
    bool have = row < N && gs < gp;
    if (have) load_group(wq, scales, row, g0 + gs, row_bytes, nblk, w, sw);  // in flight
    build_table<M>(tab, xs, x, K, g0, gp);                                   // meanwhile
    __syncthreads();
    while (have) {
      compute_group<M>(w, sw, tab + gs * kGroupStride, per, acc);
      gs += nwarps;
      have = gs < gp;
      if (have) load_group(wq, scales, row, g0 + gs, row_bytes, nblk, w, sw);
    }
    __syncthreads();
  }
  // fixed-order reduction across warps
  float* red = smem;
#pragma unroll
  for (int m = 0; m < M; ++m) red[(warp * M + m) * 32 + lane] = acc[m];
  __syncthreads();
  if (warp == 0 && row < N) {
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float s = 0.0f;
      for (int w2 = 0; w2 < nwarps; ++w2) s += red[(w2 * M + m) * 32 + lane];
      y[(size_t)m * N + row] = s;
    }
  }
}

// Any K % 128 == 0: one thread per output row, byte-wise loads.  Serves the
// shapes the tiled kernel does not (K not a multiple of 1024).
template <int M>
__global__ void __launch_bounds__(128) gemv_ptq1_f32_any_k(const uint8_t* __restrict__ wq,
                                                           const uint16_t* __restrict__ scales,
                                                           const float* __restrict__ x,
                                                           float* __restrict__ y, int N, int K) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= N) return;
  const int nblk = K / kBlockWeights;
  const uint8_t* rw = wq + (size_t)row * nblk * kBlockBytes;
  float acc[M];
#pragma unroll
  for (int m = 0; m < M; ++m) acc[m] = 0.0f;
  for (int b = 0; b < nblk; ++b) {
    float blk[M];
#pragma unroll
    for (int m = 0; m < M; ++m) blk[m] = 0.0f;
    for (int j = 0; j < kBlockBytes; ++j) {
      const float tb = __uint_as_float(0x4B000000u | rw[b * kBlockBytes + j]);
      float fprev = 0.0f;
      for (int n = 0; n < 5 && 5 * j + n < kBlockWeights; ++n) {
        const float fnext = floor_pow3(tb, n + 1);
        const float t = fnext - 3.0f * fprev - 1.0f;
        fprev = fnext;
#pragma unroll
        for (int m = 0; m < M; ++m)
          blk[m] = fmaf(t, x[(size_t)m * K + b * kBlockWeights + 5 * j + n], blk[m]);
      }
    }
    const float s = __half2float(__ushort_as_half(scales[(size_t)row * nblk + b]));
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = fmaf(s, blk[m], acc[m]);
  }
#pragma unroll
  for (int m = 0; m < M; ++m) y[(size_t)m * N + row] = acc[m];
}

template <int M>
cudaError_t launch_m(const uint8_t* wq, const uint16_t* scales, const float* x, float* y, int N,
                     int K, cudaStream_t st) {
  if (K % kRot != 0) {
    gemv_ptq1_f32_any_k<M><<<(N + 127) / 128, 128, 0, st>>>(wq, scales, x, y, N, K);
    return cudaGetLastError();
  }
  const int G = K / kRot;
  int gp = kSmemBudget / (M * (kGroupStride + kRot) * 4);
  if (gp > G) gp = G;
  if (gp < 1) gp = 1;
  const int warps = gp < 8 ? gp : 8;
  size_t smem = (size_t)M * gp * (kGroupStride + kRot) * 4;
  const size_t red = (size_t)warps * M * 32 * 4;
  if (smem < red) smem = red;
  static bool attr_set[64] = {};  // per device; setting the attribute twice is harmless
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(gemv_ptq1_f32_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBudget + 8 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  gemv_ptq1_f32_kernel<M><<<(N + 31) / 32, 32 * warps, smem, st>>>(wq, scales, x, y, N, K, gp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const uint8_t* wq, const uint16_t* scales, const float* x, float* y,
                        int64_t M, int64_t N, int64_t K, cudaStream_t st) {
  if (N > INT32_MAX || K > INT32_MAX) return cudaErrorInvalidValue;
  const int n = (int)N, k = (int)K;
  // At most three tokens per launch: a kernel instance for more tokens no
  // longer unrolls its loop over the 52 words of a group, indexes them in
  // local memory and ran 15-30x slower (measured at M = 4 and 8).  More
  // tokens take several launches, the weights read again (mostly from L2).
  if (M > 3) {
    for (int64_t m0 = 0; m0 < M; m0 += 3) {
      const int64_t c = M - m0 < 3 ? M - m0 : 3;
      const cudaError_t e = launch_gemv(wq, scales, x + m0 * K, y + m0 * N, c, N, K, st);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  switch (M) {
    case 1: return launch_m<1>(wq, scales, x, y, n, k, st);
    case 2: return launch_m<2>(wq, scales, x, y, n, k, st);
    case 3: return launch_m<3>(wq, scales, x, y, n, k, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ptq

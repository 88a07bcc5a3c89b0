// k_gemm_tc.cu -- prefill GEMM over PTQ1_0 weights on the 5th-generation
// tensor cores (tcgen05, accumulator in TMEM).
//
//   y[m, n] = sum_b s[n, b] * sum_{i<128} t[n, 128b + i] * x[m, 128b + i]
//
// "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally", section "What
// Ferrox does with it": prefill runs a GEMM over the same packed blocks the
// decode matvec reads; the trits are peeled as floor(3^(n+1) u) - 3 floor(3^n
// u), u = byte / 256.
//
// Operands.  A = activations (16-bit, M x K), B = the weight tile expanded in
// shared memory to t * s.  Both are fp16: the block scale is an fp16 number,
// so +-s and 0 are exact and the MMA (kind::f16, fp32 accumulation in TMEM)
// needs no per-block epilogue.  Activations that arrive as bf16 are converted
// to fp16 in shared memory, in place (exact for |x| in fp16's normal range;
// bf16 values beyond +-65504 are outside the supported domain).
//
// Tile: 128 (M) x 128 (N), K consumed in 64-wide slices (one 128-byte
// swizzle atom of fp16), kStages slices in flight.  Warp roles:
//   warp 0      TMA producer: A slices (box 64 x 128, 128B swizzle) and, per
//               1024-wide group, the packed trits (box 208 B x 128 rows) and
//               scales (box 8 x 128) into a 2-deep group ring.
//   warp 1      TMEM allocation; lane 0 issues tcgen05.mma (4 per slice).
//   warps 2-3   convert bf16 A slices to fp16 in place (idle for fp16 A).
//   warps 4-7   one thread per weight row: peel the row's bytes and write the
//               fp16 values t * s in the canonical K-major 128B-swizzled
//               layout; afterwards, the epilogue (TMEM -> registers -> y).
// Every mbarrier wait is bounded; a wait that runs out raises the device
// status word, the CTA drains what it has in flight (bounded) and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int BM = 128, BN = 128, BK = 64;
constexpr int kStages = 4;
constexpr int kSliceBytes = BM * BK * 2;                    // 16 KB (A) = BN * BK * 2 (B)
constexpr int kQsBytes = BN * kGroupBytes;                  // 26,624
constexpr int kScBytes = BN * kGroupBlocks * 2;             // 2,048
constexpr int kGroupBuf = kQsBytes + kScBytes;              // 28,672 = 28 * 1024
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 22;

// shared memory layout (offsets from a 1024-aligned base)
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kSliceBytes;
constexpr int kOffQ = kOffB + kStages * kSliceBytes;
constexpr int kOffBar = kOffQ + 2 * kGroupBuf;
// barriers: a_full[S], a_ready[S], b_full[S], empty[S], q_full[2], q_empty[2], acc
constexpr int kNumBars = 4 * kStages + 4 + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;            // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;            // + alignment slack

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bounded wait for phase `parity`.  Returns false when the limit ran out or
// (when `abort` is given) another role has already aborted the CTA.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const uint32_t a = smem_u32(bar);
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if (abort && (i & 1023) == 1023 && *abort) return false;
  }
  return false;
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor of a K-major, 128B-swizzled tile whose
// 8-row x 128-byte atoms are stacked every 1024 bytes (SBO).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);        // start address
  d |= (uint64_t)1 << 16;                       // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset
  d |= (uint64_t)1 << 46;                       // descriptor version
  d |= (uint64_t)2 << 61;                       // 128-byte swizzle
  return d;
}

// Instruction descriptor: fp32 accumulator, fp16 A and B, both K-major,
// N = 128, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Byte offset of element (r, k) (k < 64) inside a 128-row, 64-wide fp16 tile
// in the canonical K-major 128B-swizzled layout.
__device__ __forceinline__ uint32_t sw128_off(int r, int k) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((k >> 3) ^ (r & 7)) << 4) + (k & 7) * 2);
}

// fp16 bits of t * s for the digit d = t + 1 (s16: fp16 bits of the scale)
__device__ __forceinline__ uint32_t trit_times(uint32_t d, uint32_t s16) {
  return d == 1u ? 0u : (d == 2u ? s16 : (s16 ^ 0x8000u));
}

// Peels 64 weights of one row (half `h` of block `bb` in the staged group)
// into the B slice at `bslice`: the fp16 values t * s, 8 per 16-byte store.
template <int h>
__device__ __forceinline__ void expand_half(const unsigned char* qrow, uint32_t s16,
                                            unsigned char* bslice, int r) {
  // weights 64h .. 64h + 63 of the block; byte j holds weights 5j .. 5j + 4
  uint32_t vals[32];  // 64 fp16, two per register, in k order
#pragma unroll
  for (int i = 0; i < 32; ++i) vals[i] = 0u;
  constexpr int w0 = 64 * h;
  constexpr int j_first = w0 / 5, j_last = (w0 + 63) / 5;
#pragma unroll
  for (int j = j_first; j <= j_last && j < kBlockBytes; ++j) {
    const uint32_t byte = qrow[j];
    uint32_t fprev = 0;
#pragma unroll
    for (int n = 0; n < 5; ++n) {
      const uint32_t pw = n == 0 ? 3u : n == 1 ? 9u : n == 2 ? 27u : n == 3 ? 81u : 243u;
      const uint32_t fnext = (byte * pw) >> 8;  // floor(3^(n+1) byte / 256)
      const uint32_t d = fnext - 3u * fprev;
      fprev = fnext;
      const int k = 5 * j + n;                    // weight index in the block
      if (k < w0 || k >= w0 + 64 || k >= kBlockWeights) continue;
      const int kk = k - w0;
      vals[kk >> 1] |= trit_times(d, s16) << (16 * (kk & 1));
    }
  }
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 v = make_uint4(vals[4 * c], vals[4 * c + 1], vals[4 * c + 2], vals[4 * c + 3]);
    *reinterpret_cast<uint4*>(bslice + sw128_off(r, 8 * c)) = v;
  }
}

template <bool kConvertA, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_s, void* __restrict__ y, int M, int N,
                   int K, int* status) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* a_full = bars;
  uint64_t* a_ready = bars + kStages;
  uint64_t* b_full = bars + 2 * kStages;
  uint64_t* empty = bars + 3 * kStages;
  uint64_t* q_full = bars + 4 * kStages;
  uint64_t* q_empty = q_full + 2;
  uint64_t* acc_full = q_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int nk = K / BK;            // 64-wide slices
  const int ng = K / kRot;          // 1024-wide groups

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_ready[s], 64);
      mbar_init(&b_full[s], 128);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 128);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // TMEM: 128 fp32 columns x 128 lanes
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // A may come from the previous kernel

  bool ok = true;
  if (warp == 0) {
    // ---- TMA producer ----------------------------------------------------------
    if (lane == 0) {
      // packed weights run one 1024-wide group ahead of the A slices
      auto issue_group = [&](int g) {
        const int qb = g & 1;
        if (g >= 2 && !mbar_wait(&q_empty[qb], ((g >> 1) - 1) & 1, abort_flag)) return false;
        const uint32_t qdst = smem_u32(smem + kOffQ + qb * kGroupBuf);
        mbar_expect_tx(&q_full[qb], kGroupBuf);
        tma_2d(qdst, &map_q, g * kGroupBytes, n0, &q_full[qb]);
        tma_2d(qdst + kQsBytes, &map_s, g * kGroupBlocks, n0, &q_full[qb]);
        return true;
      };
      ok = issue_group(0) && (ng < 2 || issue_group(1));
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kStages, round = kb / kStages;
        if (kb % 16 == 0 && kb > 0 && kb / 16 + 1 < ng) ok = issue_group(kb / 16 + 1);
        if (!ok) break;
        if (round > 0) ok = mbar_wait(&empty[s], (round - 1) & 1, abort_flag);
        if (!ok) break;
        mbar_expect_tx(&a_full[s], kSliceBytes);
        tma_2d(smem_u32(smem + kOffA + s * kSliceBytes), &map_a, kb * BK, m0, &a_full[s]);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ------------------------------------------------------------------
    if (lane == 0) {
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kStages, round = kb / kStages;
        ok = mbar_wait(kConvertA ? &a_ready[s] : &a_full[s], round & 1, abort_flag) &&
             mbar_wait(&b_full[s], round & 1, abort_flag);
        if (!ok) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a_addr = smem_u32(smem + kOffA + s * kSliceBytes);
        const uint32_t b_addr = smem_u32(smem + kOffB + s * kSliceBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)  // K = 16 per MMA: 32 bytes along the atom
          umma_f16(tmem, sw128_desc(a_addr + 32 * kk), sw128_desc(b_addr + 32 * kk),
                   (kb | kk) != 0);
        umma_commit(&empty[s]);  // frees the slice once these MMAs have read it
      }
      umma_commit(acc_full);     // all MMAs issued by this thread
    }
  } else if (warp < 4) {
    // ---- A conversion bf16 -> fp16, in place ---------------------------------------
    if (kConvertA) {
      const int t = threadIdx.x - 64;  // 0..63
      for (int kb = 0; kb < nk && ok; ++kb) {
        const int s = kb % kStages, round = kb / kStages;
        ok = mbar_wait(&a_full[s], round & 1, abort_flag);
        if (!ok) break;
        uint4* a = reinterpret_cast<uint4*>(smem + kOffA + s * kSliceBytes);
#pragma unroll 4
        for (int c = t; c < kSliceBytes / 16; c += 64) {
          uint4 v = a[c];
          uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
            const __half2 hv = __floats2half2_rn(lo, hi);
            w[i] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          a[c] = v;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&a_ready[s]);
      }
    }
  } else {
    // ---- B expansion: thread r = weight row n0 + r --------------------------------
    const int r = threadIdx.x - 128;  // 0..127
    for (int g = 0; g < ng && ok; ++g) {
      const int qb = g & 1;
      ok = mbar_wait(&q_full[qb], (g >> 1) & 1, abort_flag);
      if (!ok) break;
      const unsigned char* qrow = smem + kOffQ + qb * kGroupBuf + r * kGroupBytes;
      const uint16_t* srow =
          reinterpret_cast<const uint16_t*>(smem + kOffQ + qb * kGroupBuf + kQsBytes) + r * 8;
#pragma unroll 1
      for (int bb = 0; bb < kGroupBlocks && ok; ++bb) {
        const uint32_t s16 = srow[bb];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kb = g * 16 + bb * 2 + h;
          const int s = kb % kStages, round = kb / kStages;
          if (round > 0) ok = mbar_wait(&empty[s], (round - 1) & 1, abort_flag);
          if (!ok) break;
          unsigned char* bslice = smem + kOffB + s * kSliceBytes;
          if (h == 0)
            expand_half<0>(qrow + bb * kBlockBytes, s16, bslice, r);
          else
            expand_half<1>(qrow + bb * kBlockBytes, s16, bslice, r);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          mbar_arrive(&b_full[s]);
        }
      }
      if (ok) mbar_arrive(&q_empty[qb]);
    }
  }
  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) atomicOr(status, kDevTimeout);
  }

  // ---- epilogue: warps 4-7 read TMEM lanes 32 (warp % 4) .. + 31 -------------------
  if (warp >= 4) {
    const bool done = !*abort_flag && mbar_wait(acc_full, 0, abort_flag);
    if (done) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int q = warp & 3;
      const int row = m0 + 32 * q + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
            "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, "
            "%26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
              "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]),
              "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]),
              "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
              "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
              "=r"(v[30]), "=r"(v[31])
            : "r"(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (row < M) {
          const int ncol = n0 + c0;
          if constexpr (kOutF32) {
            float* out = static_cast<float*>(y) + (size_t)row * N + ncol;
            if (ncol + 32 <= N && (N & 3) == 0) {
#pragma unroll
              for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(out + i) =
                    make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
            } else {
              for (int i = 0; i < 32 && ncol + i < N; ++i) out[i] = __uint_as_float(v[i]);
            }
          } else {
            uint16_t* out = static_cast<uint16_t*>(y) + (size_t)row * N + ncol;
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const __nv_bfloat162 b2 =
                  __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
              pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            if (ncol + 32 <= N && (N & 7) == 0) {
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<uint4*>(out + 2 * i) = make_uint4(pk[i], pk[i + 1], pk[i + 2], pk[i + 3]);
            } else {
              for (int i = 0; i < 32 && ncol + i < N; ++i)
                out[i] = (uint16_t)(pk[i >> 1] >> (16 * (i & 1)));
            }
          }
        }
      }
    }
  }
  if (*abort_flag && warp == 1 && lane == 0) {
    // let the MMAs already issued finish before TMEM is released (bounded;
    // acc_full was committed after the issuing loop, aborted or not)
    static_cast<void>(mbar_wait(acc_full, 0, nullptr));
  }
  if (*abort_flag && warp == 0 && lane == 0) {
    // let this CTA's copies in flight land before its shared memory goes away
    for (int s = 0; s < kStages; ++s) static_cast<void>(mbar_wait(&a_full[s], 0, nullptr));
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  pdl_release();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(BN)
                 : "memory");
  }
}

// ---- host side -------------------------------------------------------------------------
template <bool kConvertA, bool kOutF32>
cudaError_t launch_t(const CUtensorMap& ma, const CUtensorMap& mq, const CUtensorMap& ms, void* y,
                     int M, int N, int K, int* status, cudaStream_t st) {
  auto kern = gemm_tc_kernel<kConvertA, kOutF32>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
  return launch_pdl(kern, grid, dim3(kThreads), (size_t)kSmemBytes, st, ma, mq, ms, y, M, N, K,
                    status);
}

}  // namespace

// Tensor-core GEMM for K % 1024 == 0 (cudaErrorNotSupported otherwise).
cudaError_t launch_gemm_tc(const uint8_t* wq, const uint16_t* scales, const void* x, Act x_t,
                           void* y, Act y_t, int64_t M, int64_t N, int64_t K, cudaStream_t st) {
  if (K % kRot != 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX ||
      (M + BM - 1) / BM > 65535)
    return cudaErrorNotSupported;
  cudaError_t e;
  const int64_t nblk = K / kBlockWeights, row_bytes = nblk * kBlockBytes;
  CUtensorMap ma, mq, ms;
  if ((e = encode_tma_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, K, M, K * 2, BK, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  if ((e = encode_tma_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, row_bytes, N, row_bytes,
                         kGroupBytes, BN, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  if ((e = encode_tma_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, nblk, N, nblk * 2,
                         kGroupBlocks, BN, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevice;
  const int m = (int)M, n = (int)N, k = (int)K;
  const bool conv = x_t == Act::BF16, f32 = y_t == Act::F32;
  if (conv && f32) return launch_t<true, true>(ma, mq, ms, y, m, n, k, status, st);
  if (conv) return launch_t<true, false>(ma, mq, ms, y, m, n, k, status, st);
  if (f32) return launch_t<false, true>(ma, mq, ms, y, m, n, k, status, st);
  return launch_t<false, false>(ma, mq, ms, y, m, n, k, status, st);
}

}  // namespace ptq

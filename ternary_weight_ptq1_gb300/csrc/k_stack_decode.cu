// k_stack_decode.cu -- the chained pre-norm feed-forward stack for 1 to 8
// decode tokens as one persistent, cooperative launch.
//
// "A 27B model in 5.5 GB: Bonsai ternary on Ferrox, locally", section "Speed,
// and where it goes", names running a whole layer without leaving the device
// as the next step.  Per layer l the stack computes
//   xn = x / sqrt(mean(x^2) + eps) * g_l,   x = x + FFN_l(xn),
// FFN_l = rotate, gate+up, SwiGLU, rotate, down, with x the fp32 residual.
//
// Every CTA of the grid (one per SM) runs every layer, as two phases
// separated by grid-wide barriers, each over the tokens in turn (a token
// after the first streams the same weight boxes again, from L2):
//   A  gate/up by table lookup: each CTA rotates the one or two 1024-blocks
//      of x * g_l its K-chunk touches, builds the lane tables and streams its
//      rows (as the stand-alone GEMV, k_gemv_lut.cu), adding each row's chunk
//      sum into a gate/up buffer.  The CTA that owns a rotation block adds
//      the block's sum of squares of x into the layer's norm statistic.
//   B  the down projection: each CTA forms h = silu(r g) * (r u) for the
//      rotation blocks its chunk touches, from the gate/up buffer and
//      r = 1 / sqrt(mean(x^2) + eps), rotates, builds tables, streams its
//      rows and adds each row's chunk sum into x itself: the residual add.
// The norm's scale is applied to g and u rather than to x:
// W (R (r x * g)) = r W (R (x * g)), since the rotation and the product are
// linear.  Two gate/up buffers and two norm statistics alternate by layer
// parity; phase A of layer l zeroes the pair layer l + 1 will use (last read
// by phase B of layer l - 1, two barriers earlier).  The chunk sums arrive
// in no fixed order, so results may differ between runs by fp32 rounding.
//
// The weights do not depend on the activations: once its CTA has arrived at
// a barrier, a warp requests the first two boxes of its next projection into
// its weight ring before it waits, so HBM keeps streaming through the barrier
// and the requests overlap the barrier's own latency.  The barrier is a
// counter in global memory (release by a fence before the arrive, acquire
// loads while polling); a barrier that does not complete within its poll
// limit raises the device status word, and every CTA then leaves at its next
// barrier after its own boxes have landed.  Data one CTA reads from
// another's writes is loaded through L2 (ld.cg).
#include <cuda_fp16.h>
#include <string.h>

#include <vector>

#include "async_util.cuh"
#include "lut_core.cuh"
#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int kStackLayers = 24;          // layers per launch (their tensor maps are parameters)
constexpr uint32_t kSpinLimit = 1u << 22;  // polls of one grid barrier before it gives up

// One projection's geometry, the same for every layer.
struct Proj {
  int N, nblk, words, nch, cpc;
};

struct StackArgs {
  CUtensorMap tw_gu[kStackLayers], ts_gu[kStackLayers];  // gate/up trits, scales
  CUtensorMap tw_d[kStackLayers], ts_d[kStackLayers];    // down trits, scales
  const int8_t* signs_in[kStackLayers];
  const int8_t* signs_mid[kStackLayers];
  const float* norm_w[kStackLayers];
  float* x;         // H: the residual stream (phase B adds into it)
  float* gu[2];     // M x 2I each: gate/up row sums of even / odd layers
  float* ss[2];     // M each: sums of squares of the x rows at even / odd layers
  unsigned* bar;    // this launch's barrier counter, zero at launch
  int* status;
  Proj pgu, pd;
  int L, l0, M, H, I;  // l0: stack index of this launch's first layer; M tokens
  float eps;
};

// This CTA's and warp's share of one projection.
struct Work {
  int c, ws, we, ra, rb, nbat, xsw;
};

__device__ __forceinline__ Work work_of(const Proj& p, int cta, int warp) {
  Work w;
  if (cta >= p.nch * p.cpc) {
    w.c = w.ws = w.we = w.ra = w.rb = w.xsw = 0;
    w.nbat = 0;
    return w;
  }
  w.c = cta / p.cpc;
  const int k = cta % p.cpc;
  const int R0 = (int)((long long)k * p.N / p.cpc);
  const int R1 = (int)((long long)(k + 1) * p.N / p.cpc);
  const int Q = p.words / 4;
  w.ws = 4 * (int)((long long)w.c * Q / p.nch);
  w.we = 4 * (int)((long long)(w.c + 1) * Q / p.nch);
  const int nr = R1 - R0;
  w.ra = R0 + (int)((long long)warp * nr / kWarps);
  w.rb = R0 + (int)((long long)(warp + 1) * nr / kWarps);
  w.nbat = (w.rb - w.ra + kBoxRows - 1) / kBoxRows;
  w.xsw = ((4 * w.ws / kBlockBytes) >> 1) & ~3;
  return w;
}

__device__ __forceinline__ float4 ldcg4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

// Grid-wide barrier number `n` (0, 1, ...), in two halves: grid_arrive
// publishes this CTA's writes and counts it in; grid_wait returns once the
// counter reaches (n + 1) * gridDim.x.  Work that reads nothing other CTAs
// write (requesting weight boxes) may run between the two.  grid_wait
// returns false (in every thread of the CTA) when the wait ran out or
// another CTA has raised the status word.
__device__ __forceinline__ void grid_arrive(unsigned* ctr) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // release: this CTA's writes before its arrival
    atomicAdd(ctr, 1u);
  }
}

__device__ __forceinline__ bool grid_wait(unsigned* ctr, unsigned n, int* status,
                                          uint32_t limit = kSpinLimit) {
  int ok = 1;
  if (threadIdx.x == 0) {
    const unsigned target = (n + 1u) * gridDim.x;
    uint32_t i = 0;
    for (;; ++i) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= target) break;
      if (i >= limit || *reinterpret_cast<volatile int*>(status) != 0) {
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    if (!ok) atomicOr(status, kDevTimeout);
  }
  return __syncthreads_and(ok) != 0;
}

__device__ __forceinline__ bool grid_sync(unsigned* ctr, unsigned n, int* status,
                                          uint32_t limit = kSpinLimit) {
  grid_arrive(ctr);
  return grid_wait(ctr, n, status, limit);
}

// kOne: a single token, known at compile time (the token loops fold away)
template <bool kOne>
__global__ void __launch_bounds__(kThreads, 1) stack_decode_kernel(const __grid_constant__ StackArgs P) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int L = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t raw = smem_u32(smem);
  const uint32_t base = (raw + 127u) & ~127u;
  const uint32_t exch = base, xs = base + (uint32_t)kExchBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (base - raw) + kBarOff);
  const uint32_t ring_lo = base + (uint32_t)kRingOff;
  // the same layout as the stand-alone GEMV, at fixed offsets of the shared
  // window (the same for every CTA, so either all run or none does)
  const uint32_t tab = table_base(raw), tab_end = tab + (kTabEnd - kTab);
  if (ring_lo + (uint32_t)(kLowSlots * kSlotBytes) > tab ||
      tab_end + (uint32_t)((kSlots - kLowSlots) * kSlotBytes) > raw + (uint32_t)kSmemTma) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(P.status, kDevTimeout);
    return;
  }
  const int cta = blockIdx.x, G = gridDim.x;

  // ---- this warp's weight ring: batch g (counted over the whole launch) goes
  // to slot g % 2 and completes phase (g / 2) % 2 of that slot's barrier -----
  uint64_t* full = bars + kSlotsPerWarp * warp;
  const uint32_t slot0 = 2 * warp < kLowSlots ? ring_lo + (uint32_t)(2 * warp * kSlotBytes)
                                               : tab_end + (uint32_t)((2 * warp - kLowSlots) * kSlotBytes);
  const uint32_t slot1 = 2 * warp + 1 < kLowSlots
                             ? ring_lo + (uint32_t)((2 * warp + 1) * kSlotBytes)
                             : tab_end + (uint32_t)((2 * warp + 1 - kLowSlots) * kSlotBytes);
  int issued = 0, done = 0;  // batches requested / consumed by this warp
  auto request = [&](const Work& w, const CUtensorMap* tw, const CUtensorMap* ts, int b) {
    const int s = issued & 1;
    const uint32_t dst = s ? slot1 : slot0;
    if (L == 0) {
      mbar_expect_tx(&full[s], (uint32_t)kSlotBytes);
      tma_2d(dst, tw, w.ws, w.ra + kBoxRows * b, &full[s]);
      tma_2d(dst + (uint32_t)kSlotTrits, ts, w.xsw, w.ra + kBoxRows * b, &full[s]);
    }
    ++issued;
  };
  // the first two batches of a projection
  auto prefetch = [&](const Work& w, const CUtensorMap* tw, const CUtensorMap* ts) {
    for (int b = 0; b < w.nbat && b < 2; ++b) request(w, tw, ts, b);
  };
  // let the boxes still in flight land before the CTA's shared memory goes
  auto drain = [&]() {
    for (; done < issued; ++done)
      static_cast<void>(mbar_wait(&full[done & 1], (uint32_t)((done >> 1) & 1), nullptr));
  };

  if (L == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // ---- one projection: stage and rotate the activations of this CTA's
  // chunk (load(f, i): elements 4i..4i+3 of rotation block f), build the
  // tables, stream the rows adding each row's sum into out[row]; the first
  // two boxes were requested earlier ------------------------------------------
  auto gemv = [&](const Proj& p, const Work& w, const CUtensorMap* tw, const CUtensorMap* ts,
                  const int8_t* signs, float* out, auto load) -> bool {
    if (cta >= p.nch * p.cpc) return true;
    const int Wc = w.we - w.ws;
    const bool live = L < Wc;
    const int wl = w.ws + (live ? L : Wc - 1);
    const int P0 = 4 * wl;
    const int bA = P0 / kBlockBytes, bB = (P0 + 2) / kBlockBytes;
    const uint32_t ssel = (bB != bA) ? 0x3210u : ((bA & 1) ? 0x3232u : 0x1010u);
    const uint32_t soff = 4u * (uint32_t)((bA >> 1) - w.xsw);
    int f0, f1;
    chunk_rot_blocks<false>(w.ws, w.we, &f0, &f1);
    const int half = warp >> 3, g8 = threadIdx.x & 255;
    auto bar = [half]() { asm volatile("bar.sync %0, 256;" ::"r"(1 + half) : "memory"); };
    if (f0 + half <= f1) {
      const int f = f0 + half;
      rotate_block([&](int i) { return load(f, i); }, signs + (size_t)f * kRot,
                   exch + (uint32_t)(half * kRot * 4), xs + (uint32_t)(half * kRot * 4), g8, bar);
    }
    __syncthreads();
    build_tables<false>(w.ws, live, xs, f0 * kRot, tab);
    __syncthreads();

    const uint32_t lb0 = tab + 4u * L, lb1 = lb0 + 128u, lb2 = lb0 + 0x10000u, lb3 = lb2 + 128u;
    const Lanes ln{lb0, lb1, lb2, lb3, ssel, 0u, 0u, 0u};
    bool ok = true;
    for (int b = 0; b < w.nbat; ++b, ++done) {
      const int s = done & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (uint32_t)((done >> 1) & 1), nullptr));
      if (!ok) break;
      const uint32_t slot = s ? slot1 : slot0;
      uint32_t wv[kBoxRows], sw[kBoxRows];
      uint32_t seen = 0u;
#pragma unroll
      for (int r = 0; r < kBoxRows; ++r) {
        wv[r] = lds_u32(slot + (uint32_t)(r * kChunkWords * 4) + 4u * (uint32_t)L);
        sw[r] = lds_u32(slot + (uint32_t)kSlotTrits + (uint32_t)(r * kBoxScaleWords * 4) + soff);
        seen ^= wv[r] ^ sw[r];
      }
      // the slot is read: `seen` consumes every load, so the data is in
      // registers before the warp synchronises and the slot goes to the TMA
      // for the batch two ahead (completed reads need no proxy fence)
      asm volatile("" ::"r"(seen));
      __syncwarp();
      if (b + 2 < w.nbat) request(w, tw, ts, b + 2);
      float k1[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        k1[j] = fold(lane_value(wv[j], sw[j], ln), lane_value(wv[j + 8], sw[j + 8], ln), L & 16, 16);
      float k2[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) k2[j] = fold(k1[j], k1[j + 4], L & 8, 8);
      const float k3a = fold(k2[0], k2[2], L & 4, 4), k3b = fold(k2[1], k2[3], L & 4, 4);
      float v = fold(k3a, k3b, L & 2, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      const int row = w.ra + kBoxRows * b + (L >> 1);
      if (!(L & 1) && row < w.rb) atomicAdd(out + row, v);
    }
    return ok;
  };

  // whether this CTA adds rotation block `f` of x into the norm statistic:
  // the first CTA (k = 0) of the first chunk that touches the block
  auto owns_block = [&](const Proj& p, const Work& w, int f) -> bool {
    if (cta >= p.nch * p.cpc || cta % p.cpc != 0) return false;
    int f0, f1;
    chunk_rot_blocks<false>(w.ws, w.we, &f0, &f1);
    if (f < f0 || f > f1) return false;
    if (w.c == 0) return true;
    const int Q = p.words / 4;
    const int pws = 4 * (int)((long long)(w.c - 1) * Q / p.nch);
    int pf0, pf1;
    chunk_rot_blocks<false>(pws, w.ws, &pf0, &pf1);
    return pf1 < f;
  };

  unsigned nbar = 0;
  bool ok = true;
  const Work wa = work_of(P.pgu, cta, warp), wb = work_of(P.pd, cta, warp);
  const int I = P.I, M = kOne ? 1 : P.M;
  prefetch(wa, &P.tw_gu[0], &P.ts_gu[0]);
  for (int l = 0; l < P.L && ok; ++l) {
    const int par = (P.l0 + l) & 1;
    float* gu = P.gu[par];   // M x 2I
    float* ssl = P.ss[par];  // M
    // ---- A: gate/up of every token, and the sums of squares of x ----
    {
      // zero the buffers the next layer adds into (a contiguous slice per CTA)
      float* gn = P.gu[par ^ 1];
      const int tot = M * 2 * I;
      const int per = (tot + 4 * G - 1) / (4 * G) * 4;
      const int z1 = min(tot, (cta + 1) * per);
      for (int i = cta * per + 4 * threadIdx.x; i < z1; i += 4 * kThreads)
        *reinterpret_cast<float4*>(gn + i) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (cta == 0 && threadIdx.x < M) P.ss[par ^ 1][threadIdx.x] = 0.0f;
    }
    const float* g = P.norm_w[l];
    for (int m = 0; m < M && ok; ++m) {
      // token m > 0 streams the same boxes again (from L2)
      if (m > 0) prefetch(wa, &P.tw_gu[l], &P.ts_gu[l]);
      const float* xm = P.x + (size_t)m * P.H;
      float sq = 0.0f;  // this thread's share of one rotation block's sum of squares
      bool okm = gemv(P.pgu, wa, &P.tw_gu[l], &P.ts_gu[l], P.signs_in[l], gu + (size_t)m * 2 * I,
                      [&](int f, int i) {
                        const float4 a = ldcg4(xm + (size_t)f * kRot + 4 * i);
                        const float4 s = __ldg(reinterpret_cast<const float4*>(g + (size_t)f * kRot) + i);
                        sq = fmaf(a.x, a.x, fmaf(a.y, a.y, fmaf(a.z, a.z, a.w * a.w)));
                        return make_float4(a.x * s.x, a.y * s.y, a.z * s.z, a.w * s.w);
                      });
      if (cta < P.pgu.nch * P.pgu.cpc) {
        int f0, f1;
        chunk_rot_blocks<false>(wa.ws, wa.we, &f0, &f1);
        const int f = f0 + (warp >> 3);
        if (f <= f1 && owns_block(P.pgu, wa, f)) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
          if (L == 0) atomicAdd(ssl + m, sq);
        }
      }
      // every warp of the CTA leaves the token loop together
      ok = __syncthreads_and(okm) != 0;
    }
    if (!ok) {
      if (threadIdx.x == 0) atomicOr(P.status, kDevTimeout);
      break;
    }
    // arrive, request B's first boxes while the others arrive, then wait
    grid_arrive(P.bar);
    prefetch(wb, &P.tw_d[l], &P.ts_d[l]);
    ok = grid_wait(P.bar, nbar++, P.status);
    if (!ok) break;
    // ---- B: h from the gate/up sums, the down projection into each x row ----
    for (int m = 0; m < M && ok; ++m) {
      if (m > 0) prefetch(wb, &P.tw_d[l], &P.ts_d[l]);
      const float* gum = gu + (size_t)m * 2 * I;
      const float r = 1.0f / sqrtf(__ldcg(ssl + m) / (float)P.H + P.eps);
      bool okm = gemv(P.pd, wb, &P.tw_d[l], &P.ts_d[l], P.signs_mid[l], P.x + (size_t)m * P.H,
                      [&](int f, int i) {
                        const float4 a = ldcg4(gum + (size_t)f * kRot + 4 * i);
                        const float4 b = ldcg4(gum + I + (size_t)f * kRot + 4 * i);
                        auto hv = [r](float gg, float uu) {
                          gg *= r;
                          return gg / (1.0f + expf(-gg)) * (uu * r);
                        };
                        return make_float4(hv(a.x, b.x), hv(a.y, b.y), hv(a.z, b.z), hv(a.w, b.w));
                      });
      ok = __syncthreads_and(okm) != 0;
    }
    if (!ok) {
      if (threadIdx.x == 0) atomicOr(P.status, kDevTimeout);
      break;
    }
    if (l + 1 < P.L) {
      grid_arrive(P.bar);
      prefetch(wa, &P.tw_gu[l + 1], &P.ts_gu[l + 1]);
      ok = grid_wait(P.bar, nbar++, P.status);
    }
  }
  drain();
}

int g_stack_ready[64];  // per device: kernel attributes set

// The grid barrier made to run out, without a fault: CTA 0 never arrives,
// so the others poll up to their (short) limit, raise the status word and
// return.  Nothing else is in flight.
__global__ void selftest_grid_kernel(unsigned* ctr, int* status) {
  if (blockIdx.x == 0) return;
  static_cast<void>(grid_sync(ctr, 0u, status, 4096u));
}

__device__ unsigned g_selftest_ctr;

}  // namespace

cudaError_t launch_selftest_grid_timeout(cudaStream_t st) {
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevice;
  void* ctr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ctr, g_selftest_ctr);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(ctr, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  selftest_grid_kernel<<<8, 32, 0, st>>>(static_cast<unsigned*>(ctr), status);
  return cudaGetLastError();
}

size_t stack_decode_ss_bytes(int64_t M) { return (size_t)(2 * M) * sizeof(float); }
size_t stack_decode_bar_bytes(int64_t L) {
  return (size_t)((L + kStackLayers - 1) / kStackLayers) * sizeof(unsigned);
}

// The device's SM count once the kernel can run there (its attributes set,
// one CTA per SM resident), else an error.
static cudaError_t stack_device(int* sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (sms > 1024) return cudaErrorNotSupported;
  if (!g_stack_ready[dev]) {
    for (auto kern : {stack_decode_kernel<true>, stack_decode_kernel<false>}) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTma);
      if (e != cudaSuccess) return e;
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmemTma);
      if (e != cudaSuccess) return e;
      if (per_sm < 1) return cudaErrorNotSupported;
    }
    g_stack_ready[dev] = 1;
  }
  *sms_out = sms;
  return cudaSuccess;
}

bool stack_decode_supported(int64_t H, int64_t I) {
  if (H <= 0 || I <= 0 || H % kRot || I % kRot || H > (1 << 24) || I > (1 << 24)) return false;
  if (device_status_ptr() == nullptr) return false;
  int sms = 0;
  if (stack_device(&sms) != cudaSuccess) return false;
  const int64_t a = gemv_lut_chunks(H), b = gemv_lut_chunks(I);
  return a >= 1 && b >= 1 && a <= sms && b <= sms;
}

// Runs layers [0, L) of the stack as ceil(L / 24) cooperative launches of
// one CTA per SM.
cudaError_t launch_stack_decode(const ptq_ffn_layer* layers, int64_t L, float* x, int64_t M,
                                float* gu0, float* gu1, float* ss, unsigned* bars, int64_t H,
                                int64_t I, float eps, cudaStream_t st) {
  if (L <= 0 || M <= 0) return cudaSuccess;
  if (M > kStackMaxTokens) return cudaErrorNotSupported;
  if (!stack_decode_supported(H, I)) return cudaErrorNotSupported;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevice;
  int sms = 0;
  cudaError_t e = stack_device(&sms);
  if (e != cudaSuccess) return e;
  Proj pg, d;
  const int nblk_gu = (int)(H / kBlockWeights), nblk_d = (int)(I / kBlockWeights);
  pg.N = (int)(2 * I);
  pg.nblk = nblk_gu;
  pg.words = 13 * nblk_gu / 2;
  pg.nch = (int)gemv_lut_chunks(H);
  d.N = (int)H;
  d.nblk = nblk_d;
  d.words = 13 * nblk_d / 2;
  d.nch = (int)gemv_lut_chunks(I);
  if (pg.nch < 1 || d.nch < 1 || pg.nch > sms || d.nch > sms) return cudaErrorNotSupported;
  pg.cpc = (int)gemv_lut_ctas_per_chunk(sms, pg.nch, pg.N);
  d.cpc = (int)gemv_lut_ctas_per_chunk(sms, d.nch, d.N);
  // every launch's arguments (tensor maps included) before the first launch
  const int64_t nl = (L + kStackLayers - 1) / kStackLayers;
  std::vector<StackArgs> args((size_t)nl);
  for (int64_t j = 0; j < nl; ++j) {
    StackArgs& A = args[(size_t)j];
    memset(&A, 0, sizeof A);
    const int64_t l0 = j * kStackLayers;
    const int n = (int)(L - l0 < kStackLayers ? L - l0 : kStackLayers);
    for (int i = 0; i < n; ++i) {
      const ptq_ffn_layer& ly = layers[l0 + i];
      if (encode_tma_2d(&A.tw_gu[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, ly.wgu_q, (uint64_t)pg.words,
                        (uint64_t)pg.N, (uint64_t)pg.words * 4, kChunkWords, kBoxRows,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess ||
          encode_tma_2d(&A.ts_gu[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, ly.wgu_s,
                        (uint64_t)(nblk_gu / 2), (uint64_t)pg.N, (uint64_t)nblk_gu * 2,
                        kBoxScaleWords, kBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess ||
          encode_tma_2d(&A.tw_d[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, ly.wd_q, (uint64_t)d.words,
                        (uint64_t)d.N, (uint64_t)d.words * 4, kChunkWords, kBoxRows,
                        CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess ||
          encode_tma_2d(&A.ts_d[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, ly.wd_s,
                        (uint64_t)(nblk_d / 2), (uint64_t)d.N, (uint64_t)nblk_d * 2,
                        kBoxScaleWords, kBoxRows, CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess)
        return cudaErrorNotSupported;
      A.signs_in[i] = ly.signs_in;
      A.signs_mid[i] = ly.signs_mid;
      A.norm_w[i] = ly.norm_w;
    }
    A.x = x;
    A.gu[0] = gu0;
    A.gu[1] = gu1;
    A.ss[0] = ss;
    A.ss[1] = ss + M;
    A.M = (int)M;
    A.bar = bars + j;
    A.status = status;
    A.pgu = pg;
    A.pd = d;
    A.L = n;
    A.l0 = (int)l0;
    A.H = (int)H;
    A.I = (int)I;
    A.eps = eps;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemTma;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the first layer adds into zeroed buffers (each later layer's are zeroed
  // inside the kernel, by the layer before it)
  e = cudaMemsetAsync(bars, 0, stack_decode_bar_bytes(L), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(gu0, 0, (size_t)(M * 2 * I) * sizeof(float), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(gu1, 0, (size_t)(M * 2 * I) * sizeof(float), st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ss, 0, stack_decode_ss_bytes(M), st);
  int64_t j = 0;
  for (; j < nl && e == cudaSuccess; ++j)
    e = M == 1 ? cudaLaunchKernelEx(&cfg, stack_decode_kernel<true>, args[(size_t)j])
               : cudaLaunchKernelEx(&cfg, stack_decode_kernel<false>, args[(size_t)j]);
  // a device whose SMs are partly held elsewhere (MPS, a green context) cannot
  // take the whole grid at once: when the first launch is refused nothing
  // ran, and the caller takes the per-layer path (the memsets only cleared
  // scratch)
  if (e == cudaErrorCooperativeLaunchTooLarge && j == 1) {
    static_cast<void>(cudaGetLastError());
    return cudaErrorNotSupported;
  }
  return e;
}

}  // namespace ptq

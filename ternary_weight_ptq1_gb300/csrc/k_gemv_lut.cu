// k_gemv_lut.cu -- decode GEMV over PTQ1_0 weights at M = 1 by table lookup.
//
//   y[n] = sum_b s[n, b] * sum_{i<128} t[n, 128b + i] * x[128b + i]
//
// A PTQ1_0 byte carries five trits ("A 27B model in 5.5 GB: Bonsai ternary on
// Ferrox, locally", section "What Bonsai is"), so its whole contribution
// sum_{i<5} t_i x_{5q+i} depends only on the byte value and on the five
// activations at its position.  For each byte position p of a K-chunk this
// kernel tabulates
//
//   T_p[e] = sum_{i<5} (d_i(e) - 1) x_{5q+i},   e = 0..255,
//
// where d_i(e) is digit i of the page's peel (section "What Ferrox does with
// it": digit n = floor(3^(n+1) u) - 3 floor(3^n u), u = e / 256).  Those are
// the base-3 digits of V(e) = floor(243 e / 256), the identity that makes the
// decode total over all 256 byte values.  A weight byte then costs one byte
// permute (which forms the table address) and one shared-memory load, and
// the per-block scale is applied in fp32 to the sum of the lookups that fall
// into that block.  The peel itself runs once per table entry, as the two
// partial sums A[V / 27] (digits 0, 1) + B[V % 27] (digits 2..4).
//
// Layout of the work.  A row of W has 13 * nblk / 2 32-bit words of trits.
// They are cut into nch chunks of at most 32 words.  A CTA owns one chunk and
// a range of rows, and lane L of every warp owns word L of the chunk, i.e.
// byte positions 4L..4L+3.  The four tables of lane L live in shared-memory
// bank L only (entry e of position j at 0x10000 * (1 + j/2) + 256 e +
// 128 (j%2) + 4L from the start of the CTA's shared window), so the 32
// lookups of a warp never conflict, whatever the bytes are.  The table
// region starts 0x10000 into the window, so one byte permute builds the
// whole address: byte 1 is the weight byte, byte 0 the lane's column, bytes
// 2-3 the region (and, in a cluster, the CTA's rank).
//
// Two kernels stream the rows.  The register-ring kernel (any K/128 even)
// keeps 16 rows of 4-byte coalesced loads in flight in registers and sums
// the 32 lanes of 16 rows through a padded shared-memory transpose.  The
// TMA-fed kernel (K % 1024 == 0) is described before LutTmaArgs.  In both the
// first weight loads are issued before griddepcontrol.wait (the weights do
// not depend on the previous kernel), and every row becomes one fp32 value
// per lane, the block scales of the lane's two half-words applied.  The nch
// chunk sums of a row are added in a fixed chunk order, so the result is
// bitwise reproducible: by a second kernel from part[c][n], or, at one token,
// by the row group's own cluster in distributed shared memory.  Only the
// cluster waits on other CTAs: its hardware barriers, which every CTA of
// the cluster reaches.
#include <cuda_fp16.h>

#include <atomic>

#include "async_util.cuh"
#include "lut_core.cuh"
#include "ptq_internal.cuh"

namespace ptq {
namespace {

constexpr int kRows = 16;                  // rows per batch = prefetch distance
constexpr int kRedPitch = 36;              // words per row of a reduction buffer
constexpr int kRedBytes = kRows * kRedPitch * 4;             // 2304 per warp
constexpr int kLowBytes = kWarps * kRedBytes + kXFloats * 4;
constexpr size_t kSmemBytes = kTabEnd;     // dynamic bytes requested (covers
                                           // [base, kTabEnd) for any base)
constexpr int kMinRowsPerCta = 256;        // below this the table build dominates

struct LutArgs {
  const uint8_t* wq;
  const uint16_t* sc;
  const float* x;
  const int8_t* signs;  // non-null: x is not rotated yet (K % 1024 == 0)
  float* part;   // nch x N row sums (y itself when nch == 1)
  int N, nblk, words, nch, cpc;  // cpc: CTAs per chunk
};

// v = *p when `ok`, else v keeps its value.  The predicate sits inside the
// instruction: a conditional assignment in C++ would load into a temporary and
// copy it, and the copy would wait for the load -- the prefetch would be lost.
__device__ __forceinline__ void ldg_stream(uint32_t& v, const uint32_t* p, bool ok) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.b32 q, %2, 0;\n"
      " @q ld.global.nc.L1::no_allocate.u32 %0, [%1];\n}"
      : "+r"(v)
      : "l"(p), "r"((uint32_t)ok));
}

__device__ __forceinline__ void ldg_stream(uint32_t& v, const uint32_t* p) {
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "+r"(v) : "l"(p));
}

// One batch of up to 16 rows: slot r holds row r0 + r; it is consumed, then
// refilled with row r0 + r + 16 from pb/qb + r rows (when r < nref).  Each
// lane turns its word of the row into one fp32 value (the two half-words
// with their block scales) and stores it in row r of the reduction buffer.
template <bool kFull>
__device__ __forceinline__ void rows_batch(uint32_t (&wr)[kRows], uint32_t (&sr)[kRows], int nrows,
                                           int nref, const uint32_t* pb, const uint32_t* qb,
                                           const Lanes& ln) {
  const int L = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    if (!kFull && r >= nrows) break;
    const uint32_t a0 = __byte_perm(wr[r], ln.lb0, 0x7604), a1 = __byte_perm(wr[r], ln.lb1, 0x7614);
    const uint32_t a2 = __byte_perm(wr[r], ln.lb2, 0x7624), a3 = __byte_perm(wr[r], ln.lb3, 0x7634);
    const uint32_t s2 = __byte_perm(sr[r], 0u, ln.ssel);
    const uint32_t* p = pb + (size_t)((uint32_t)r * ln.wrow);
    const uint32_t* q = qb + (size_t)((uint32_t)r * ln.srow);
    if (kFull) {
      ldg_stream(wr[r], p);
      ldg_stream(sr[r], q);
    } else {
      ldg_stream(wr[r], p, r < nref);
      ldg_stream(sr[r], q, r < nref);
    }
    const float t0 = lds_f32(a0), t1 = lds_f32(a1), t2 = lds_f32(a2), t3 = lds_f32(a3);
    const float sA = __half2float(__ushort_as_half((unsigned short)(s2 & 0xffffu)));
    const float sB = __half2float(__ushort_as_half((unsigned short)(s2 >> 16)));
    sts_f32(ln.red + 4u * (uint32_t)(r * kRedPitch + L), fmaf(t2 + t3, sB, (t0 + t1) * sA));
  }
}

// Sum of the 32 lane values of each row of the batch, in a fixed order:
// lanes L and L + 16 each add half of row L % 16.
__device__ __forceinline__ void reduce_batch(uint32_t red, int L, float* out, int r0, int rb) {
  __syncwarp();
  const int rr = L & 15, h = L >> 4;
  const uint32_t src = red + 4u * (uint32_t)(rr * kRedPitch + 16 * h);
  float acc = 0.0f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = lds_f32x4(src + 16u * q);
    acc += (v.x + v.y) + (v.z + v.w);
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 16);
  if (h == 0 && r0 + rr < rb) out[r0 + rr] = acc;
  __syncwarp();
}

// Entries e = 64 R .. 64 R + 63 of one table: T[e] = A[V / 27] + B[V % 27].

__global__ void __launch_bounds__(kThreads, 1) gemv_lut_kernel(const LutArgs P) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int L = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t base = (smem_u32(smem) + 15u) & ~15u;
  // The tables sit at a fixed offset of the shared window; the layout needs
  // the dynamic window to start low enough.  (It starts after the 1 KB the
  // driver reserves.)
  const uint32_t tab = table_base(smem_u32(smem));
  if (base + (uint32_t)kLowBytes > tab) return;
  const uint32_t red = base + (uint32_t)(warp * kRedBytes);
  const uint32_t xs = base + (uint32_t)(kWarps * kRedBytes);

  // ---- this CTA's chunk and rows ------------------------------------------------
  const int c = blockIdx.x / P.cpc, k = blockIdx.x % P.cpc;
  const int R0 = (int)((long long)k * P.N / P.cpc);
  const int R1 = (int)((long long)(k + 1) * P.N / P.cpc);
  const int ws = (int)((long long)c * P.words / P.nch);
  const int we = (int)((long long)(c + 1) * P.words / P.nch);
  const int Wc = we - ws;                      // 1..32 words
  const bool live = L < Wc;
  const int wl = ws + (live ? L : Wc - 1);     // lanes past the chunk re-read its last word
  const int P0 = 4 * wl;                       // first byte of the word within the row
  const int bA = P0 / kBlockBytes, bB = (P0 + 2) / kBlockBytes;
  // A block boundary can only fall in the middle of a word (26 is even), and
  // then the first half's block is even, so the two scales are the two halves
  // of one aligned 32-bit word.  The permute puts s[bA] low and s[bB] high.
  const uint32_t ssel = (bB != bA) ? 0x3210u : ((bA & 1) ? 0x3232u : 0x1010u);
  const int pw = bA >> 1;

  const int nr = R1 - R0;
  const int ra = R0 + (int)((long long)warp * nr / kWarps);
  const int rb = R0 + (int)((long long)(warp + 1) * nr / kWarps);

  // ---- weight prefetch (independent of the previous kernel) ---------------------
  // Slot r of the ring holds the trits word and the scale pair of row r0 + r
  // of the current batch.
  const size_t wrow = (size_t)P.words, srow = (size_t)(P.nblk / 2);
  uint32_t wr[kRows], sr[kRows];
  {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(P.wq) + (size_t)ra * wrow + wl;
    const uint32_t* q = reinterpret_cast<const uint32_t*>(P.sc) + (size_t)ra * srow + pw;
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      wr[r] = 0u;
      sr[r] = 0u;
      const bool ok = ra + r < rb;
      ldg_stream(wr[r], p + (size_t)r * wrow, ok);
      ldg_stream(sr[r], q + (size_t)r * srow, ok);
    }
  }

  // ---- activations of the chunk, then its tables ---------------------------------
  pdl_wait();
  stage_tables(P.x, P.signs, ws, we, live, base, xs, tab);
  __syncthreads();
  pdl_release();  // the reduction kernel may start its prologue

  // ---- main loop: 16 rows per batch ----------------------------------------------
  // address of entry e of position j: byte 0 = lane column (+128 for odd j),
  // byte 1 = e, byte 2 = region 1 + j / 2
  const uint32_t lb0 = tab + 4u * L, lb1 = lb0 + 128u, lb2 = lb0 + 0x10000u, lb3 = lb2 + 128u;
  const Lanes ln{lb0, lb1, lb2, lb3, ssel, red, (uint32_t)P.words, (uint32_t)(P.nblk / 2)};
  const uint32_t* pw0 = reinterpret_cast<const uint32_t*>(P.wq) + (size_t)ra * wrow + wl;
  const uint32_t* qw0 = reinterpret_cast<const uint32_t*>(P.sc) + (size_t)ra * srow + pw;
  float* out = P.part + (size_t)c * P.N;
  int r0 = ra;
  // batches whose 16 rows and 16 refills are all inside the warp's rows
  for (; r0 + 2 * kRows <= rb; r0 += kRows) {
    const size_t next = (size_t)(r0 - ra + kRows);
    rows_batch<true>(wr, sr, kRows, kRows, pw0 + next * wrow, qw0 + next * srow, ln);
    reduce_batch(red, L, out, r0, rb);
  }
  for (; r0 < rb; r0 += kRows) {
    const size_t next = (size_t)(r0 - ra + kRows);
    const int nrows = rb - r0 < kRows ? rb - r0 : kRows;
    const int nref = rb - r0 - kRows;  // rows left to fetch (may be <= 0)
    rows_batch<false>(wr, sr, nrows, nref, pw0 + next * wrow, qw0 + next * srow, ln);
    reduce_batch(red, L, out, r0, rb);
  }
}

// ---- the same GEMV with the weights staged by TMA (K % 1024 == 0) --------------
// Rows are 26 nblk / 8 ... bytes apart: with nblk % 8 == 0 both weight planes
// have 16-byte aligned rows, and chunks cut at multiples of 4 words start on
// 16-byte boundaries, so a chunk's trits of 16 rows (16 x 128 bytes) and the
// 8 scale words that cover its blocks (16 x 32 bytes) are two TMA boxes.
// Each warp owns a ring of two such slots: while it works on one batch, the
// next is landing and the one after is on its way -- twice the register
// ring's depth, with no register cost.  The first two boxes of every warp
// are requested before griddepcontrol.wait, so they stream in while the
// previous kernel finishes and the tables are built.  The 32 lane values of
// a row are summed by a butterfly of shuffles (no shared memory), whose
// space the ring takes.


struct LutTmaArgs {
  CUtensorMap tw;      // trits: N rows of `words` 32-bit words, boxes 32 x 16
  CUtensorMap ts;      // scales: N rows of nblk / 2 words (fp16 pairs), boxes 8 x 16
  const float* x;
  const int8_t* signs;  // non-null: x is not rotated yet
  float* part;          // M x nch x N row sums (y itself when nch == 1)
  int* status;          // device status word (a wait that ran out)
  int N, nblk, words, nch, cpc;
  int M;                // tokens: x is M x (128 nblk), taken in turn
};


// ---- one token, a row group's chunks as one thread-block cluster ------------------
// The nch CTAs that share a row group's nr rows (one K-chunk each) can run as
// one cluster.  Each keeps its chunk's row sums in its own shared memory
// while it runs.  The rows are cut into slices of S = ceil(nr / nch), slice o
// owned by the CTA of rank o; at the end every CTA stores its sums of each
// slice into the owner's shared memory (entry [chunk][row in slice]), and
// after one cluster barrier each owner adds the nch sums of its rows in chunk
// order (the order of the reduction kernel, so the bits are the same) and
// writes y.  No workspace, no second kernel.  Both the own sums (nr floats)
// and the entries (nch S floats) take the rotation scratch and the staged
// activations, free once a CTA's tables are built (a CTA announces that with
// a barrier arrival and waits for its peers' before its first remote store):
// 16 KB, kClusterRows floats.
constexpr int kClusterRows = kBarOff / 4;
constexpr int kMaxClusterCtas = 16;  // non-portable cluster size limit

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t a, uint32_t rank, float v) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}

// kOne: a single token, known at compile time (the token loop folds away).
// kCl (with kOne): the CTAs of a row group are a cluster and write y (P.part).
template <bool kPQ2, bool kOne, bool kCl = false>
__global__ void __launch_bounds__(kThreads, 1) gemv_lut_tma_kernel(const __grid_constant__ LutTmaArgs P) {
  constexpr int kBB = kPQ2 ? 32 : kBlockBytes;  // bytes per 128-weight block
  extern __shared__ __align__(16) unsigned char smem[];
  const int L = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t raw = smem_u32(smem);
  const uint32_t base = (raw + 127u) & ~127u;
  const uint32_t exch = base, xs = base + (uint32_t)kExchBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (base - raw) + kBarOff);
  const uint32_t ring_lo = base + (uint32_t)kRingOff;
  // The tables and the upper slots sit at fixed offsets of the shared window
  // (the same in every CTA of a cluster): the dynamic memory must start low
  // enough for the lower slots to end below the tables (it starts after the
  // 1 KB the driver reserves); otherwise nothing runs, in any CTA.
  const uint32_t tab = table_base(raw), tab_end = tab + (kTabEnd - kTab);
  if (ring_lo + (uint32_t)(kLowSlots * kSlotBytes) > tab ||
      tab_end + (uint32_t)((kSlots - kLowSlots) * kSlotBytes) > raw + (uint32_t)kSmemTma)
    return;

  // ---- this CTA's chunk and rows ------------------------------------------------
  // a cluster is nch consecutive CTAs: rank = chunk
  const int c = kCl ? (int)blockIdx.x % P.nch : (int)blockIdx.x / P.cpc;
  const int k = kCl ? (int)blockIdx.x / P.nch : (int)blockIdx.x % P.cpc;
  const int R0 = (int)((long long)k * P.N / P.cpc);
  const int R1 = (int)((long long)(k + 1) * P.N / P.cpc);
  const int Q = P.words / 4;                   // 4-word quads per row
  const int ws = 4 * (int)((long long)c * Q / P.nch);
  const int we = 4 * (int)((long long)(c + 1) * Q / P.nch);
  const int Wc = we - ws;                      // 4..32 words
  const bool live = L < Wc;
  const int wl = ws + (live ? L : Wc - 1);     // lanes past the chunk take its last word's scales
  const int P0 = 4 * wl;
  // PTQ1_0: a block boundary falls mid-word at most, so the word's two halves
  // have scales s[bA], s[bB]; PQ2_0: a word (16 weights) lies in one block
  const int bA = P0 / kBB, bB = kPQ2 ? bA : (P0 + 2) / kBB;
  const uint32_t ssel = (bB != bA) ? 0x3210u : ((bA & 1) ? 0x3232u : 0x1010u);
  // the scale box starts at the chunk's first scale word rounded down to a
  // multiple of 4; a chunk spans at most 6 blocks, so 8 words cover it
  const int xsw = ((4 * ws / kBB) >> 1) & ~3;
  const uint32_t soff = 4u * (uint32_t)((bA >> 1) - xsw);

  const int nr = R1 - R0;
  const int ra = R0 + (int)((long long)warp * nr / kWarps);
  const int rb = R0 + (int)((long long)(warp + 1) * nr / kWarps);
  const int nbat = (rb - ra + kBoxRows - 1) / kBoxRows;
  // batch g of the warp's stream is batch g % nbat of token g / nbat: every
  // token streams the same rows, so the ring runs on across token boundaries
  const int M = kOne ? 1 : P.M;
  const int nall = nbat * M;

  // ---- this warp's ring; its first two boxes (weights only) -----------------------
  uint64_t* full = bars + kSlotsPerWarp * warp;
  auto slot_of = [&](int s) -> uint32_t {
    const int g = kSlotsPerWarp * warp + s;
    return g < kLowSlots ? ring_lo + (uint32_t)(g * kSlotBytes)
                         : tab_end + (uint32_t)((g - kLowSlots) * kSlotBytes);
  };
  auto request = [&](int g) {  // lane 0: batch g into slot g % 2
    const int s = g & 1, r = ra + kBoxRows * (kOne ? g : g % nbat);
    const uint32_t dst = slot_of(s);
    mbar_expect_tx(&full[s], (uint32_t)kSlotBytes);
    tma_2d(dst, &P.tw, ws, r, &full[s]);
    tma_2d(dst + (uint32_t)kSlotTrits, &P.ts, xsw, r, &full[s]);
  };
  if (L == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (nall > 0) request(0);
    if (nall > 1) request(1);
  }
  __syncwarp();

  if constexpr (kOne) {
    // One token: a single pass over the rows, written apart from the token
    // loop below, which with M fixed at 1 measured 2.4% slower per call
    // (10.93 against 10.67 us at N = 17408, K = 5120).
    // ---- activations of the chunk, then its tables ---------------------------------
    pdl_wait();
    stage_tables<kPQ2>(P.x, P.signs, ws, we, live, exch, xs, tab);
    __syncthreads();
    pdl_release();  // the reduction kernel may start its prologue
    // clustered: this CTA's staging space may now take its peers' row sums
    if constexpr (kCl) cluster_arrive();

    // ---- main loop: one box of 16 rows per batch -------------------------------------
    const uint32_t lb0 = tab + 4u * L, lb1 = lb0 + 128u, lb2 = lb0 + 0x10000u, lb3 = lb2 + 128u;
    const Lanes ln{lb0, lb1, lb2, lb3, ssel, 0u, 0u, 0u};
    float* out = P.part + (size_t)c * P.N;
    int b = 0;
    bool ok = true;
    for (; b < nbat; ++b) {
      const int s = b & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (uint32_t)((b >> 1) & 1), nullptr));
      if (!ok) break;
      const uint32_t slot = slot_of(s);
      uint32_t w[kBoxRows], sw[kBoxRows];
      uint32_t seen = 0u;
  #pragma unroll
      for (int r = 0; r < kBoxRows; ++r) {
        w[r] = lds_u32(slot + (uint32_t)(r * kChunkWords * 4) + 4u * (uint32_t)L);
        sw[r] = lds_u32(slot + (uint32_t)kSlotTrits + (uint32_t)(r * kBoxScaleWords * 4) + soff);
        seen ^= w[r] ^ sw[r];
      }
      // The slot is read: `seen` consumes every load, so all the data is in
      // registers before the warp synchronises and lane 0 hands the slot to
      // the TMA for the batch two ahead.  Completed reads need no proxy fence
      // before the asynchronous writes (a TMA pipeline's consumer hands its
      // stage back the same way, by a barrier arrival alone); the fence cost
      // 0.18 us per one-token call and 1 us per four-token call.
      asm volatile("" ::"r"(seen));
      __syncwarp();
      if (L == 0 && b + 2 < nbat) request(b + 2);
      // rows j and j + 8 meet first (lane bit 4), then the halves fold over
      // lane bits 3, 2, 1, 0: lanes 2i and 2i + 1 end with row i of the batch
      float k1[8];
  #pragma unroll
      for (int j = 0; j < 8; ++j)
        k1[j] = fold(lane_value(w[j], sw[j], ln), lane_value(w[j + 8], sw[j + 8], ln), L & 16, 16);
      float k2[4];
  #pragma unroll
      for (int j = 0; j < 4; ++j) k2[j] = fold(k1[j], k1[j + 4], L & 8, 8);
      const float k3a = fold(k2[0], k2[2], L & 4, 4), k3b = fold(k2[1], k2[3], L & 4, 4);
      float v = fold(k3a, k3b, L & 2, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      const int row = ra + kBoxRows * b + (L >> 1);
      if (!(L & 1) && row < rb) {
        if constexpr (kCl)
          sts_f32(base + 4u * (uint32_t)(row - R0), v);
        else
          out[row] = v;
      }
    }
    if (!ok) {
      if (L == 0) atomicOr(P.status, kDevTimeout);
      // let the boxes still in flight land before the CTA's shared memory goes
      for (int bb = b; bb < nbat && bb < b + 2; ++bb)
        static_cast<void>(mbar_wait(&full[bb & 1], (uint32_t)((bb >> 1) & 1), nullptr));
    }
    if constexpr (kCl) {
      // Every thread of the cluster takes both barrier phases.  After the
      // first every peer's staging space is free; after the second every
      // entry of this CTA's slice is in its shared memory, and no CTA touches
      // another's afterwards.
      const int S = (nr + P.nch - 1) / P.nch;
      const uint32_t ent = base + 4u * (uint32_t)nr;  // entries [chunk][row in slice]
      __syncthreads();                                // this CTA's row sums are written
      cluster_wait();
      for (int i = (int)threadIdx.x; i < nr; i += kThreads) {
        const int o = i / S;
        st_cluster_f32(ent + 4u * (uint32_t)(c * S + i - o * S), (uint32_t)o,
                       lds_f32(base + 4u * (uint32_t)i));
      }
      cluster_arrive();
      cluster_wait();
      const int q0 = c * S, q1 = q0 + S < nr ? q0 + S : nr;
      for (int j = (int)threadIdx.x; j < q1 - q0; j += kThreads) {
        float acc = 0.0f;
        for (int cc = 0; cc < P.nch; ++cc) acc += lds_f32(ent + 4u * (uint32_t)(cc * S + j));
        P.part[R0 + q0 + j] = acc;
      }
    }
  } else {
    // ---- per token: its activations and tables, then its rows -----------------------
    pdl_wait();
    const uint32_t lb0 = tab + 4u * L, lb1 = lb0 + 128u, lb2 = lb0 + 0x10000u, lb3 = lb2 + 128u;
    const Lanes ln{lb0, lb1, lb2, lb3, ssel, 0u, 0u, 0u};
    const size_t K = (size_t)P.nblk * kBlockWeights;
    int g = 0;  // the warp's next batch: the one its ring waits on
    bool ok = true;
    for (int m = 0; m < M; ++m) {
      // every warp is done with the previous token's tables; a warp whose wait
      // ran out stops the CTA here
      if (m > 0 && !__syncthreads_and(ok)) {
        ok = false;
        break;
      }
      stage_tables<kPQ2>(P.x + (size_t)m * K, P.signs, ws, we, live, exch, xs, tab);
      __syncthreads();
      if (m == 0) pdl_release();  // the reduction kernel may start its prologue

      // ---- main loop: one box of 16 rows per batch -----------------------------------
      float* out = P.part + ((size_t)m * P.nch + c) * P.N;
      for (int b = 0; b < nbat; ++b, ++g) {
        const int s = g & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (uint32_t)((g >> 1) & 1), nullptr));
        if (!ok) break;
        const uint32_t slot = slot_of(s);
        uint32_t w[kBoxRows], sw[kBoxRows];
        uint32_t seen = 0u;
  #pragma unroll
        for (int r = 0; r < kBoxRows; ++r) {
          w[r] = lds_u32(slot + (uint32_t)(r * kChunkWords * 4) + 4u * (uint32_t)L);
          sw[r] = lds_u32(slot + (uint32_t)kSlotTrits + (uint32_t)(r * kBoxScaleWords * 4) + soff);
          seen ^= w[r] ^ sw[r];
        }
        // The slot is read: `seen` consumes every load, so all the data is in
        // registers before the warp synchronises and lane 0 hands the slot to
        // the TMA for the batch two ahead.  Completed reads need no proxy fence
        // before the asynchronous writes (a TMA pipeline's consumer hands its
        // stage back the same way, by a barrier arrival alone); the fence cost
        // 0.18 us per one-token call and 1 us per four-token call.
        asm volatile("" ::"r"(seen));
        __syncwarp();
        if (L == 0 && g + 2 < nall) request(g + 2);
        // rows j and j + 8 meet first (lane bit 4), then the halves fold over
        // lane bits 3, 2, 1, 0: lanes 2i and 2i + 1 end with row i of the batch
        float k1[8];
  #pragma unroll
        for (int j = 0; j < 8; ++j)
          k1[j] = fold(lane_value(w[j], sw[j], ln), lane_value(w[j + 8], sw[j + 8], ln), L & 16, 16);
        float k2[4];
  #pragma unroll
        for (int j = 0; j < 4; ++j) k2[j] = fold(k1[j], k1[j + 4], L & 8, 8);
        const float k3a = fold(k2[0], k2[2], L & 4, 4), k3b = fold(k2[1], k2[3], L & 4, 4);
        float v = fold(k3a, k3b, L & 2, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        const int row = ra + kBoxRows * b + (L >> 1);
        if (!(L & 1) && row < rb) out[row] = v;
      }
    }
    if (!ok) {
      if (L == 0) atomicOr(P.status, kDevTimeout);
      // let the boxes still in flight land before the CTA's shared memory goes
      for (int gg = g; gg < nall && gg < g + 2; ++gg)
        static_cast<void>(mbar_wait(&full[gg & 1], (uint32_t)((gg >> 1) & 1), nullptr));
    }
  }
}

__device__ __forceinline__ float chunk_sum(const float* __restrict__ part, int N, int nch, int n) {
  float acc = 0.0f;
  for (int c = 0; c < nch; ++c) acc += __ldcg(part + (size_t)c * N + n);
  return acc;
}

// y[m][n] = sum over chunks c = 0..nch-1 of part[m][c][n], in that order;
// blockIdx.y = m (y is M x N).
__global__ void __launch_bounds__(256) gemv_lut_reduce_kernel(const float* __restrict__ part,
                                                              float* __restrict__ y, int N,
                                                              int nch) {
  pdl_release();
  pdl_wait();
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const size_t m = blockIdx.y;
  y[m * N + n] = chunk_sum(part + m * nch * N, N, nch, n);
}

// The same sums for a fused gate+up weight (rows 0..I-1 gate, I..2I-1 up),
// followed by h[i] = silu(g_i) * u_i with silu(a) = a / (1 + e^-a): the
// feed-forward block of "Speed, and where it goes".
__global__ void __launch_bounds__(256) gemv_lut_reduce_swiglu_kernel(
    const float* __restrict__ part, float* __restrict__ h, int N, int nch) {
  pdl_release();
  pdl_wait();
  const int I = N / 2;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= I) return;
  const float g = chunk_sum(part, N, nch, i), u = chunk_sum(part, N, nch, i + I);
  h[i] = g / (1.0f + expf(-g)) * u;
}

int g_sms[64];
// Clusters of n CTAs of the one-token kernel (PTQ1_0, PQ2_0) that the device
// holds at once, by device and n: 0 not asked yet, -1 none.
std::atomic<int> g_clusters[64][2][kMaxClusterCtas + 1];

}  // namespace

int64_t gemv_lut_chunks(int64_t K) {
  const int64_t nblk = K / kBlockWeights;
  if (K % kBlockWeights != 0 || nblk % 2 != 0) return 0;
  const int64_t words = 13 * nblk / 2;
  return (words + kChunkWords - 1) / kChunkWords;
}

size_t gemv_lut_workspace_bytes(int64_t N, int64_t K, int64_t M) {
  const int64_t nch = gemv_lut_chunks(K);
  if (nch <= 1 || M < 1) return 0;
  return (size_t)(((M * nch * N * 4) + 255) / 256 * 256);
}

static cudaError_t device_sms(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (g_sms[dev] == 0) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemv_lut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    for (auto kern : {gemv_lut_tma_kernel<false, true>, gemv_lut_tma_kernel<false, false>,
                      gemv_lut_tma_kernel<true, true>, gemv_lut_tma_kernel<true, false>,
                      gemv_lut_tma_kernel<false, true, true>, gemv_lut_tma_kernel<true, true, true>}) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTma);
      if (e != cudaSuccess) return e;
    }
    for (auto kern : {gemv_lut_tma_kernel<false, true, true>, gemv_lut_tma_kernel<true, true, true>}) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    g_sms[dev] = sms;
  }
  *out = g_sms[dev];
  return cudaSuccess;
}

bool gemv_lut_supported(int64_t N, int64_t K, bool rotate) {
  const int64_t nch = gemv_lut_chunks(K);
  if (nch == 0 || N > INT32_MAX / 2 || K > (1 << 24)) return false;
  if (rotate && K % kRot != 0) return false;
  int sms = 0;
  return device_sms(&sms) == cudaSuccess && nch <= sms;
}

// CTAs per chunk: enough to fill the SMs, but at least kMinRowsPerCta rows each.
static int64_t ctas_per_chunk(int64_t sms, int64_t nch, int64_t N) {
  int64_t cpc = sms / nch;
  const int64_t by_rows = (N + kMinRowsPerCta - 1) / kMinRowsPerCta;
  if (cpc > by_rows) cpc = by_rows;
  return cpc < 1 ? 1 : cpc;
}

int64_t gemv_lut_ctas_per_chunk(int64_t sms, int64_t nch, int64_t N) {
  return ctas_per_chunk(sms, nch, N);
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), unsigned ctas, unsigned cl,
                                      size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cl;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// How many clusters of nch one-token CTAs the device runs at once (0: none;
// asked once per device, format and nch).
template <bool kPQ2>
static int resident_clusters(int64_t nch) {
  if (nch < 2 || nch > kMaxClusterCtas) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::atomic<int>& slot = g_clusters[dev][kPQ2 ? 1 : 0][nch];
  int n = slot.load(std::memory_order_relaxed);
  if (n == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemTma;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nch;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int got = 0;
    if (cudaOccupancyMaxActiveClusters(&got, gemv_lut_tma_kernel<kPQ2, true, true>, &cfg) !=
        cudaSuccess) {
      static_cast<void>(cudaGetLastError());  // the query's own error, not sticky
      got = 0;
    }
    n = got > 0 ? got : -1;
    slot.store(n, std::memory_order_relaxed);
  }
  return n > 0 ? n : 0;
}

// Row groups for the clustered one-token kernel: as many as ctas_per_chunk
// gives when that many clusters fit at once (fewer, down to 7/8 of them, when
// not); 0 when the clustered kernel does not serve the shape.
template <bool kPQ2>
static int64_t cluster_row_groups(int64_t nch, int64_t cpc, int64_t N) {
  const int64_t fit = resident_clusters<kPQ2>(nch);
  const int64_t g = fit < cpc ? fit : cpc;
  if (g < 1 || 8 * g < 7 * cpc) return 0;
  const int64_t rows = (N + g - 1) / g;  // the most rows a group has
  return rows + nch * ((rows + nch - 1) / nch) <= kClusterRows ? g : 0;
}

// The TMA-fed kernel for `words` 32-bit words of codes per row (both planes
// need 16-byte aligned rows: K % 1024 == 0).  cudaErrorNotSupported when a
// tensor map cannot be made.
// clustered (one token, nch > 1): cpc row groups of nch CTAs, each group a
// cluster that writes y itself; `part` is then not used.
template <bool kPQ2>
static cudaError_t launch_lut_tma(const void* wq, const uint16_t* scales, const float* x,
                                  const int8_t* signs, float* y, float* part, int64_t M, int64_t N,
                                  int nblk, int words, int64_t nch, int64_t cpc, bool clustered,
                                  cudaStream_t st) {
  int* status = device_status_ptr();
  if (status == nullptr) return cudaErrorNotSupported;
  LutTmaArgs T;
  if (encode_tma_2d(&T.tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, wq, (uint64_t)words, (uint64_t)N,
                    (uint64_t)words * 4, kChunkWords, kBoxRows,
                    CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess ||
      encode_tma_2d(&T.ts, CU_TENSOR_MAP_DATA_TYPE_UINT32, scales, (uint64_t)(nblk / 2), (uint64_t)N,
                    (uint64_t)nblk * 2, kBoxScaleWords, kBoxRows,
                    CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess)
    return cudaErrorNotSupported;
  T.x = x;
  T.signs = signs;
  T.part = (nch == 1 || clustered) ? y : part;
  T.status = status;
  T.N = (int)N;
  T.nblk = nblk;
  T.words = words;
  T.nch = (int)nch;
  T.cpc = (int)cpc;
  T.M = (int)M;
  if (clustered)
    return launch_pdl_cluster(gemv_lut_tma_kernel<kPQ2, true, true>, (unsigned)(nch * cpc),
                              (unsigned)nch, kSmemTma, st, T);
  if (M == 1)
    return launch_pdl(gemv_lut_tma_kernel<kPQ2, true>, dim3((unsigned)(nch * cpc)),
                      dim3(kThreads), kSmemTma, st, T);
  return launch_pdl(gemv_lut_tma_kernel<kPQ2, false>, dim3((unsigned)(nch * cpc)), dim3(kThreads),
                    kSmemTma, st, T);
}

// The fixed-order sum of the nch chunk sums of every row (or h = silu(g) u).
// (SwiGLU: one token.)
static cudaError_t launch_chunk_sums(const float* part, float* y, int64_t M, int64_t N,
                                     int64_t nch, LutEpilogue ep, cudaStream_t st) {
  if (ep == LutEpilogue::SwiGLU)
    return launch_pdl(gemv_lut_reduce_swiglu_kernel, dim3((unsigned)((N / 2 + 255) / 256)),
                      dim3(256), 0, st, part, y, (int)N, (int)nch);
  return launch_pdl(gemv_lut_reduce_kernel, dim3((unsigned)((N + 255) / 256), (unsigned)M),
                    dim3(256), 0, st, part, y, (int)N, (int)nch);
}

// cudaErrorNotSupported when the shape does not fit this kernel (odd K/128,
// more chunks than SMs, sizes past int32; with signs, K % 1024 != 0; with the
// SwiGLU epilogue, odd N, a single chunk or M != 1); the caller then runs the
// general path.  x is M x K, y is M x N.  `part` holds
// gemv_lut_workspace_bytes(N, K, M) bytes (unused when the row has a single
// chunk).  signs != NULL: x is rotated inside the kernel.  SwiGLU: y
// receives h = silu(g) * u of the N/2 gate and N/2 up rows.
cudaError_t launch_gemv_lut(const uint8_t* wq, const uint16_t* scales, const float* x,
                            const int8_t* signs, float* y, float* part, int64_t M, int64_t N,
                            int64_t K, LutEpilogue ep, cudaStream_t st) {
  const int64_t nch = gemv_lut_chunks(K);
  if (nch == 0 || N < 1 || N > INT32_MAX / 2 || K > (1 << 24) || M < 1 || M > INT32_MAX / N)
    return cudaErrorNotSupported;
  if (signs != nullptr && K % kRot != 0) return cudaErrorNotSupported;
  if (ep == LutEpilogue::SwiGLU && (N % 2 != 0 || nch == 1 || M != 1))
    return cudaErrorNotSupported;
  int sms = 0;
  cudaError_t e = device_sms(&sms);
  if (e != cudaSuccess) return e;
  if (nch > sms) return cudaErrorNotSupported;
  if (nch > 1 && part == nullptr) return cudaErrorInvalidValue;
  const int64_t cpc = ctas_per_chunk(sms, nch, N);
  const int nblk = (int)(K / kBlockWeights), words = 13 * nblk / 2;
  // With K % 1024 == 0 both weight planes have 16-byte aligned rows: the
  // TMA-fed kernel (its 4-word aligned chunks number the same nch) takes all
  // M tokens in one launch, and one reduction sums all M x N rows.
  if (K % kRot == 0) {
    // one token: the row groups as clusters when the device holds them
    const int64_t g = (M == 1 && ep == LutEpilogue::Plain) ? cluster_row_groups<false>(nch, cpc, N)
                                                             : 0;
    e = launch_lut_tma<false>(wq, scales, x, signs, y, part, M, N, nblk, words, nch,
                              g > 0 ? g : cpc, g > 0, st);
    if (e != cudaErrorNotSupported)
      return (e != cudaSuccess || nch == 1 || g > 0) ? e
                                                     : launch_chunk_sums(part, y, M, N, nch, ep, st);
  }
  // the register-ring kernel: one token per launch, the scratch reused
  for (int64_t m = 0; m < M; ++m) {
    LutArgs A;
    A.wq = wq;
    A.sc = scales;
    A.x = x + m * K;
    A.signs = signs;
    A.part = nch == 1 ? y + m * N : part;
    A.N = (int)N;
    A.nblk = nblk;
    A.words = words;
    A.nch = (int)nch;
    A.cpc = (int)cpc;
    e = launch_pdl(gemv_lut_kernel, dim3((unsigned)(nch * cpc)), dim3(kThreads), kSmemBytes, st,
                   A);
    if (e == cudaSuccess && nch > 1) e = launch_chunk_sums(part, y + m * N, 1, N, nch, ep, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t gemv_lut_plan(int64_t M, int64_t N, int64_t K, bool pq2, LutPlan* plan) {
  const int64_t nch = pq2 ? gemv_lut_pq2_chunks(K) : gemv_lut_chunks(K);
  if (nch == 0 || K % kRot != 0 || N < 1 || N > INT32_MAX / 2 || K > (1 << 24) || M < 1 ||
      M > INT32_MAX / N)
    return cudaErrorNotSupported;
  int sms = 0;
  cudaError_t e = device_sms(&sms);
  if (e != cudaSuccess) return e;
  if (nch > sms) return cudaErrorNotSupported;
  const int64_t cpc = ctas_per_chunk(sms, nch, N);
  const int64_t g =
      M == 1 ? (pq2 ? cluster_row_groups<true>(nch, cpc, N) : cluster_row_groups<false>(nch, cpc, N))
             : 0;
  plan->ctas = (int)(nch * (g > 0 ? g : cpc));
  plan->cluster = g > 0 ? (int)nch : 0;
  plan->chunks = (int)nch;
  plan->kernels = (g > 0 || nch == 1) ? 1 : 2;
  return cudaSuccess;
}

// ---- PQ2_0 ------------------------------------------------------------------------
// A row is 8 nblk words of 2-bit codes, cut into chunks of at most 32 words.
int64_t gemv_lut_pq2_chunks(int64_t K) {
  if (K % kRot != 0 || K <= 0) return 0;
  const int64_t words = 8 * (K / kBlockWeights);
  return (words + kChunkWords - 1) / kChunkWords;
}

size_t gemv_lut_pq2_workspace_bytes(int64_t N, int64_t K, int64_t M) {
  const int64_t nch = gemv_lut_pq2_chunks(K);
  if (nch <= 1 || M < 1) return 0;
  return (size_t)(((M * nch * N * 4) + 255) / 256 * 256);
}

cudaError_t launch_gemv_lut_pq2(const uint8_t* wq, const uint16_t* scales, const float* x,
                                const int8_t* signs, float* y, float* part, int64_t M, int64_t N,
                                int64_t K, cudaStream_t st) {
  const int64_t nch = gemv_lut_pq2_chunks(K);
  if (nch == 0 || N < 1 || N > INT32_MAX / 2 || K > (1 << 24) || M < 1 || M > INT32_MAX / N)
    return cudaErrorNotSupported;
  int sms = 0;
  cudaError_t e = device_sms(&sms);
  if (e != cudaSuccess) return e;
  if (nch > sms) return cudaErrorNotSupported;
  if (nch > 1 && part == nullptr) return cudaErrorInvalidValue;
  const int nblk = (int)(K / kBlockWeights);
  const int64_t cpc = ctas_per_chunk(sms, nch, N);
  const int64_t g = M == 1 ? cluster_row_groups<true>(nch, cpc, N) : 0;
  e = launch_lut_tma<true>(wq, scales, x, signs, y, part, M, N, nblk, 8 * nblk, nch,
                           g > 0 ? g : cpc, g > 0, st);
  if (e != cudaSuccess || nch == 1 || g > 0) return e;
  return launch_chunk_sums(part, y, M, N, nch, LutEpilogue::Plain, st);
}

}  // namespace ptq

// api.cu -- the C ABI: argument validation, the (M, dtype) routing table,
// the host-side PTQ1_0 encoder and error reporting.  Every public entry point
// validates everything before it launches anything.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "ptq_internal.cuh"

namespace ptq {

static thread_local char t_msg[512];

ptq_status fail(ptq_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof t_msg, fmt, ap);
  va_end(ap);
  return s;
}

ptq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PTQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
              cudaGetErrorString(e));
}

// ---- device status word ----------------------------------------------------
static __device__ int g_device_status;
static constexpr int kMaxDevices = 64;
static std::atomic<int*> g_status_ptr[kMaxDevices];

// The status word's device address on the current device.  Only a lookup
// that succeeded is cached: a failed one (a sticky error left by an earlier
// call, a lookup attempted during stream capture) is retried by the next call.
int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return nullptr;
  int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* q = nullptr;
  if (cudaGetSymbolAddress(&q, g_device_status) != cudaSuccess || q == nullptr) return nullptr;
  g_status_ptr[dev].store(static_cast<int*>(q), std::memory_order_release);
  return static_cast<int*>(q);
}

cudaError_t read_and_clear_device_status(int* out, cudaStream_t st) {
  int* p = device_status_ptr();
  if (!p) return cudaErrorInvalidDevice;
  cudaError_t e = cudaMemcpyAsync(out, p, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(int), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e;
}

// ---- routing table ---------------------------------------------------------
// The single source of truth for which kernel serves which (dtype, M); both
// ptq_matmul and ptq_ffn dispatch through it and ptq_route reports it.
enum class Kernel { GemvF32, GemmBf16 };
struct Route {
  ptq_dtype dtype;
  int64_t m_min, m_max;
  Kernel kernel;
  const char* name;
};
static const Route kRoutes[] = {
    {PTQ_F32, 1, 8, Kernel::GemvF32, "gemv_ptq1_f32_lut"},
    {PTQ_BF16, 1, INT64_MAX, Kernel::GemmBf16, "gemm_ptq1_bf16"},
};

static const Route* find_route(int64_t M, ptq_dtype dt) {
  for (const Route& r : kRoutes)
    if (r.dtype == dt && M >= r.m_min && M <= r.m_max) return &r;
  return nullptr;
}

// ---- validation helpers ----------------------------------------------------
static bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > INT64_MAX / a) return false;
  *out = a * b;
  return true;
}

static bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

static bool dtype_ok(ptq_dtype dt) { return dt == PTQ_F32 || dt == PTQ_BF16; }

static size_t dsize(ptq_dtype dt) { return dt == PTQ_F32 ? 4 : 2; }

}  // namespace ptq

using namespace ptq;

// ---- public ABI ------------------------------------------------------------
extern "C" {

PTQ_API const char* ptq_status_str(ptq_status s) {
  switch (s) {
    case PTQ_OK: return "PTQ_OK";
    case PTQ_ERR_NULL: return "PTQ_ERR_NULL";
    case PTQ_ERR_SHAPE: return "PTQ_ERR_SHAPE";
    case PTQ_ERR_ALIGN: return "PTQ_ERR_ALIGN";
    case PTQ_ERR_VALUE: return "PTQ_ERR_VALUE";
    case PTQ_ERR_UNSUPPORTED: return "PTQ_ERR_UNSUPPORTED";
    case PTQ_ERR_WORKSPACE: return "PTQ_ERR_WORKSPACE";
    case PTQ_ERR_CUDA: return "PTQ_ERR_CUDA";
    case PTQ_ERR_TIMEOUT: return "PTQ_ERR_TIMEOUT";
    case PTQ_ERR_RANGE: return "PTQ_ERR_RANGE";
  }
  return "PTQ_ERR_UNKNOWN";
}

PTQ_API const char* ptq_last_error(void) { return t_msg; }

PTQ_API ptq_status ptq_route(int64_t M, ptq_dtype dtype, const char** name) {
  t_msg[0] = 0;
  if (!name) return fail(PTQ_ERR_NULL, "ptq_route: kernel_name is NULL");
  if (!dtype_ok(dtype)) return fail(PTQ_ERR_VALUE, "ptq_route: unknown dtype %d", (int)dtype);
  const Route* r = find_route(M, dtype);
  if (!r)
    return fail(PTQ_ERR_UNSUPPORTED, "no kernel for M=%lld dtype=%s", (long long)M,
                dtype == PTQ_F32 ? "f32" : "bf16");
  *name = r->name;
  return PTQ_OK;
}

PTQ_API ptq_status ptq1_pack(const int8_t* trits, uint8_t* wq, int64_t N, int64_t K) {
  t_msg[0] = 0;
  if (N < 0 || K <= 0 || K % kBlockWeights != 0)
    return fail(PTQ_ERR_SHAPE, "ptq1_pack: need N >= 0, K > 0, K %% 128 == 0 (N=%lld K=%lld)",
                (long long)N, (long long)K);
  int64_t total;
  if (!mul_ok(N, K, &total)) return fail(PTQ_ERR_SHAPE, "ptq1_pack: N*K overflows");
  if (total == 0) return PTQ_OK;
  if (!trits || !wq) return fail(PTQ_ERR_NULL, "ptq1_pack: NULL pointer");
  for (int64_t i = 0; i < total; ++i)
    if (trits[i] < -1 || trits[i] > 1)
      return fail(PTQ_ERR_VALUE, "ptq1_pack: trit %d at index %lld is not in {-1,0,1}",
                  (int)trits[i], (long long)i);
  const int64_t nb = K / kBlockWeights;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const int8_t* t = trits + n * K + b * kBlockWeights;
      uint8_t* out = wq + (n * nb + b) * kBlockBytes;
      for (int j = 0; j < kBlockBytes; ++j) {
        int v = 0;  // sum_i (t_i + 1) 3^(4-i), pads carry digit 1
        for (int i = 0; i < 5; ++i) {
          const int pos = 5 * j + i;
          v = v * 3 + (pos < kBlockWeights ? t[pos] + 1 : 1);
        }
        out[j] = static_cast<uint8_t>((v * 256 + 242) / 243);
      }
    }
  }
  return PTQ_OK;
}

PTQ_API ptq_status ptq1_unpack(const uint8_t* wq, int8_t* trits, int64_t N, int64_t K,
                               ptq_stream_t stream) {
  t_msg[0] = 0;
  int64_t total;
  if (N < 0 || K <= 0 || K % kBlockWeights != 0 || !mul_ok(N, K, &total))
    return fail(PTQ_ERR_SHAPE, "ptq1_unpack: bad shape N=%lld K=%lld", (long long)N,
                (long long)K);
  if (total == 0) return PTQ_OK;
  if (!wq || !trits) return fail(PTQ_ERR_NULL, "ptq1_unpack: NULL pointer");
  cudaError_t e = launch_unpack(wq, trits, N, K, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq1_unpack launch");
}

static ptq_status check_fwht(const void* x, const void* y, const int8_t* signs, int64_t M,
                             int64_t K, ptq_dtype dt, const char* who) {
  if (!dtype_ok(dt)) return fail(PTQ_ERR_VALUE, "%s: unknown dtype %d", who, (int)dt);
  int64_t total;
  if (M < 0 || K <= 0 || K % kRot != 0 || !mul_ok(M, K, &total) ||
      !mul_ok(total, (int64_t)dsize(dt), &total))
    return fail(PTQ_ERR_SHAPE, "%s: need M >= 0, K > 0, K %% 1024 == 0 (M=%lld K=%lld)", who,
                (long long)M, (long long)K);
  if (M == 0) return PTQ_OK;
  if (!x || !y || !signs) return fail(PTQ_ERR_NULL, "%s: NULL pointer", who);
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(signs, 4))
    return fail(PTQ_ERR_ALIGN, "%s: x and y need 16-byte, signs 4-byte alignment", who);
  return PTQ_OK;
}

PTQ_API ptq_status ptq_fwht(const void* x, void* y, const int8_t* signs, int64_t M, int64_t K,
                            ptq_dtype dtype, ptq_stream_t stream) {
  t_msg[0] = 0;
  ptq_status s = check_fwht(x, y, signs, M, K, dtype, "ptq_fwht");
  if (s != PTQ_OK || M == 0) return s;
  cudaError_t e =
      launch_fwht(x, act_of(dtype), y, act_of(dtype), signs, M, K,
                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_fwht launch");
}

static ptq_status check_embed(const void* table, const void* scales, const int32_t* ids,
                              const int8_t* signs, const void* out, int64_t M, int64_t V,
                              int64_t H, ptq_dtype dt, bool ptq1, const char* who) {
  if (!dtype_ok(dt)) return fail(PTQ_ERR_VALUE, "%s: unknown dtype %d", who, (int)dt);
  int64_t t;
  if (M < 0 || V < 1 || H <= 0 || H % kRot != 0 || !mul_ok(V, H, &t) || !mul_ok(t, 4, &t) ||
      !mul_ok(M, H, &t) || !mul_ok(t, 4, &t))
    return fail(PTQ_ERR_SHAPE, "%s: need M >= 0, V >= 1, H > 0, H %% 1024 == 0 (M=%lld V=%lld H=%lld)",
                who, (long long)M, (long long)V, (long long)H);
  if (M == 0) return PTQ_OK;
  if (!table || !ids || !signs || !out || (ptq1 && !scales))
    return fail(PTQ_ERR_NULL, "%s: NULL pointer", who);
  if (!aligned(table, 16) || !aligned(out, 16) || !aligned(ids, 4) || !aligned(signs, 4) ||
      (ptq1 && !aligned(scales, 16)))
    return fail(PTQ_ERR_ALIGN, "%s: the table%s and out need 16-byte, ids and signs 4-byte alignment",
                who, ptq1 ? " (wq and scales)" : "");
  return PTQ_OK;
}

PTQ_API ptq_status ptq_embed(const void* table, const int32_t* ids, const int8_t* signs, void* out,
                             int64_t M, int64_t V, int64_t H, ptq_dtype dtype,
                             ptq_stream_t stream) {
  t_msg[0] = 0;
  ptq_status s = check_embed(table, nullptr, ids, signs, out, M, V, H, dtype, false, "ptq_embed");
  if (s != PTQ_OK || M == 0) return s;
  cudaError_t e = launch_embed(table, act_of(dtype), ids, signs, out, act_of(dtype), M, V, H,
                               reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_embed launch");
}

PTQ_API ptq_status ptq_embed_ptq1(const uint8_t* wq, const uint16_t* scales, const int32_t* ids,
                                  const int8_t* signs, void* out, int64_t M, int64_t V, int64_t H,
                                  ptq_dtype out_dtype, ptq_stream_t stream) {
  t_msg[0] = 0;
  ptq_status s =
      check_embed(wq, scales, ids, signs, out, M, V, H, out_dtype, true, "ptq_embed_ptq1");
  if (s != PTQ_OK || M == 0) return s;
  cudaError_t e = launch_embed_ptq1(wq, scales, ids, signs, out, act_of(out_dtype), M, V, H,
                                    reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_embed_ptq1 launch");
}

static ptq_status check_matmul(const uint8_t* wq, const uint16_t* scales, const void* x,
                               const void* y, int64_t M, int64_t N, int64_t K, ptq_dtype dt,
                               const char* who, const Route** route) {
  if (!dtype_ok(dt)) return fail(PTQ_ERR_VALUE, "%s: unknown dtype %d", who, (int)dt);
  int64_t t;
  if (M < 0 || N < 0 || K <= 0 || K % kBlockWeights != 0 || !mul_ok(N, K, &t) ||
      !mul_ok(M, K, &t) || !mul_ok(M, N, &t) || !mul_ok(t, 4, &t))
    return fail(PTQ_ERR_SHAPE, "%s: need M, N >= 0, K > 0, K %% 128 == 0 (M=%lld N=%lld K=%lld)",
                who, (long long)M, (long long)N, (long long)K);
  if (M == 0 || N == 0) return PTQ_OK;
  *route = find_route(M, dt);
  if (!*route)
    return fail(PTQ_ERR_UNSUPPORTED, "%s: no kernel for M=%lld dtype=%s (fp32 serves M <= 8)",
                who, (long long)M, dt == PTQ_F32 ? "f32" : "bf16");
  if (!wq || !scales || !x || !y) return fail(PTQ_ERR_NULL, "%s: NULL pointer", who);
  if (!aligned(wq, 16) || !aligned(scales, 16) || !aligned(x, 16) || !aligned(y, 16))
    return fail(PTQ_ERR_ALIGN, "%s: wq, scales, x and y need 16-byte alignment", who);
  return PTQ_OK;
}

// x_t / y_t: the GEMV is fp32 in and out; the GEMM reads bf16 (public call)
// or fp16 (inside the feed-forward block) and writes bf16 (public call) or
// fp32 (the feed-forward block keeps gate/up in fp32).
// The table-lookup GEMV of the M tokens (one launch takes them in turn: its
// tables hold one token's activations at a time), then one reduction.
static cudaError_t gemv_lut_tokens(const uint8_t* wq, const uint16_t* scales, const float* x,
                                   const int8_t* signs, float* y, float* part, int64_t M,
                                   int64_t N, int64_t K, cudaStream_t st) {
  return launch_gemv_lut(wq, scales, x, signs, y, part, M, N, K, LutEpilogue::Plain, st);
}

// ws: ws_bytes of scratch, matmul_ws_bytes(M, N, K, dtype) for full speed
// (NULL when that is 0).  The GEMM runs with fewer K splits when it gets less.
static cudaError_t run_matmul(const Route* r, const uint8_t* wq, const uint16_t* scales,
                              const void* x, Act x_t, void* y, Act y_t, int64_t M, int64_t N,
                              int64_t K, void* ws, size_t ws_bytes, cudaStream_t st) {
  switch (r->kernel) {
    case Kernel::GemvF32:
      if (gemv_lut_supported(N, K, false))  // table-lookup decode, the tokens in turn
        return gemv_lut_tokens(wq, scales, static_cast<const float*>(x), nullptr,
                               static_cast<float*>(y), static_cast<float*>(ws), M, N, K, st);
      return launch_gemv(wq, scales, static_cast<const float*>(x), static_cast<float*>(y), M, N,
                         K, st);
    case Kernel::GemmBf16:
      return launch_gemm(wq, scales, x, x_t, y, y_t, M, N, K, ws, ws_bytes, st);
  }
  return cudaErrorInvalidValue;
}

// Scratch of ptq_matmul for valid arguments: the GEMV's per-chunk row sums.
static size_t matmul_ws_bytes(int64_t M, int64_t N, int64_t K, ptq_dtype dt) {
  if (dt == PTQ_F32) return (M >= 1 && M <= 8) ? gemv_lut_workspace_bytes(N, K, M) : 0;
  return gemm_tc_workspace_bytes(M, N, K);  // split-K partial sums
}

PTQ_API size_t ptq_matmul_workspace_bytes(int64_t M, int64_t N, int64_t K, ptq_dtype dtype) {
  int64_t t;
  if (!dtype_ok(dtype) || M < 0 || N < 0 || K <= 0 || K % kBlockWeights != 0 ||
      !mul_ok(N, K, &t) || !mul_ok(M, N, &t) || !mul_ok(t, 4, &t))
    return 0;
  return matmul_ws_bytes(M, N, K, dtype);
}

PTQ_API ptq_status ptq_matmul(const uint8_t* wq, const uint16_t* scales, const void* x, void* y,
                              int64_t M, int64_t N, int64_t K, ptq_dtype dtype, void* ws,
                              size_t ws_bytes, ptq_stream_t stream) {
  t_msg[0] = 0;
  const char* who = "ptq_matmul";
  const Route* r = nullptr;
  ptq_status s = check_matmul(wq, scales, x, y, M, N, K, dtype, who, &r);
  if (s != PTQ_OK || M == 0 || N == 0) return s;
  // the decode GEMV needs its scratch; the GEMM runs unsplit (or with fewer
  // K splits) on less
  const size_t need = matmul_ws_bytes(M, N, K, dtype);
  const bool required = dtype == PTQ_F32 && need > 0;
  if (required && !ws)
    return fail(PTQ_ERR_WORKSPACE, "%s: workspace is NULL (%zu bytes needed)", who, need);
  if (required && ws_bytes < need)
    return fail(PTQ_ERR_WORKSPACE, "%s: workspace has %zu bytes, %zu needed", who, ws_bytes, need);
  if (ws && !aligned(ws, 16))
    return fail(PTQ_ERR_ALIGN, "%s: workspace needs 16-byte alignment", who);
  cudaError_t e = run_matmul(r, wq, scales, x, act_of(dtype), y, act_of(dtype), M, N, K,
                             ws, ws ? ws_bytes : 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_matmul launch");
}

// Test export: the bf16 route's prefill GEMM writing its fp32 accumulator.
// Same kernel, tiles and split-K choice as ptq_matmul with PTQ_BF16; only the
// output's own bf16 rounding is left out, so the arithmetic error of the
// route can be checked against the bare 1e-2 rms(y) bound.
PTQ_API ptq_status ptq_matmul_bf16_accumulator(const uint8_t* wq, const uint16_t* scales,
                                               const void* x, float* y, int64_t M, int64_t N,
                                               int64_t K, void* ws, size_t ws_bytes,
                                               ptq_stream_t stream) {
  t_msg[0] = 0;
  const char* who = "ptq_matmul_bf16_accumulator";
  const Route* r = nullptr;
  ptq_status s = check_matmul(wq, scales, x, y, M, N, K, PTQ_BF16, who, &r);
  if (s != PTQ_OK || M == 0 || N == 0) return s;
  if (ws && !aligned(ws, 16))
    return fail(PTQ_ERR_ALIGN, "%s: workspace needs 16-byte alignment", who);
  cudaError_t e = launch_gemm(wq, scales, x, Act::BF16, y, Act::F32, M, N, K, ws,
                              ws ? ws_bytes : 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_matmul_bf16_accumulator launch");
}

// The fp32 route's other kernel, forced: the SIMT peel GEMV that the route
// runs when K/128 is odd, here on any shape, so that the two decode designs
// can be timed on the same weights.
PTQ_API ptq_status ptq_matmul_f32_peel(const uint8_t* wq, const uint16_t* scales, const float* x,
                                       float* y, int64_t M, int64_t N, int64_t K,
                                       ptq_stream_t stream) {
  t_msg[0] = 0;
  const char* who = "ptq_matmul_f32_peel";
  const Route* r = nullptr;
  ptq_status s = check_matmul(wq, scales, x, y, M, N, K, PTQ_F32, who, &r);
  if (s != PTQ_OK || M == 0 || N == 0) return s;
  const cudaError_t e = launch_gemv(wq, scales, x, y, M, N, K, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_matmul_f32_peel launch");
}

PTQ_API ptq_status ptq_gemv_plan(int64_t M, int64_t N, int64_t K, int pq2, int32_t plan[4]) {
  t_msg[0] = 0;
  if (!plan) return fail(PTQ_ERR_NULL, "ptq_gemv_plan: plan is NULL");
  LutPlan p{};
  const cudaError_t e = gemv_lut_plan(M, N, K, pq2 != 0, &p);
  if (e == cudaErrorNotSupported)
    return fail(PTQ_ERR_UNSUPPORTED,
                "ptq_gemv_plan: the TMA-fed decode GEMV does not serve M=%lld N=%lld K=%lld",
                (long long)M, (long long)N, (long long)K);
  if (e != cudaSuccess) return cuda_fail(e, "ptq_gemv_plan");
  plan[0] = p.ctas;
  plan[1] = p.cluster;
  plan[2] = p.chunks;
  plan[3] = p.kernels;
  return PTQ_OK;
}

// ---- PQ2_0 ----------------------------------------------------------------
// "Why I Am Building Another Inference Engine", section "Level 2: The short
// answer": two bits per ternary weight plus one 16-bit scale per 128
// weights.  Same routing as PTQ1_0 (fp32 M <= 8: the table-lookup GEMV,
// bf16: the tensor-core GEMM), both on the TMA-fed paths, so K % 1024 == 0.

PTQ_API ptq_status ptq2_pack(const int8_t* trits, uint8_t* wq, int64_t N, int64_t K) {
  t_msg[0] = 0;
  if (N < 0 || K <= 0 || K % kBlockWeights != 0)
    return fail(PTQ_ERR_SHAPE, "ptq2_pack: need N >= 0, K > 0, K %% 128 == 0 (N=%lld K=%lld)",
                (long long)N, (long long)K);
  int64_t total;
  if (!mul_ok(N, K, &total)) return fail(PTQ_ERR_SHAPE, "ptq2_pack: N*K overflows");
  if (total == 0) return PTQ_OK;
  if (!trits || !wq) return fail(PTQ_ERR_NULL, "ptq2_pack: NULL pointer");
  for (int64_t i = 0; i < total; ++i)
    if (trits[i] < -1 || trits[i] > 1)
      return fail(PTQ_ERR_VALUE, "ptq2_pack: trit %d at index %lld is not in {-1,0,1}",
                  (int)trits[i], (long long)i);
  for (int64_t i = 0; i < total / 4; ++i) {  // weight 4j + k: bits 2k, 2k+1 of byte j
    uint32_t v = 0;
    for (int k = 0; k < 4; ++k) v |= (uint32_t)(trits[4 * i + k] + 1) << (2 * k);
    wq[i] = static_cast<uint8_t>(v);
  }
  return PTQ_OK;
}

PTQ_API ptq_status ptq2_unpack(const uint8_t* wq, int8_t* trits, int64_t N, int64_t K,
                               ptq_stream_t stream) {
  t_msg[0] = 0;
  int64_t total;
  if (N < 0 || K <= 0 || K % kBlockWeights != 0 || !mul_ok(N, K, &total))
    return fail(PTQ_ERR_SHAPE, "ptq2_unpack: bad shape N=%lld K=%lld", (long long)N,
                (long long)K);
  if (total == 0) return PTQ_OK;
  if (!wq || !trits) return fail(PTQ_ERR_NULL, "ptq2_unpack: NULL pointer");
  if (!aligned(trits, 4)) return fail(PTQ_ERR_ALIGN, "ptq2_unpack: trits need 4-byte alignment");
  cudaError_t e = launch_unpack_pq2(wq, trits, N, K, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq2_unpack launch");
}

static size_t matmul_pq2_ws_bytes(int64_t M, int64_t N, int64_t K, ptq_dtype dt) {
  if (dt == PTQ_F32) return (M >= 1 && M <= 8) ? gemv_lut_pq2_workspace_bytes(N, K, M) : 0;
  return gemm_tc_workspace_bytes(M, N, K);
}

PTQ_API size_t ptq_matmul_pq2_workspace_bytes(int64_t M, int64_t N, int64_t K, ptq_dtype dtype) {
  int64_t t;
  if (!dtype_ok(dtype) || M < 0 || N < 0 || K <= 0 || K % kRot != 0 || !mul_ok(N, K, &t) ||
      !mul_ok(M, N, &t) || !mul_ok(t, 4, &t))
    return 0;
  return matmul_pq2_ws_bytes(M, N, K, dtype);
}

PTQ_API ptq_status ptq_matmul_pq2(const uint8_t* wq, const uint16_t* scales, const void* x,
                                  void* y, int64_t M, int64_t N, int64_t K, ptq_dtype dtype,
                                  void* ws, size_t ws_bytes, ptq_stream_t stream) {
  t_msg[0] = 0;
  const char* who = "ptq_matmul_pq2";
  const Route* r = nullptr;
  ptq_status s = check_matmul(wq, scales, x, y, M, N, K, dtype, who, &r);
  if (s != PTQ_OK || M == 0 || N == 0) return s;
  if (K % kRot != 0)
    return fail(PTQ_ERR_UNSUPPORTED, "%s: PQ2_0 is served for K %% 1024 == 0 only (K=%lld)", who,
                (long long)K);
  const size_t need = matmul_pq2_ws_bytes(M, N, K, dtype);
  const bool required = dtype == PTQ_F32 && need > 0;
  if (required && !ws)
    return fail(PTQ_ERR_WORKSPACE, "%s: workspace is NULL (%zu bytes needed)", who, need);
  if (required && ws_bytes < need)
    return fail(PTQ_ERR_WORKSPACE, "%s: workspace has %zu bytes, %zu needed", who, ws_bytes, need);
  if (ws && !aligned(ws, 16))
    return fail(PTQ_ERR_ALIGN, "%s: workspace needs 16-byte alignment", who);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (r->kernel == Kernel::GemvF32) {  // the tokens in turn in one launch, as for PTQ1_0
    e = launch_gemv_lut_pq2(wq, scales, static_cast<const float*>(x), nullptr,
                            static_cast<float*>(y), static_cast<float*>(ws), M, N, K, st);
  } else {
    e = launch_gemm_tc_pq2(wq, scales, x, y, M, N, K, ws, ws ? ws_bytes : 0, st);
  }
  if (e == cudaErrorNotSupported)
    return fail(PTQ_ERR_UNSUPPORTED, "%s: shape N=%lld K=%lld not served for PQ2_0", who,
                (long long)N, (long long)K);
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_matmul_pq2 launch");
}

// ---- rotate + matmul ------------------------------------------------------
// Workspace: [matmul scratch | R x (M x K of dtype), used when the rotation
// runs as its own kernel], each rounded up to 256 bytes.
static bool rotmm_layout(int64_t M, int64_t N, int64_t K, ptq_dtype dt, size_t* xr_off,
                         size_t* total) {
  int64_t xb;
  if (!mul_ok(M, K, &xb) || !mul_ok(xb, (int64_t)dsize(dt), &xb)) return false;
  *xr_off = (matmul_ws_bytes(M, N, K, dt) + 255) / 256 * 256;
  *total = *xr_off + (size_t)((xb + 255) / 256 * 256);
  return true;
}

PTQ_API size_t ptq_rotate_matmul_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                                 ptq_dtype dtype) {
  int64_t t;
  size_t off, total;
  if (!dtype_ok(dtype) || M < 0 || N < 0 || K <= 0 || K % kRot != 0 || !mul_ok(N, K, &t) ||
      !mul_ok(M, N, &t) || !mul_ok(t, 4, &t) || !rotmm_layout(M, N, K, dtype, &off, &total))
    return 0;
  return total;
}

PTQ_API ptq_status ptq_rotate_matmul(const uint8_t* wq, const uint16_t* scales, const void* x,
                                     const int8_t* signs, void* y, int64_t M, int64_t N,
                                     int64_t K, ptq_dtype dtype, void* ws, size_t ws_bytes,
                                     ptq_stream_t stream) {
  t_msg[0] = 0;
  const char* who = "ptq_rotate_matmul";
  if (dtype_ok(dtype) && K > 0 && K % kRot != 0)
    return fail(PTQ_ERR_SHAPE, "%s: need K %% 1024 == 0 (K=%lld)", who, (long long)K);
  const Route* r = nullptr;
  ptq_status s = check_matmul(wq, scales, x, y, M, N, K, dtype, who, &r);
  if (s != PTQ_OK || M == 0 || N == 0) return s;
  if (!signs) return fail(PTQ_ERR_NULL, "%s: signs is NULL", who);
  if (!aligned(signs, 4)) return fail(PTQ_ERR_ALIGN, "%s: signs need 4-byte alignment", who);
  size_t xr_off, need;
  if (!rotmm_layout(M, N, K, dtype, &xr_off, &need)) return fail(PTQ_ERR_SHAPE, "%s: size overflow", who);
  if (!ws) return fail(PTQ_ERR_WORKSPACE, "%s: workspace is NULL (%zu bytes needed)", who, need);
  if (ws_bytes < need)
    return fail(PTQ_ERR_WORKSPACE, "%s: workspace has %zu bytes, %zu needed", who, ws_bytes, need);
  if (!aligned(ws, 16)) return fail(PTQ_ERR_ALIGN, "%s: workspace needs 16-byte alignment", who);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (r->kernel == Kernel::GemvF32 && gemv_lut_supported(N, K, true)) {
    // the rotation runs inside the GEMV, on the activations each CTA reads
    e = gemv_lut_tokens(wq, scales, static_cast<const float*>(x), signs, static_cast<float*>(y),
                        static_cast<float*>(ws), M, N, K, st);
  } else {
    // R x is kept in fp32 (fp32 routes) or fp16 (bf16 route): with an fp16
    // operand the GEMM's weight tile t * s is exact, so the one rounding of
    // the rotated activation (2^-11) is the only error before the output's
    // own bf16 rounding
    void* xr = static_cast<char*>(ws) + xr_off;
    const Act op = dtype == PTQ_BF16 ? Act::F16 : Act::F32;
    e = launch_fwht(x, act_of(dtype), xr, op, signs, M, K, st);
    if (e == cudaSuccess)
      e = run_matmul(r, wq, scales, xr, op, y, act_of(dtype), M, N, K, ws, xr_off, st);
  }
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_rotate_matmul launch");
}

// ptq_rotate_matmul on host buffers: the workspace holds x (M x K), y (M x
// N) and then ptq_rotate_matmul's own workspace, each rounded up to 256 bytes.
static bool rotmm_host_layout(int64_t M, int64_t N, int64_t K, ptq_dtype dt, size_t* y_off,
                              size_t* ws_off, size_t* total) {
  int64_t xb, yb;
  if (!mul_ok(M, K, &xb) || !mul_ok(xb, (int64_t)dsize(dt), &xb) || !mul_ok(M, N, &yb) ||
      !mul_ok(yb, (int64_t)dsize(dt), &yb))
    return false;
  const size_t inner = ptq_rotate_matmul_workspace_bytes(M, N, K, dt);
  auto up = [](int64_t v) { return (size_t)((v + 255) / 256 * 256); };
  *y_off = up(xb);
  *ws_off = *y_off + up(yb);
  *total = *ws_off + inner;
  return true;
}

PTQ_API size_t ptq_rotate_matmul_host_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                                      ptq_dtype dtype) {
  size_t y_off, ws_off, total;
  if (ptq_rotate_matmul_workspace_bytes(M, N, K, dtype) == 0 ||
      !rotmm_host_layout(M, N, K, dtype, &y_off, &ws_off, &total))
    return 0;
  return total;
}

PTQ_API ptq_status ptq_rotate_matmul_host(const uint8_t* wq, const uint16_t* scales,
                                          const void* x_host, const int8_t* signs, void* y_host,
                                          int64_t M, int64_t N, int64_t K, ptq_dtype dtype,
                                          void* ws, size_t ws_bytes, ptq_stream_t stream) {
  t_msg[0] = 0;
  const char* who = "ptq_rotate_matmul_host";
  if (!dtype_ok(dtype)) return fail(PTQ_ERR_VALUE, "%s: unknown dtype %d", who, (int)dtype);
  if (M < 0 || N < 0 || K <= 0 || K % kRot != 0)
    return fail(PTQ_ERR_SHAPE, "%s: need M, N >= 0 and K %% 1024 == 0 (M=%lld N=%lld K=%lld)", who,
                (long long)M, (long long)N, (long long)K);
  if (M == 0 || N == 0) return PTQ_OK;
  if (!x_host || !y_host) return fail(PTQ_ERR_NULL, "%s: NULL host buffer", who);
  size_t y_off, ws_off, need;
  if (ptq_rotate_matmul_workspace_bytes(M, N, K, dtype) == 0 ||
      !rotmm_host_layout(M, N, K, dtype, &y_off, &ws_off, &need))
    return fail(PTQ_ERR_SHAPE, "%s: size overflow", who);
  if (!ws) return fail(PTQ_ERR_WORKSPACE, "%s: workspace is NULL (%zu bytes needed)", who, need);
  if (ws_bytes < need)
    return fail(PTQ_ERR_WORKSPACE, "%s: workspace has %zu bytes, %zu needed", who, ws_bytes, need);
  if (!aligned(ws, 256)) return fail(PTQ_ERR_ALIGN, "%s: workspace needs 256-byte alignment", who);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  const size_t es = dsize(dtype);
  // Page-locked memory that the runtime maps into the device's address space
  // (a device address for both buffers): the kernels read x and write y there
  // directly, over the host link, with no copy engine in between.
  cudaPointerAttributes ax, ay;
  const cudaError_t qx = cudaPointerGetAttributes(&ax, x_host);
  const cudaError_t qy = cudaPointerGetAttributes(&ay, y_host);
  if (qx != cudaSuccess || qy != cudaSuccess)
    static_cast<void>(cudaGetLastError());  // the query's own error: use the copies
  else if (ax.type == cudaMemoryTypeHost && ay.type == cudaMemoryTypeHost &&
           ax.devicePointer != nullptr && ay.devicePointer != nullptr &&
           aligned(ax.devicePointer, 16) && aligned(ay.devicePointer, 16))
    return ptq_rotate_matmul(wq, scales, ax.devicePointer, signs, ay.devicePointer, M, N, K,
                             dtype, base + ws_off, need - ws_off, stream);
  cudaError_t e = cudaMemcpyAsync(base, x_host, (size_t)(M * K) * es, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "ptq_rotate_matmul_host: copy of x");
  const ptq_status s = ptq_rotate_matmul(wq, scales, base, signs, base + y_off, M, N, K, dtype,
                                         base + ws_off, need - ws_off, stream);
  if (s != PTQ_OK) return s;
  e = cudaMemcpyAsync(y_host, base + y_off, (size_t)(M * N) * es, cudaMemcpyDeviceToHost, st);
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_rotate_matmul_host: copy of y");
}

// Workspace of ptq_ffn, each region rounded up to 256 bytes:
//   xr (M x H) | gu (M x 2I, fp32) | h (M x I, fp32) [| hr (M x I, fp16)]
//   | part (the decode GEMV's row sums, shared by the two projections, which
//     never hold it at the same time; for the prefill GEMM, gate/up's split-K
//     partial sums)
// fp32 path: xr fp32, h rotated in place.  bf16 path: xr and hr are fp16
// (the tensor-core operands; 11 significant bits against bf16's 8, and the
// block scale times a trit is exact in fp16), gate/up and SwiGLU stay fp32,
// so the only bf16 rounding is the output.
static bool ffn_layout(int64_t M, int64_t H, int64_t I, ptq_dtype dt, size_t off[5],
                       size_t* total) {
  int64_t a, b, c, d = 0;
  const int64_t ds = (int64_t)dsize(dt);
  if (!mul_ok(M, H, &a) || !mul_ok(a, ds, &a) || !mul_ok(M, 2 * I, &b) || !mul_ok(b, 4, &b) ||
      !mul_ok(M, I, &c) || !mul_ok(c, 4, &c))
    return false;
  if (dt == PTQ_BF16 && (!mul_ok(M, I, &d) || !mul_ok(d, 2, &d))) return false;
  auto up = [](int64_t v) { return (v + 255) / 256 * 256; };
  off[0] = 0;
  off[1] = (size_t)up(a);
  off[2] = off[1] + (size_t)up(b);
  off[3] = off[2] + (size_t)up(c);
  off[4] = off[3] + (size_t)up(d);
  // decode: the larger of the two projections' row sums; prefill: gate/up's
  // split-K sums (the down projection's use the gate/up region, dead by
  // then, and on the bf16 path the h region after it)
  const size_t p1 = matmul_ws_bytes(M, 2 * I, H, dt), p2 = matmul_ws_bytes(M, H, I, dt);
  *total = off[4] + (dt == PTQ_BF16 ? p1 : (p1 > p2 ? p1 : p2));
  return true;
}

PTQ_API size_t ptq_ffn_workspace_bytes(int64_t M, int64_t H, int64_t I, ptq_dtype dtype) {
  size_t off[5], total;
  if (!dtype_ok(dtype) || M < 0 || H <= 0 || I <= 0 || H % kRot || I % kRot ||
      I > INT64_MAX / 2 || !ffn_layout(M, H, I, dtype, off, &total))
    return 0;
  return total;
}

// The per-block checks of ptq_ffn (weights, signs, dtype routing); the
// shape and workspace checks are the caller's.
struct FfnRoutes {
  const Route* gu;
  const Route* d;
};

static ptq_status check_ffn_block(const uint8_t* wgu_q, const uint16_t* wgu_s, const uint8_t* wd_q,
                                  const uint16_t* wd_s, const int8_t* signs_in,
                                  const int8_t* signs_mid, const void* x, const void* y,
                                  int64_t M, int64_t H, int64_t I, ptq_dtype dtype, const char* who,
                                  FfnRoutes* r) {
  ptq_status s = check_matmul(wgu_q, wgu_s, x, y, M, 2 * I, H, dtype, who, &r->gu);
  if (s != PTQ_OK) return s;
  s = check_matmul(wd_q, wd_s, x, y, M, H, I, dtype, who, &r->d);
  if (s != PTQ_OK) return s;
  if (!signs_in || !signs_mid) return fail(PTQ_ERR_NULL, "%s: NULL signs", who);
  if (!aligned(signs_in, 4) || !aligned(signs_mid, 4))
    return fail(PTQ_ERR_ALIGN, "%s: signs need 4-byte alignment", who);
  return PTQ_OK;
}

// Launches one feed-forward block; base/off/need are ffn_layout's regions.
static cudaError_t run_ffn_block(const FfnRoutes& r, const uint8_t* wgu_q, const uint16_t* wgu_s,
                                 const uint8_t* wd_q, const uint16_t* wd_s,
                                 const int8_t* signs_in, const int8_t* signs_mid, const void* x,
                                 void* y, int64_t M, int64_t H, int64_t I, ptq_dtype dtype,
                                 char* base, const size_t off[5], size_t need, cudaStream_t st) {
  void* xr = base + off[0];
  float* gu = reinterpret_cast<float*>(base + off[1]);
  float* h = reinterpret_cast<float*>(base + off[2]);
  const bool bf = dtype == PTQ_BF16;
  void* hr = bf ? static_cast<void*>(base + off[3]) : static_cast<void*>(h);
  void* part = base + off[4];
  const Act op = bf ? Act::F16 : Act::F32;  // tensor-core operand type
  if (!bf && r.gu->kernel == Kernel::GemvF32 && gemv_lut_supported(2 * I, H, true) &&
      gemv_lut_supported(H, I, true)) {
    // decode, token by token: each table-lookup GEMV rotates its own
    // activations, and the gate/up row sums are reduced straight into
    // h = silu(g) * u
    cudaError_t e = cudaSuccess;
    for (int64_t m = 0; m < M && e == cudaSuccess; ++m) {
      float* hm = h + m * I;
      e = launch_gemv_lut(wgu_q, wgu_s, static_cast<const float*>(x) + m * H, signs_in, hm,
                          static_cast<float*>(part), 1, 2 * I, H, LutEpilogue::SwiGLU, st);
      if (e == cudaSuccess)
        e = launch_gemv_lut(wd_q, wd_s, hm, signs_mid, static_cast<float*>(y) + m * H,
                            static_cast<float*>(part), 1, H, I, LutEpilogue::Plain, st);
    }
    return e;
  }
  cudaError_t e = launch_fwht(x, act_of(dtype), xr, op, signs_in, M, H, st);
  // prefill: SwiGLU in the gate/up GEMM's epilogue when that GEMM runs
  // unsplit; otherwise gate/up into fp32, then the SwiGLU kernel
  bool fused = false;
  if (e == cudaSuccess && r.gu->kernel == Kernel::GemmBf16) {
    e = launch_gemm_tc_swiglu(wgu_q, wgu_s, xr, op, h, M, I, H, st);
    fused = e == cudaSuccess;
    if (e == cudaErrorNotSupported) e = cudaSuccess;
  }
  if (e == cudaSuccess && !fused) {
    e = run_matmul(r.gu, wgu_q, wgu_s, xr, op, gu, Act::F32, M, 2 * I, H, part, need - off[4], st);
    if (e == cudaSuccess) e = launch_swiglu(gu, h, M, I, st);
  }
  if (e == cudaSuccess) e = launch_fwht(h, Act::F32, hr, op, signs_mid, M, I, st);
  // the down projection's split-K partials go where gate/up was (dead after
  // SwiGLU) and, on the bf16 path, where h was (dead once rotated into hr)
  if (e == cudaSuccess)
    e = run_matmul(r.d, wd_q, wd_s, hr, op, y, act_of(dtype), M, H, I, gu,
                   (bf ? off[3] : off[2]) - off[1], st);
  return e;
}

static bool ffn_shape_ok(int64_t M, int64_t H, int64_t I) {
  return M >= 0 && H > 0 && I > 0 && H % kRot == 0 && I % kRot == 0 && I <= INT64_MAX / 4;
}

PTQ_API ptq_status ptq_ffn(const uint8_t* wgu_q, const uint16_t* wgu_s, const uint8_t* wd_q,
                           const uint16_t* wd_s, const int8_t* signs_in, const int8_t* signs_mid,
                           const void* x, void* y, int64_t M, int64_t H, int64_t I,
                           ptq_dtype dtype, void* ws, size_t ws_bytes, ptq_stream_t stream) {
  t_msg[0] = 0;
  const char* who = "ptq_ffn";
  if (!dtype_ok(dtype)) return fail(PTQ_ERR_VALUE, "%s: unknown dtype %d", who, (int)dtype);
  if (!ffn_shape_ok(M, H, I))
    return fail(PTQ_ERR_SHAPE, "%s: need M >= 0, H and I positive multiples of 1024", who);
  size_t off[5], need;
  if (!ffn_layout(M, H, I, dtype, off, &need)) return fail(PTQ_ERR_SHAPE, "%s: size overflow", who);
  if (M == 0) return PTQ_OK;
  FfnRoutes r;
  ptq_status s =
      check_ffn_block(wgu_q, wgu_s, wd_q, wd_s, signs_in, signs_mid, x, y, M, H, I, dtype, who, &r);
  if (s != PTQ_OK) return s;
  if (!ws) return fail(PTQ_ERR_WORKSPACE, "%s: workspace is NULL (%zu bytes needed)", who, need);
  if (ws_bytes < need)
    return fail(PTQ_ERR_WORKSPACE, "%s: workspace has %zu bytes, %zu needed", who, ws_bytes, need);
  if (!aligned(ws, 16)) return fail(PTQ_ERR_ALIGN, "%s: workspace needs 16-byte alignment", who);
  const cudaError_t e = run_ffn_block(r, wgu_q, wgu_s, wd_q, wd_s, signs_in, signs_mid, x, y, M, H,
                                      I, dtype, static_cast<char*>(ws), off, need,
                                      reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_ffn launch");
}

// Workspace of ptq_ffn_stack, each region rounded up to 256 bytes:
//   xn (M x H, dtype: the block input) | y (M x H, dtype: the block output)
//   | ptq_ffn's workspace | [fp32, M <= 8: a second M x 2I fp32 gate/up buffer
//   for the persistent path]
static bool stack_layout(int64_t M, int64_t H, int64_t I, ptq_dtype dt, size_t off[4],
                         size_t ffn_off[5], size_t* ffn_need, size_t* total) {
  int64_t a, b = 0;
  if (!mul_ok(M, H, &a) || !mul_ok(a, (int64_t)dsize(dt), &a) || a > INT64_MAX / 4) return false;
  if (dt == PTQ_F32 && M <= kStackMaxTokens && (!mul_ok(M, 2 * I, &b) || !mul_ok(b, 4, &b)))
    return false;
  if (!ffn_layout(M, H, I, dt, ffn_off, ffn_need)) return false;
  const size_t r = (size_t)((a + 255) / 256 * 256);
  off[0] = 0;
  off[1] = r;
  off[2] = 2 * r;
  if (*ffn_need > SIZE_MAX / 2 - off[2]) return false;
  off[3] = off[2] + (*ffn_need + 255) / 256 * 256;
  *total = off[3] + (size_t)b;
  return true;
}

PTQ_API size_t ptq_ffn_stack_workspace_bytes(int64_t M, int64_t H, int64_t I, ptq_dtype dtype) {
  size_t off[4], foff[5], fneed, total;
  if (!dtype_ok(dtype) || !ffn_shape_ok(M, H, I) ||
      !stack_layout(M, H, I, dtype, off, foff, &fneed, &total))
    return 0;
  return total;
}

// Up to 8 decode tokens in fp32 run the stack as one persistent launch per
// 24 layers when the device and the shapes allow it, unless the caller asks
// for the bitwise-reproducible per-layer path.
static bool stack_persistent(int64_t M, int64_t H, int64_t I, ptq_dtype dt, unsigned flags) {
  return M >= 1 && M <= kStackMaxTokens && dt == PTQ_F32 &&
         !(flags & PTQ_STACK_DETERMINISTIC) && stack_decode_supported(H, I);
}

PTQ_API ptq_status ptq_ffn_stack_route(int64_t M, int64_t H, int64_t I, ptq_dtype dtype,
                                       const char** name) {
  t_msg[0] = 0;
  if (!name) return fail(PTQ_ERR_NULL, "ptq_ffn_stack_route: name is NULL");
  if (!dtype_ok(dtype))
    return fail(PTQ_ERR_VALUE, "ptq_ffn_stack_route: unknown dtype %d", (int)dtype);
  if (M < 1 || !ffn_shape_ok(M, H, I))
    return fail(PTQ_ERR_SHAPE, "ptq_ffn_stack_route: need M >= 1, H and I multiples of 1024");
  if (!find_route(M, dtype))
    return fail(PTQ_ERR_UNSUPPORTED, "ptq_ffn_stack_route: no kernel for M=%lld dtype=%s",
                (long long)M, dtype == PTQ_F32 ? "f32" : "bf16");
  *name = stack_persistent(M, H, I, dtype, 0u) ? "stack_decode_persistent" : "stack_per_layer";
  return PTQ_OK;
}

PTQ_API ptq_status ptq_ffn_stack(const ptq_ffn_layer* layers, int64_t L, float* x, int64_t M,
                                 int64_t H, int64_t I, float eps, ptq_dtype dtype, void* ws,
                                 size_t ws_bytes, ptq_stream_t stream) {
  return ptq_ffn_stack_ex(layers, L, x, M, H, I, eps, dtype, ws, ws_bytes, 0u, stream);
}

PTQ_API ptq_status ptq_ffn_stack_ex(const ptq_ffn_layer* layers, int64_t L, float* x, int64_t M,
                                    int64_t H, int64_t I, float eps, ptq_dtype dtype, void* ws,
                                    size_t ws_bytes, unsigned flags, ptq_stream_t stream) {
  t_msg[0] = 0;
  const char* who = "ptq_ffn_stack";
  if (!dtype_ok(dtype)) return fail(PTQ_ERR_VALUE, "%s: unknown dtype %d", who, (int)dtype);
  if (flags & ~(unsigned)PTQ_STACK_DETERMINISTIC)
    return fail(PTQ_ERR_VALUE, "%s: unknown flags 0x%x", who, flags);
  if (L < 0 || !ffn_shape_ok(M, H, I))
    return fail(PTQ_ERR_SHAPE, "%s: need L >= 0, M >= 0, H and I positive multiples of 1024",
                who);
  if (!(eps >= 0.0f) || !(eps < INFINITY))
    return fail(PTQ_ERR_VALUE, "%s: eps must be finite and >= 0", who);
  size_t off[4], foff[5], fneed, need;
  if (!stack_layout(M, H, I, dtype, off, foff, &fneed, &need))
    return fail(PTQ_ERR_SHAPE, "%s: size overflow", who);
  if (M == 0 || L == 0) return PTQ_OK;
  if (!layers) return fail(PTQ_ERR_NULL, "%s: layers is NULL", who);
  if (!x) return fail(PTQ_ERR_NULL, "%s: x is NULL", who);
  if (!aligned(x, 16)) return fail(PTQ_ERR_ALIGN, "%s: x needs 16-byte alignment", who);
  if (!ws) return fail(PTQ_ERR_WORKSPACE, "%s: workspace is NULL (%zu bytes needed)", who, need);
  if (ws_bytes < need)
    return fail(PTQ_ERR_WORKSPACE, "%s: workspace has %zu bytes, %zu needed", who, ws_bytes, need);
  if (!aligned(ws, 16)) return fail(PTQ_ERR_ALIGN, "%s: workspace needs 16-byte alignment", who);
  char* base = static_cast<char*>(ws);
  void* xn = base + off[0];
  void* y = base + off[1];
  char* fbase = base + off[2];
  // every layer is checked before the first launch, so a refused call leaves
  // x untouched
  FfnRoutes r0 = {nullptr, nullptr};
  for (int64_t l = 0; l < L; ++l) {
    const ptq_ffn_layer& ly = layers[l];
    char lw[64];
    snprintf(lw, sizeof lw, "%s: layer %lld", who, (long long)l);
    FfnRoutes r;
    ptq_status s = check_ffn_block(ly.wgu_q, ly.wgu_s, ly.wd_q, ly.wd_s, ly.signs_in,
                                   ly.signs_mid, xn, y, M, H, I, dtype, lw, &r);
    if (s != PTQ_OK) return s;
    if (!ly.norm_w) return fail(PTQ_ERR_NULL, "%s: norm_w is NULL", lw);
    if (!aligned(ly.norm_w, 16)) return fail(PTQ_ERR_ALIGN, "%s: norm_w needs 16-byte alignment", lw);
    if (l == 0) r0 = r;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (stack_persistent(M, H, I, dtype, flags) && stack_decode_ss_bytes(M) <= off[1] - off[0] &&
      stack_decode_bar_bytes(L) <= off[2] - off[1]) {
    // decode tokens: the whole stack as one persistent launch per 24 layers;
    // its scratch comes from this workspace (one gate/up buffer where the
    // block's gate/up sums would go, the other in the last region, the norm
    // statistics where xn would go, the barrier counters where y would)
    const cudaError_t e = launch_stack_decode(
        layers, L, x, M, reinterpret_cast<float*>(fbase + foff[1]),
        reinterpret_cast<float*>(base + off[3]), reinterpret_cast<float*>(base + off[0]),
        reinterpret_cast<unsigned*>(base + off[1]), H, I, eps, st);
    if (e != cudaErrorNotSupported)
      return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_ffn_stack launch");
  }
  const Act t = act_of(dtype);
  cudaError_t e = cudaSuccess;
  for (int64_t l = 0; l < L && e == cudaSuccess; ++l) {
    const ptq_ffn_layer& ly = layers[l];
    // x += y (from the second layer on); xn = RMSNorm(x) * g_l
    e = launch_add_rmsnorm(x, l ? y : nullptr, ly.norm_w, xn, t, M, H, eps, st);
    if (e == cudaSuccess)
      e = run_ffn_block(r0, ly.wgu_q, ly.wgu_s, ly.wd_q, ly.wd_s, ly.signs_in, ly.signs_mid, xn, y,
                        M, H, I, dtype, fbase, foff, fneed, st);
  }
  if (e == cudaSuccess) e = launch_add_rmsnorm(x, y, nullptr, nullptr, t, M, H, eps, st);
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_ffn_stack launch");
}

PTQ_API ptq_status ptq_selftest_timeout(ptq_stream_t stream) {
  t_msg[0] = 0;
  cudaError_t e = launch_selftest_timeout(reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_selftest_timeout launch");
}

PTQ_API ptq_status ptq_selftest_grid_timeout(ptq_stream_t stream) {
  t_msg[0] = 0;
  cudaError_t e = launch_selftest_grid_timeout(reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PTQ_OK : cuda_fail(e, "ptq_selftest_grid_timeout launch");
}

PTQ_API ptq_status ptq_device_check(ptq_stream_t stream) {
  t_msg[0] = 0;
  int v = 0;
  cudaError_t e = read_and_clear_device_status(&v, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ptq_device_check");
  if (v & kDevTimeout)
    return fail(PTQ_ERR_TIMEOUT, "a bounded device-side wait ran out (status word 0x%x)", v);
  if (v & kDevRange)
    return fail(PTQ_ERR_RANGE,
                "a rotated bf16-route operand exceeded the fp16 range (|v| >= 65520) and was "
                "stored as infinity (status word 0x%x)", v);
  return PTQ_OK;
}

}  // extern "C"

// ffn_noalloc.cu -- ptq_ffn for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc at all: code that runs
// while its stream is being captured into a CUDA graph (an allocation there
// would not be part of the graph), real-time decode loops that may not take
// the device-wide synchronisation and unbounded latency of an allocation,
// and hosts whose device memory is entirely reserved by another allocator
// (a framework's caching allocator) that a C-ABI caller cannot reach.  For
// them this file holds the feed-forward block's scratch in a file-scope
// device array, so the call allocates nothing.  The caller still passes the
// inputs and the output.
//
// The array lives in every device that loads this library, for as long as
// the process lives.  All calls share it: two calls whose kernels overlap on
// the GPU (different streams without ordering) race on it.  Nothing in it
// has to start at zero: every region the block reads is written earlier in
// the same call.
#include <mutex>

#include "ptq_internal.cuh"

namespace ptq {
namespace {

static __device__ __align__(256) unsigned char g_ffn_scratch[PTQ_FFN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
static void* g_scratch_addr[kMaxDev];
static cudaError_t g_scratch_err[kMaxDev];
static std::once_flag g_scratch_once[kMaxDev];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is asked of
// the runtime, once per device, with that device current.
static cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::call_once(g_scratch_once[dev], [dev] {
    void* p = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_ffn_scratch);
    g_scratch_addr[dev] = p;
  });
  *out = g_scratch_addr[dev];
  return g_scratch_err[dev];
}

}  // namespace
}  // namespace ptq

extern "C" PTQ_API ptq_status ptq_ffn_noalloc(const uint8_t* wgu_q, const uint16_t* wgu_s,
                                              const uint8_t* wd_q, const uint16_t* wd_s,
                                              const int8_t* signs_in, const int8_t* signs_mid,
                                              const void* x, void* y, int64_t M, int64_t H,
                                              int64_t I, ptq_dtype dtype, ptq_stream_t stream) {
  const size_t need = ptq_ffn_workspace_bytes(M, H, I, dtype);
  if (need == 0)  // invalid arguments: let ptq_ffn name them
    return ptq_ffn(wgu_q, wgu_s, wd_q, wd_s, signs_in, signs_mid, x, y, M, H, I, dtype, nullptr, 0,
                   stream);
  if (need > (size_t)PTQ_FFN_NOALLOC_SCRATCH_BYTES)
    return ptq::fail(PTQ_ERR_WORKSPACE,
                     "ptq_ffn_noalloc: M=%lld H=%lld I=%lld needs %zu bytes of scratch; the "
                     "built-in array holds %d (use ptq_ffn with a workspace)",
                     (long long)M, (long long)H, (long long)I, need,
                     (int)PTQ_FFN_NOALLOC_SCRATCH_BYTES);
  void* ws = nullptr;
  cudaError_t e = ptq::scratch_address(&ws);
  if (e != cudaSuccess) return ptq::cuda_fail(e, "ptq_ffn_noalloc: cudaGetSymbolAddress");
  return ptq_ffn(wgu_q, wgu_s, wd_q, wd_s, signs_in, signs_mid, x, y, M, H, I, dtype, ws,
                 (size_t)PTQ_FFN_NOALLOC_SCRATCH_BYTES, stream);
}

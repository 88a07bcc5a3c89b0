// ffn_noalloc.cu -- ptq_ffn for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: real-time decode loops
// that may not take the device-wide synchronisation and unbounded latency of
// an allocation, plug-ins and embedded hosts that are handed a stream but no
// allocator, and processes whose device memory is entirely reserved by
// another allocator (a framework's caching allocator) that a C-ABI caller
// cannot reach.  For them this file holds the feed-forward block's scratch in
// a file-scope device array, so the call allocates nothing.  The caller
// still passes the inputs and the output.
//
// The array lives in every device that loads this library, for as long as
// the process lives.  All calls share it: two calls whose kernels overlap on
// the GPU (different streams without ordering) race on it.  Nothing in it
// has to start at zero: every region the block reads is written earlier in
// the same call.
#include <atomic>

#include "ptq_internal.cuh"

namespace ptq {
namespace {

static __device__ __align__(256) unsigned char g_ffn_scratch[PTQ_FFN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
static std::atomic<void*> g_scratch_addr[kMaxDev];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is asked of
// the runtime with that device current.  Only a successful lookup is cached;
// after a failed one (for instance a sticky error from an earlier call) the
// next call asks again.
static cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_ffn_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
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

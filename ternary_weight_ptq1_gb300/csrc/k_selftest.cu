// k_selftest.cu -- a wait that runs out, to test the timeout path.
//
// The kernels that stage operands with TMA wait on mbarriers, and every wait
// is bounded: one that runs out raises the device status word and the kernel
// returns instead of hanging.  This kernel exercises that path on purpose,
// without any fault: one thread initialises an mbarrier that nothing will
// arrive on, waits on it with the library's bounded wait (a short poll
// limit), finds it ran out, and raises the status word.  Nothing is left in
// flight when it exits.
#include "async_util.cuh"
#include "ptq_internal.cuh"

namespace ptq {
namespace {

__global__ void selftest_timeout_kernel(int* status, uint32_t polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const uint32_t a = smem_addr(&bar);
  bool done = false;
  for (uint32_t i = 0; i < polls && !done; ++i) {
    uint32_t d;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(d)
        : "r"(a), "r"(0u)
        : "memory");
    done = d != 0;
  }
  if (!done) atomicOr(status, kDevTimeout);
}

}  // namespace

cudaError_t launch_selftest_timeout(cudaStream_t st) {
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidDevice;
  selftest_timeout_kernel<<<1, 32, 0, st>>>(status, 4096u);
  return cudaGetLastError();
}

}  // namespace ptq

// tma_util.cu -- host-side creation of 2-D TMA tensor maps, shared by the
// kernels that stage operands with the tensor memory accelerator.  The
// driver entry point is looked up once through the runtime, so the library
// does not link libcuda directly.
#include <cudaTypedefs.h>

#include <mutex>

#include "ptq_internal.cuh"

namespace ptq {
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;
}  // namespace

cudaError_t encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                          uint64_t inner, uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                    cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
      g_encode_err = cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode_err != cudaSuccess) return g_encode_err;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace ptq

// tma_util.cu -- host-side creation of 2-D TMA tensor maps, shared by the
// kernels that stage operands with the tensor memory accelerator.  The
// driver entry point is looked up once through the runtime, so the library
// does not link libcuda directly.  A map holds only an address, sizes,
// strides and the box, so each host thread keeps the maps it made last (64,
// replaced in turn) and hands a copy back for the same arguments: a decode
// loop over a model's weights then encodes each map once.
#include <cudaTypedefs.h>

#include <mutex>

#include "ptq_internal.cuh"

namespace ptq {
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;
}  // namespace

namespace {
struct MapKey {
  const void* base;
  uint64_t inner, rows, row_bytes;
  uint32_t box_inner, box_rows;
  int dt, swizzle;
  bool operator==(const MapKey& o) const {
    return base == o.base && inner == o.inner && rows == o.rows && row_bytes == o.row_bytes &&
           box_inner == o.box_inner && box_rows == o.box_rows && dt == o.dt &&
           swizzle == o.swizzle;
  }
};
constexpr int kMapCache = 64;
struct MapCache {
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  int used = 0, next = 0;
};
thread_local MapCache t_maps;
}  // namespace

cudaError_t encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base,
                          uint64_t inner, uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  const MapKey k{base, inner, rows, row_bytes, box_inner, box_rows, (int)dt, (int)swizzle};
  MapCache& c = t_maps;
  for (int i = 0; i < c.used; ++i)
    if (c.key[i] == k) {
      *map = c.map[i];
      return cudaSuccess;
    }
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
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const int slot = c.used < kMapCache ? c.used++ : c.next;
  c.next = (slot + 1) % kMapCache;
  c.key[slot] = k;
  c.map[slot] = *map;
  return cudaSuccess;
}

}  // namespace ptq

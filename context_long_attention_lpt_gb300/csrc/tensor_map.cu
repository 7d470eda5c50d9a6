#include "tensor_map.h"

#include <mutex>

#include <cuda_runtime.h>

#include "splitkv.h"
#include "status.h"

namespace splitkv {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_lookup_err = cudaSuccess;

void lookup() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  g_lookup_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (g_lookup_err == cudaSuccess && q == cudaDriverEntryPointSuccess) g_encode = reinterpret_cast<EncodeTiledFn>(fn);
}

}  // namespace

int encode_bf16_3d(CUtensorMap* map, const void* base, const uint64_t dims[3],
                   const uint64_t strides_bytes[2], const uint32_t box[3],
                   CUtensorMapSwizzle swizzle) {
  std::call_once(g_once, lookup);
  if (!g_encode)
    return fail(SPLITKV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable: %s", cudaGetErrorString(g_lookup_err));
  const cuuint64_t gdim[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t gstride[2] = {strides_bytes[0], strides_bytes[1]};
  const cuuint32_t bdim[3] = {box[0], box[1], box[2]};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride,
                              bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(SPLITKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return SPLITKV_OK;
}

}  // namespace splitkv
